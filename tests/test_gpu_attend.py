"""Block-sparse attend (indexer_sparse_attend) against the float64 oracle
(oracle/attend.py): every output element within the oracle's fp32 error
bound (chain of at most 64 sequential additions, exp2f within 2^-21).

The ids come from the indexer on the GPU (the buffer the attend reads in a
real step) and are given to the oracle as an input; the main KV cache is
the workloads module's hashed bf16 cache (the CPU computes only the pages
it checks)."""
import numpy as np
import pytest

import workloads
from oracle import attend as oat
from gpu_util import gpu_cache, make_plan, torch_dev, up

pytestmark = pytest.mark.gpu

SCALE = 128 ** -0.5


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _ids(w, kv):
    """The indexer's ids for every row of the workload (decode rows, then
    prefill rows), from the GPU indexer."""
    import torch
    plan = make_plan(w)
    parts = []
    if w.num_decode_reqs:
        parts.append(plan.decode(up(w.q_decode), kv, up(w.dec_page_table), up(w.dec_seq_lens), w.query_len))
    if w.num_prefill_reqs:
        parts.append(plan.prefill(up(w.q_prefill), up(w.cu_seqlens_q), kv, up(w.pre_page_table),
                                  up(w.pre_seq_lens), int(np.diff(w.cu_seqlens_q).max())))
    torch.cuda.synchronize()
    assert plan.status() == 0
    plan.close()
    return torch.cat(parts).contiguous()


def _shift16(t):
    """The same tensor at an address that is 16-byte but not 32-byte aligned."""
    import torch
    buf = torch.empty(t.numel() + 16, dtype=t.dtype, device=t.device)
    assert buf.data_ptr() % 32 == 0 and t.element_size() == 2
    out = buf[8:8 + t.numel()].view(t.shape)
    out.copy_(t)
    assert out.data_ptr() % 32 == 16
    return out


def _run(w, G, seed, rows=None, launch_rows=None, k_shift16=False):
    """Attend over the workload's rows on the GPU (all of them, or the first
    ``launch_rows``); returns the outputs of the listed rows and the oracle's
    inputs for them.  k_shift16: the K cache at a 16-byte (not 32-byte)
    aligned address."""
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    kv = gpu_cache(w)
    ids_t = _ids(w, kv)
    req, pos = workloads.attend_rows(w)
    nl = req.size if launch_rows is None else launch_rows
    ids_t, req, pos = ids_t[:nl].contiguous(), req[:nl], pos[:nl]
    H = w.num_heads
    rng = np.random.Generator(np.random.PCG64(seed))
    q_np = workloads.attend_q(nl, H * G, rng)
    kc = workloads.attend_kv_fill(seed, 0, w.num_blocks, H, torch_dev())
    if k_shift16:
        kc = _shift16(kc)
    vc = workloads.attend_kv_fill(seed, 1, w.num_blocks, H, torch_dev())
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
    out = idx.sparse_attend(up(q_np.view(np.int16)), kc, vc, up(w.page_table), up(req), up(pos), ids_t, SCALE,
                            status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    got = out.cpu().numpy().astype(np.float64)
    ids_np = ids_t.cpu().numpy()
    sel = np.arange(nl) if rows is None else np.asarray(rows)
    return got[sel], (q_np[sel], req[sel], pos[sel], ids_np[sel])


def _oracle(w, G, seed, q, req, pos, ids):
    """Oracle output and bound over the pages the rows select only (the
    cache's other pages are never read)."""
    blocks = np.unique(np.concatenate([w.page_table[req[t], ids[t][ids[t] >= 0]] for t in range(req.size)]))
    remap = np.full(w.num_blocks, -1, np.int64)
    remap[blocks] = np.arange(blocks.size)
    kc = workloads.attend_kv_pages(seed, 0, blocks, w.num_heads)
    vc = workloads.attend_kv_pages(seed, 1, blocks, w.num_heads)
    table = np.where(w.page_table >= 0, remap[np.clip(w.page_table, 0, None)], -1)
    o, n = oat.attend(q, kc, vc, table, req, pos, ids, G, SCALE)
    b = oat.error_bound(q, kc, vc, table, req, pos, ids, G, SCALE, chain=64)
    return o, b, n


def _assert_close(got, o, b, label):
    err = np.abs(got - o)
    bad = err > b
    worst = float(np.max(err / np.maximum(b, 1e-300)))
    print(f"{label}: {got.size} elements, worst error / bound = {worst:.3g}")
    assert not np.any(bad), f"{label}: {int(bad.sum())} elements outside the bound"


@pytest.mark.parametrize("cfg,G", [(0, 1), (0, 4), (1, 1), (2, 2), (3, 1), (4, 8)])
def test_attend_matches_oracle_small(cfg, G):
    """Small versions of the named workloads (decode and prefill rows, ragged
    page tails, causal cut inside the local page, G query heads per KV
    head); every row checked."""
    w = workloads.config(cfg, small=True) if cfg else workloads.config(0)
    seed = 500 + cfg
    req, _ = workloads.attend_rows(w)
    rows = np.arange(req.size)
    if rows.size > 600:                                # keep the float64 oracle to seconds
        rows = np.random.Generator(np.random.PCG64(seed)).choice(rows.size, 600, replace=False)
    got, (q, req, pos, ids) = _run(w, G, seed, rows=rows)
    o, b, n = _oracle(w, G, seed, q, req, pos, ids)
    _assert_close(got, o, b, f"{w.name} G={G}")
    assert np.all(got[n == 0] == 0)


@pytest.mark.parametrize("G", [1, 4])
def test_attend_k_cache_16_byte_aligned(G):
    """A K cache at an address that is 16-byte but not 32-byte aligned (the
    kernel then reads each K row in sixteen 16-byte loads instead of eight
    32-byte ones, in the same order): the same outputs, bit for bit, as from
    the 32-byte aligned cache, and within the oracle's bound."""
    w = workloads.config(0)
    seed = 520
    got, (q, req, pos, ids) = _run(w, G, seed)
    got16, _ = _run(w, G, seed, k_shift16=True)
    assert np.array_equal(got, got16)
    o, b, n = _oracle(w, G, seed, q, req, pos, ids)
    _assert_close(got16, o, b, f"{w.name} G={G}, K cache 16-byte aligned")


def test_attend_edge_rows():
    """Rows with only -1 ids (all zeros), a single visible token (the local
    page's first position: o = that token's v), ids in any order, and an
    unreadable page (zeros and a status bit)."""
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    w = workloads.config(0)
    H, G = w.num_heads, 2
    s0, s1 = int(w.dec_seq_lens[0]), int(w.dec_seq_lens[1])
    req = np.array([0, 1, 1, 0], np.int32)
    pos = np.array([s0 - 1, 128 * 2, s1 - 5, s0 - 3], np.int32)
    T = req.size
    ids = np.full((T, H, 16), -1, np.int32)
    ids[0, :, 3] = pos[0] // 128                       # the local page only, at an odd slot
    ids[1, :, 7] = 2                                   # page 2, one visible token (its first)
    ids[3, :, [9, 2, 0]] = [[1], [pos[3] // 128], [3]]  # three pages in no particular order
    rng = np.random.Generator(np.random.PCG64(9))
    q = workloads.attend_q(T, H * G, rng)
    kc = workloads.attend_kv_fill(9, 0, w.num_blocks, H, torch_dev())
    vc = workloads.attend_kv_fill(9, 1, w.num_blocks, H, torch_dev())
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())

    def call(ids_np, table=w.page_table):
        status.zero_()
        return idx.sparse_attend(up(q.view(np.int16)), kc, vc, up(table), up(req), up(pos), up(ids_np),
                                 SCALE, status=status).cpu().numpy().astype(np.float64)

    out = call(ids)
    assert int(status.item()) == 0
    assert np.all(out[2] == 0)                         # a row with no page
    v_first = workloads.attend_kv_pages(9, 1, [w.page_table[req[1], 2]], H)[0, 0]
    assert np.array_equal(out[1], oat.bf16_value(v_first)[np.arange(H * G) // G])
    o, b, _ = _oracle(w, G, 9, q, req, pos, ids)
    _assert_close(out, o, b, "edge rows")
    # page 1 of request 0 (selected by every head of row 3 only) maps outside the cache
    table = w.page_table.copy()
    table[0, 1] = w.num_blocks + 7
    out_bad = call(ids, table)
    assert int(status.item()) == idx.STATUS_BAD_PAGE
    assert np.all(out_bad[3] == 0)
    assert np.array_equal(out_bad[:3], out[:3])
    # a request index outside the page table: that row's heads are zeros
    req_ok = req.copy()
    req[0] = 5
    out_bad = call(ids)
    req[:] = req_ok
    assert int(status.item()) == idx.STATUS_BAD_TABLE
    assert np.all(out_bad[0] == 0) and np.array_equal(out_bad[1:], out[1:])


def test_attend_long_mixed_decode_rows_sampled():
    """The long mixed step's decode rows (16 requests x 8 queries x 8 heads,
    131072-token contexts) in the launch configuration the benchmark times;
    64 sampled rows checked against the oracle."""
    w = workloads.config(4)
    nd = w.num_decode_rows
    rows = np.random.Generator(np.random.PCG64(45)).choice(nd, 64, replace=False)
    got, (q, req, pos, ids) = _run(w, 1, 45, rows=rows, launch_rows=nd)
    o, b, _ = _oracle(w, 1, 45, q, req, pos, ids)
    _assert_close(got, o, b, "long_mixed decode rows, sampled")


@pytest.mark.parametrize("G", [1, 2])
def test_attend_row_groups_repeats_and_bad_row(G):
    """Consecutive rows of one request (they share a row-group unit of up to
    8 / G rows), cut where the request changes and at multiples of 8 / G;
    ids shuffled, with a repeated id (counted once: a set of pages); then
    one row of a group with a page outside the cache: that row is zeros with
    a status bit, the group's other rows still match the oracle."""
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    w = workloads.config(1, small=True)
    H = w.num_heads
    seq = w.dec_seq_lens.astype(np.int64)
    req = np.array([1, 1, 1, 1, 1, 0, 0, 1, 1, 1, 3, 3], np.int32)
    back = np.array([1, 3, 129, 200, 7, 1, 64, 2, 1, 300, 1, 5])
    pos = (seq[req] - back).astype(np.int32)
    T = req.size
    rng = np.random.Generator(np.random.PCG64(77))
    ids = np.full((T, H, 16), -1, np.int32)
    for t in range(T):
        L = int(pos[t]) // 128
        for h in range(H):
            hist = rng.permutation(L)[: min(L, 12)]
            row = list(hist) + [L]
            if len(row) >= 2:
                row.append(row[len(row) // 2])              # a repeat
            row = row + [-1] * (16 - len(row))
            ids[t, h] = np.array(row, np.int32)[rng.permutation(16)]
    # page X of request 1: selected by row 2 only (every head), read nowhere else
    X = int(pos[2]) // 128 - 1
    for t in range(T):
        if req[t] == 1 and t != 2:
            ids[t][ids[t] == X] = -1
    for h in range(H):
        if X not in ids[2, h]:
            ids[2, h, int(np.nonzero(ids[2, h] == -1)[0][0])] = X
    q = workloads.attend_q(T, H * G, rng)
    kc = workloads.attend_kv_fill(78, 0, w.num_blocks, H, torch_dev())
    vc = workloads.attend_kv_fill(78, 1, w.num_blocks, H, torch_dev())
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())

    def call(table):
        status.zero_()
        return idx.sparse_attend(up(q.view(np.int16)), kc, vc, up(table), up(req), up(pos), up(ids), SCALE,
                                 status=status).cpu().numpy().astype(np.float64)

    out = call(w.page_table)
    assert int(status.item()) == 0
    o, b, _ = _oracle(w, G, 78, q, req, pos, ids)
    _assert_close(out, o, b, f"row groups G={G}")
    table = w.page_table.copy()
    table[1, X] = w.num_blocks + 3
    out_bad = call(table)
    assert int(status.item()) == idx.STATUS_BAD_PAGE
    assert np.all(out_bad[2] == 0)
    keep = np.arange(T) != 2
    _assert_close(out_bad[keep], o[keep], b[keep], f"row groups G={G}, one bad row")
