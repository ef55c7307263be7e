"""Decode indexer on the GPU against the CPU oracle (ids modulo score ties,
debug scores within 1e-5 * sum|q k|)."""
import numpy as np
import pytest

import workloads
from oracle import indexer as oidx
from gpu_util import (assert_ids, assert_scores, gpu_cache, make_plan, oracle_cache, run_decode,
                      torch_dev, up)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _check_workload(w, kv_gpu=None, kv_ref=None, dbg=True):
    kv_gpu = gpu_cache(w) if kv_gpu is None else kv_gpu
    kv_ref = oracle_cache(w) if kv_ref is None else kv_ref
    plan = make_plan(w)
    out, sc = run_decode(plan, w, kv_gpu, dbg=dbg)
    ref = oidx.decode(w.q_decode, kv_ref, w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads)
    rep = assert_ids(out, ref, w.name)
    if dbg:
        assert_scores(sc, ref, w.name)
    assert plan.status() == 0
    plan.close()
    return rep


@pytest.mark.parametrize("idx", [0, 1, 2, 4])
def test_decode_parity_small_workloads(idx):
    w = workloads.config(idx, small=(idx != 0))
    _check_workload(w)


@pytest.mark.parametrize("H,qlen", [(1, 1), (1, 8), (2, 3), (4, 1), (4, 5), (8, 1), (8, 2), (8, 4), (8, 7), (8, 8)])
def test_decode_heads_and_query_lengths(H, qlen):
    """Every rows-per-request shape (R = qlen*H -> MMA N of 16, 32, 64), with
    queries straddling page boundaries, padding requests and short requests."""
    rng = np.random.Generator(np.random.PCG64(100 + 10 * H + qlen))
    seq = [qlen - 1, 0, 5, 128, 129, 130 + qlen, 128 * 7 + 3, 128 * 16 + qlen - 2, 128 * 23, 1777]
    seq = [max(0, s) for s in seq] + list(rng.integers(200, 3000, size=6))
    w = workloads.make_workload(name=f"dec_H{H}_q{qlen}", seed=1, rng=rng, num_heads=H,
                                dec_seq_lens=seq, query_len=qlen, outlier_channels=4)
    _check_workload(w)


@pytest.mark.parametrize("H,qlen", [(8, 4), (4, 1), (2, 4)])
def test_decode_arbitrary_page_bytes(H, qlen):
    """Pages of arbitrary bytes (all finite scales, subnormal scales included):
    exercises the exact fp16 dequantisation beyond what the insert produces,
    on the quad kernel (32 rows) and the small-row path (4 and 8 rows)."""
    rng = np.random.Generator(np.random.PCG64(31 + H + qlen))
    seq = np.array([128 * 40 + 7, 128 * 3 + 1, 128 * 17], np.int32)
    nb = 70
    table = np.zeros((3, 41), np.int32)
    perm = rng.permutation(nb)
    off = 0
    for r, s in enumerate(seq):
        npg = (s + 127) // 128
        table[r, :npg] = perm[off:off + npg]
        off += npg
    kv = workloads.random_pages(nb, rng)
    q = workloads.random_q(3 * qlen, H, rng)
    w = workloads.Workload(name="arb_bytes", num_heads=H, query_len=qlen, dec_seq_lens=seq,
                           pre_seq_lens=np.zeros(0, np.int32), pre_query_lens=np.zeros(0, np.int32),
                           page_table=table, num_blocks=nb, k_bf16=np.zeros((0, 128), np.uint16),
                           slot_mapping=np.zeros(0, np.int64), q_e4m3=q)
    _check_workload(w, kv_gpu=up(kv), kv_ref=kv)


@pytest.mark.parametrize("H,qlen", [(4, 2), (8, 4), (8, 8)])
def test_decode_ties_take_lowest_ids_across_splits(H, qlen):
    """Identical pages: every score ties, so every row must be [0..14, L]
    exactly, also when a long request is split across many split units
    (warps of the small-row kernel for 8 rows, CTAs of the quad kernel for
    32 and 64)."""
    rng = np.random.Generator(np.random.PCG64(32))
    seq = np.array([128 * 3000 + 77, 128 * 20 + 1, 128 * 900], np.int32)
    pages = (seq + 127) // 128
    nb = int(pages.sum())
    one = workloads.random_pages(1, rng)
    kv = np.repeat(one, nb, axis=0)
    table = np.zeros((3, int(pages.max())), np.int32)
    perm = rng.permutation(nb)
    off = 0
    for r in range(3):
        table[r, :pages[r]] = perm[off:off + pages[r]]
        off += pages[r]
    q = workloads.random_q(3 * qlen, H, rng)
    plan = make_plan(workloads.Workload("ties", H, qlen, seq, np.zeros(0, np.int32), np.zeros(0, np.int32),
                                        table, nb, np.zeros((0, 128), np.uint16), np.zeros(0, np.int64), q))
    out = plan.decode(up(q), up(kv), up(table), up(seq), qlen).cpu().numpy()
    for r in range(3):
        for i in range(qlen):
            L = (int(seq[r]) - qlen + i) // 128
            want = list(range(min(15, L))) + [L] + [-1] * (15 - min(15, L))
            assert np.all(out[r * qlen + i] == np.array(want, np.int32)), (r, i, out[r * qlen + i])


@pytest.mark.parametrize("H,qlen", [(8, 8), (4, 1), (8, 1)])
def test_decode_one_long_request_many_splits(H, qlen):
    """One request spread over every split unit: more than 32 CTAs of the
    quad kernel (64 rows), or more than 64 warps of the small-row kernel (4
    and 8 rows: about one page a warp, so the merge folds the lists beyond
    the 64 a warp holds)."""
    rng = np.random.Generator(np.random.PCG64(33))
    w = workloads.make_workload(name=f"one_long_H{H}_q{qlen}", seed=33, rng=rng, num_heads=H,
                                dec_seq_lens=[128 * 1500 + 9], query_len=qlen, outlier_channels=4,
                                page_scale_spread=6.0)
    _check_workload(w)


def test_decode_bad_page_id_gives_minus_one_rows_and_status():
    import sparse_attention_block_nvfp4_gb300 as idx
    rng = np.random.Generator(np.random.PCG64(34))
    w = workloads.make_workload(name="bad", seed=34, rng=rng, num_heads=4,
                                dec_seq_lens=[128 * 5 + 3, 128 * 900 + 1, 128 * 3], query_len=2)
    kv = gpu_cache(w)
    kv_ref = oracle_cache(w)
    table = w.page_table.copy()
    table[0, 2] = w.num_blocks + 5          # request 0: out of range
    table[1, 700] = -3                      # request 1 (split over CTAs): negative
    w.page_table = table
    plan = make_plan(w)
    out, _ = run_decode(plan, w, kv)
    ref = oidx.decode(w.q_decode, kv_ref, table, w.dec_seq_lens, w.query_len, w.num_heads)
    assert ref.bad.tolist() == [True, True, True, True, False, False]
    assert_ids(out, ref, "bad page")
    assert plan.status() & idx.STATUS_BAD_PAGE
    # a history wider than the page table
    plan2 = make_plan(w)
    narrow = np.ascontiguousarray(table[:, :4])
    out2 = plan2.decode(up(w.q_decode), kv, up(narrow), up(w.dec_seq_lens), w.query_len).cpu().numpy()
    ref2 = oidx.decode(w.q_decode, kv_ref, narrow, w.dec_seq_lens, w.query_len, w.num_heads)
    assert_ids(out2, ref2, "narrow table")
    assert plan2.status() & idx.STATUS_BAD_TABLE


def test_decode_cuda_graph_replay():
    """Captured once, replayed after the batch's seq_lens / page table change
    in place (the decode wrappers re-plan outside capture every step)."""
    import torch
    rng = np.random.Generator(np.random.PCG64(35))
    H, qlen, nreq = 8, 4, 12
    seq0 = rng.integers(1000, 9000, size=nreq).astype(np.int32)
    w = workloads.make_workload(name="graph", seed=35, rng=rng, num_heads=H, dec_seq_lens=seq0 + 400,
                                query_len=qlen, outlier_channels=4)
    kv = gpu_cache(w)
    kv_ref = oracle_cache(w)
    plan = make_plan(w)
    q_t, kv_t = up(w.q_decode), kv
    table_t, seq_t = up(w.dec_page_table), up(seq0)
    out_t = torch.empty((nreq * qlen, H, 16), dtype=torch.int32, device=torch_dev())
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        plan.decode(q_t, kv_t, table_t, seq_t, qlen, out=out_t, stream=s)   # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        plan.decode(q_t, kv_t, table_t, seq_t, qlen, out=out_t, stream=s)
    for step in range(3):
        seq = (seq0 + 137 * step).astype(np.int32)
        seq_t.copy_(up(seq))
        out_t.fill_(-99)
        g.replay()
        torch.cuda.synchronize()
        ref = oidx.decode(w.q_decode, kv_ref, w.dec_page_table, seq, qlen, H)
        assert_ids(out_t.cpu().numpy(), ref, f"graph replay {step}")


@pytest.mark.parametrize("idx", [1, 2, 4])
def test_decode_full_size_sampled(idx):
    """The full-size workload, in the launch configuration the benchmark times;
    every row of a sample of requests checked against the oracle."""
    w = workloads.config(idx)
    kv = gpu_cache(w)
    plan = make_plan(w)
    out, _ = run_decode(plan, w, kv)
    assert plan.status() == 0
    rng = np.random.Generator(np.random.PCG64(200 + idx))
    reqs = sorted(rng.choice(w.num_decode_reqs, size=min(3, w.num_decode_reqs), replace=False).tolist())
    kv_ref = oracle_cache(w, reqs)
    rows = np.concatenate([np.arange(r * w.query_len, (r + 1) * w.query_len) for r in reqs])
    ref = oidx.decode(w.q_decode, kv_ref, w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads,
                      rows=rows)
    assert_ids(out[rows], ref, w.name)
    # every row obeys the structure (local page last, -1 tail, distinct ids < L)
    pos = np.repeat(w.dec_seq_lens, w.query_len) - w.query_len + np.tile(np.arange(w.query_len), w.num_decode_reqs)
    L = pos // 128
    m = np.minimum(15, L)
    for t in range(0, out.shape[0], max(1, out.shape[0] // 512)):
        for h in range(w.num_heads):
            o = out[t, h]
            assert o[m[t]] == L[t] and np.all(o[m[t] + 1:] == -1)
            assert len(set(o[:m[t]].tolist())) == m[t] and np.all(o[:m[t]] < L[t]) and np.all(o[:m[t]] >= 0)


def test_decode_small_batch_after_wide_batch_same_plan():
    """A batch with fewer history pages than CTAs, run on a plan whose scratch
    still holds a previous, wider batch's candidates: every candidate slot the
    merge reads must have been written by the current call."""
    rng = np.random.Generator(np.random.PCG64(36))
    wide = workloads.make_workload(name="wide", seed=36, rng=rng, num_heads=8,
                                   dec_seq_lens=rng.integers(3000, 9000, size=16), query_len=8)
    small = workloads.make_workload(name="small", seed=37, rng=np.random.Generator(np.random.PCG64(37)),
                                    num_heads=8, dec_seq_lens=[2000, 3100, 700, 129, 4000], query_len=2)
    import sparse_attention_block_nvfp4_gb300 as idx
    plan = idx.Plan(num_heads=8, max_reqs=16, max_query_len=8,
                    max_pages_per_req=max(wide.page_table.shape[1], small.page_table.shape[1]))
    for w in (wide, small, wide, small):
        out, _ = run_decode(plan, w, gpu_cache(w))
        ref = oidx.decode(w.q_decode, oracle_cache(w), w.dec_page_table, w.dec_seq_lens, w.query_len, 8)
        assert_ids(out, ref, w.name)
    assert plan.status() == 0


@pytest.mark.parametrize("H,qlen", [(2, 3), (8, 4), (8, 8)])
def test_decode_partial_quads_and_split_segments(H, qlen):
    """Many short requests: every CTA walks several segments, most of them
    starting inside a request, and ends of segments leave partial groups of
    1, 2 or 3 pages (the kernel takes pages four at a time)."""
    rng = np.random.Generator(np.random.PCG64(500 + H * 10 + qlen))
    hist = np.concatenate([np.arange(1, 14), rng.integers(1, 14, size=67), [41, 42, 43, 45]])
    rng.shuffle(hist)
    seq = 128 * hist + rng.integers(1, 129, size=hist.size)     # history = hist pages exactly
    w = workloads.make_workload(name=f"quads_H{H}_q{qlen}", seed=5, rng=rng, num_heads=H,
                                dec_seq_lens=seq, query_len=qlen, outlier_channels=4)
    _check_workload(w)
