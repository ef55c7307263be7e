"""Decode context parallelism on one GPU: `world` ranks are emulated by
indexer_decode_partial calls over disjoint page ranges of the same cache
(one after another: no kernel waits on another), their candidates stacked
rank-major and merged by indexer_merge_candidates; the rows must be the
whole-history oracle rows, and each share's candidates the oracle's."""
import numpy as np
import pytest

import workloads
from oracle import indexer as oidx
from oracle import mxfp4 as omx
from gpu_util import assert_ids, gpu_cache, make_plan, oracle_cache, torch_dev, up

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _bounds(w, world, rng):
    hist = np.maximum(w.dec_seq_lens.astype(np.int64) - 1, 0) // 128
    cuts = np.sort(rng.integers(0, hist[:, None] + 1, size=(len(hist), world - 1)), axis=1)
    return np.concatenate([np.zeros((len(hist), 1), np.int64), cuts, hist[:, None]], axis=1)


def _run(w, pages, ref, world, seed, page_format="nvfp4"):
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    rng = np.random.Generator(np.random.PCG64(seed))
    b = _bounds(w, world, rng)
    plan = make_plan(w)
    q, table, seq = up(w.q_decode), up(w.dec_page_table), up(w.dec_seq_lens)
    cands = []
    for k in range(world):
        lo, hi = b[:, k].astype(np.int32), b[:, k + 1].astype(np.int32)
        c = plan.decode_partial(q, pages, table, seq, up(lo), up(hi), w.query_len, page_format=page_format)
        cands.append(c)
        ids = c[..., 1].contiguous().view(torch.int32).cpu().numpy()
        sc = c[..., 0].cpu().numpy().astype(np.float64)
        want_ids, want_sc = oidx.partial_candidates(ref, lo, hi, w.query_len)
        assert np.array_equal(ids, want_ids), f"rank {k} of {world}: candidate ids"
        ok = want_ids >= 0
        # the score band |S_gpu - S| <= 1e-5 * A, A = max over the page's
        # tokens of sum |q_i k_i| (the oracle's tolerance)
        A = np.take_along_axis(ref.A[:, :, :], np.maximum(want_ids, 0).astype(np.int64), axis=2)
        assert np.all(np.abs(sc[ok] - want_sc[ok]) <= 1e-5 * A[ok])
    out = idx.merge_candidates(torch.stack(cands), seq, w.query_len, w.num_heads)
    assert_ids(out.cpu().numpy(), ref, f"{w.name} world {world}")
    assert plan.status() == 0
    plan.close()


@pytest.mark.parametrize("idx,world", [(1, 2), (2, 3), (4, 4), (2, 1)])
def test_cp_emulated_ranks_nvfp4(idx, world):
    w = workloads.config(idx, small=True)
    ref = oidx.decode(w.q_decode, oracle_cache(w), w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads)
    _run(w, gpu_cache(w), ref, world, seed=300 + idx)


def test_cp_emulated_ranks_mxfp4():
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    w = workloads.config(2, small=True)
    pages = torch.zeros((w.num_blocks, omx.PAGE_BYTES), dtype=torch.uint8, device=torch_dev())
    idx.mxfp4_insert(up(w.k_bf16.view(np.int16)), up(w.slot_mapping), pages)
    ref_pages = omx.insert(w.k_bf16, w.slot_mapping, np.zeros((w.num_blocks, omx.PAGE_BYTES), np.uint8))
    ref = oidx.decode(w.q_decode, ref_pages, w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads,
                      page_format="mxfp4")
    _run(w, pages, ref, 3, seed=310, page_format="mxfp4")


def test_cp_unreadable_page_in_one_share():
    """A page id outside the cache inside one rank's range: that rank marks
    the request, the merge writes its rows as -1 and flags the status."""
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    w = workloads.config(1, small=True)
    kv = gpu_cache(w)
    table = w.dec_page_table.copy()
    hist = (w.dec_seq_lens.astype(np.int64) - 1) // 128
    table[0, hist[0] - 1] = w.num_blocks + 3                 # last history page of request 0
    plan = make_plan(w)
    q, seq = up(w.q_decode), up(w.dec_seq_lens)
    lo0 = np.zeros_like(hist, dtype=np.int32)
    mid = (hist // 2).astype(np.int32)
    hi1 = hist.astype(np.int32)
    c0 = plan.decode_partial(q, kv, up(table), seq, up(lo0), up(mid), w.query_len)
    c1 = plan.decode_partial(q, kv, up(table), seq, up(mid), up(hi1), w.query_len)
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
    out = idx.merge_candidates(torch.stack([c0, c1]), seq, w.query_len, w.num_heads, status=status).cpu().numpy()
    rows0 = out[: w.query_len]
    assert np.all(rows0 == -1)
    assert int(status.item()) & 1
    ref = oidx.decode(w.q_decode, oracle_cache(w), w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads)
    assert np.array_equal(out[w.query_len:], ref.out[w.query_len:])
    assert plan.status() & 1                                 # the scoring kernel flagged the page too
    plan.close()
