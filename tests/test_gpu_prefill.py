"""Prefill indexer on the GPU against the CPU oracle."""
import numpy as np
import pytest

import workloads
from oracle import indexer as oidx
from gpu_util import (assert_ids, assert_scores, gpu_cache, make_plan, oracle_cache, run_prefill,
                      torch_dev, up)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _check(w, kv_gpu=None, kv_ref=None, dbg=True):
    kv_gpu = gpu_cache(w) if kv_gpu is None else kv_gpu
    kv_ref = oracle_cache(w) if kv_ref is None else kv_ref
    plan = make_plan(w)
    out, sc = run_prefill(plan, w, kv_gpu, dbg=dbg)
    ref = oidx.prefill(w.q_prefill, w.cu_seqlens_q, kv_ref, w.pre_page_table, w.pre_seq_lens, w.num_heads)
    assert_ids(out, ref, w.name)
    if dbg:
        assert_scores(sc, ref, w.name)
    assert plan.status() == 0
    plan.close()


@pytest.mark.parametrize("idx", [3, 4])
def test_prefill_parity_small_workloads(idx):
    _check(workloads.config(idx, small=True))


@pytest.mark.parametrize("H", [1, 2, 4, 8])
def test_prefill_heads_ragged_and_context(H):
    """Tiles of 128/H tokens with ragged tails, prompts with and without
    context, prompts shorter than a page and shorter than a tile."""
    rng = np.random.Generator(np.random.PCG64(40 + H))
    ctx = [0, 0, 300, 128 * 9, 5, 128 * 4 - 1]
    new = [1, 129, 77, 530, 300, 2]
    seq = [c + n for c, n in zip(ctx, new)]
    w = workloads.make_workload(name=f"pre_H{H}", seed=40 + H, rng=rng, num_heads=H,
                                pre_seq_lens=seq, pre_query_lens=new, outlier_channels=4)
    _check(w)


def test_prefill_ties_take_lowest_ids():
    rng = np.random.Generator(np.random.PCG64(41))
    H = 8
    seq = np.array([128 * 40 + 3], np.int32)
    ql = np.array([700], np.int32)
    nb = 41
    kv = np.repeat(workloads.random_pages(1, rng), nb, axis=0)
    table = rng.permutation(nb).astype(np.int32)[None, :]
    q = workloads.random_q(700, H, rng)
    w = workloads.Workload("pre_ties", H, 0, np.zeros(0, np.int32), seq, ql, table, nb,
                           np.zeros((0, 128), np.uint16), np.zeros(0, np.int64), q)
    plan = make_plan(w)
    out, _ = run_prefill(plan, w, up(kv))
    for t in range(700):
        L = (int(seq[0]) - 700 + t) // 128
        want = list(range(min(15, L))) + [L] + [-1] * (15 - min(15, L))
        assert np.all(out[t] == np.array(want, np.int32)), (t, out[t])


def test_prefill_bad_page_gives_minus_one_rows():
    import sparse_attention_block_nvfp4_gb300 as idx
    rng = np.random.Generator(np.random.PCG64(42))
    w = workloads.make_workload(name="pre_bad", seed=42, rng=rng, num_heads=4,
                                pre_seq_lens=[900, 1500], pre_query_lens=[900, 600])
    kv = gpu_cache(w)
    kv_ref = oracle_cache(w)
    table = w.page_table.copy()
    table[1, 3] = w.num_blocks
    w.page_table = table
    plan = make_plan(w)
    out, _ = run_prefill(plan, w, kv)
    ref = oidx.prefill(w.q_prefill, w.cu_seqlens_q, kv_ref, w.pre_page_table, w.pre_seq_lens, 4)
    assert ref.bad[:900].sum() == 0 and ref.bad[900:].all()
    assert_ids(out, ref, "bad page")
    assert plan.status() & idx.STATUS_BAD_PAGE


@pytest.mark.parametrize("idx", [3, 4])
def test_prefill_full_size_sampled(idx):
    """Full-size ragged prefill / long-context chunks as the benchmark runs
    them; a sample of rows of every request checked against the oracle."""
    w = workloads.config(idx)
    kv = gpu_cache(w)
    plan = make_plan(w)
    out, _ = run_prefill(plan, w, kv)
    assert plan.status() == 0
    nd = w.num_decode_reqs
    kv_ref = oracle_cache(w, list(range(nd, nd + w.num_prefill_reqs)))
    rng = np.random.Generator(np.random.PCG64(300 + idx))
    cu = w.cu_seqlens_q
    rows = []
    for r in range(w.num_prefill_reqs):
        a, b = int(cu[r]), int(cu[r + 1])
        rows += [a, b - 1] + rng.integers(a, b, size=48).tolist()
    rows = np.unique(np.array(rows))
    ref = oidx.prefill(w.q_prefill, cu, kv_ref, w.pre_page_table, w.pre_seq_lens, w.num_heads, rows=rows)
    assert_ids(out[rows], ref, w.name)


@pytest.mark.parametrize("H", [1, 8])
def test_prefill_tile_pairs_every_row(H):
    """Many tiles per request: the kernel forms pairs of consecutive query
    tiles (one dequantised page multiplied against both) and takes each
    request's odd tile as a single; every row checked against the oracle."""
    rng = np.random.Generator(np.random.PCG64(60 + H))
    tq = 128 // H
    nreq = 160 if H == 1 else 40
    tiles = rng.integers(1, 5, size=nreq) if H == 1 else rng.integers(6, 11, size=nreq)
    ql = [int(t) * tq - int(rng.integers(0, tq // 2 + 1)) for t in tiles]
    ctx = [int(c) for c in rng.choice([0, 0, 37, 128, 300, 1000], size=nreq)]
    seq = [c + n for c, n in zip(ctx, ql)]
    w = workloads.make_workload(name=f"pairs_H{H}", seed=60 + H, rng=rng, num_heads=H,
                                pre_seq_lens=seq, pre_query_lens=ql, outlier_channels=4)
    assert sum((n + tq - 1) // tq for n in ql) >= 2 * 152
    _check(w)


@pytest.mark.parametrize("H", [2, 8])
def test_prefill_units_cut_across_ctas(H):
    """Few units with long histories next to empty and one-token prompts: the
    even split by pages cuts most units over several CTAs (each leaves its
    top-15 candidates, merged afterwards in page order) and leaves some CTAs a
    range with no page at all; every row checked against the oracle."""
    rng = np.random.Generator(np.random.PCG64(70 + H))
    ctx = [20000, 0, 5000, 0, 130 * 128, 127, 0]
    new = [700, 0, 3, 1, 260, 1, 129]
    seq = [c + n for c, n in zip(ctx, new)]
    w = workloads.make_workload(name=f"cut_H{H}", seed=70 + H, rng=rng, num_heads=H,
                                pre_seq_lens=seq, pre_query_lens=new, outlier_channels=4)
    _check(w)
