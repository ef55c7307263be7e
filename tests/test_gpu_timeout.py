"""Bounded waits inside the decode and prefill kernels: a plan whose wait
limit is a few nanoseconds makes the waits between the kernels' roles run
out on an ordinary small call.  The call must still return, report
IDX_STATUS_TIMEOUT (or, if no wait ever had to block, produce the oracle's
rows), leave every row either exact or all -1, and leave the plan usable: a
following call with the default limit is correct.  Nothing here faults or
hangs a GPU: a wait that runs out sets a status bit, the kernel drains its
own copies and tensor-core work and frees its tensor memory."""
import numpy as np
import pytest

import workloads
from oracle import checker
from oracle import indexer as oidx
from gpu_util import assert_ids, gpu_cache, make_plan, oracle_cache, up

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _rows_exact_or_empty(got, ref, label):
    """Every (row, head) is all -1 or passes the oracle's check."""
    rep = checker.check_ids(got, ref, max_report=got.shape[0] * got.shape[1])
    for r, h, why, g in rep["examples"]:
        assert all(x == -1 for x in g), f"{label}: row {r} head {h} is neither -1 nor the oracle's ({why})"
    empty = int(np.all(got == -1, axis=2).sum())
    return got.shape[0] * got.shape[1] - empty, empty


@pytest.mark.parametrize("cfg,rows", [(4, 64), (2, 32), (1, 4)],
                         ids=["quad_kernel_rows64", "quad_kernel_rows32", "small_row_kernel_rows4"])
def test_decode_wait_limit_runs_out_then_recovers(cfg, rows):
    """Decode with 1 ns waits: on the quad kernel (64 and 32 rows per
    request, its waits are the hand-offs between roles) and on the small-row
    kernel (4 rows per request, its waits are on the page copies of each
    warp's ring)."""
    import sparse_attention_block_nvfp4_gb300 as idx
    w = workloads.config(cfg, small=True)
    assert w.query_len * w.num_heads == rows
    kv = gpu_cache(w)
    ref = oidx.decode(w.q_decode, oracle_cache(w), w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads)
    plan = make_plan(w)
    plan.set_wait_limit(1)
    out = plan.decode(up(w.q_decode), kv, up(w.dec_page_table), up(w.dec_seq_lens), w.query_len)
    st = plan.status()
    got = out.cpu().numpy()
    if st & idx.STATUS_TIMEOUT:
        done, empty = _rows_exact_or_empty(got, ref, "decode, 1 ns waits")
        print(f"decode with 1 ns waits: timeout reported, {done} rows exact, {empty} rows -1")
    else:
        assert st == 0
        assert_ids(got, ref, "decode, 1 ns waits (no wait had to block)")
    plan.set_wait_limit(0)
    out = plan.decode(up(w.q_decode), kv, up(w.dec_page_table), up(w.dec_seq_lens), w.query_len)
    assert_ids(out.cpu().numpy(), ref, "decode after restoring the limit")
    assert plan.status() == 0
    plan.close()


def test_prefill_wait_limit_runs_out_then_recovers():
    import sparse_attention_block_nvfp4_gb300 as idx
    w = workloads.config(3, small=True)
    kv = gpu_cache(w)
    ref = oidx.prefill(w.q_prefill, w.cu_seqlens_q, oracle_cache(w), w.pre_page_table, w.pre_seq_lens,
                       w.num_heads)
    plan = make_plan(w)

    def call():
        return plan.prefill(up(w.q_prefill), up(w.cu_seqlens_q), kv, up(w.pre_page_table), up(w.pre_seq_lens),
                            int(np.diff(w.cu_seqlens_q).max())).cpu().numpy()

    plan.set_wait_limit(1)
    got = call()
    st = plan.status()
    if st & idx.STATUS_TIMEOUT:
        done, empty = _rows_exact_or_empty(got, ref, "prefill, 1 ns waits")
        print(f"prefill with 1 ns waits: timeout reported, {done} rows exact, {empty} rows -1")
    else:
        assert st == 0
        assert_ids(got, ref, "prefill, 1 ns waits (no wait had to block)")
    plan.set_wait_limit(0)
    assert_ids(call(), ref, "prefill after restoring the limit")
    assert plan.status() == 0
    plan.close()
