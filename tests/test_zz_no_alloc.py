"""indexer_decode_noalloc: the decode entry point for callers that cannot
allocate device memory.

A caller such as a custom-op hook inside a serving engine (handed only its
input and output buffers, the engine owning all device memory) or a
latency-critical loop that must never call cudaMalloc cannot create a plan,
because the plan allocates its scratch.  indexer_decode_noalloc runs the same
kernels with their scratch in a fixed array inside the library.  These tests
call it through the C ABI (ctypes, no binding helper) and compare it with
indexer_decode on the same inputs, on two calls in a row, so a call that
depends on what the previous call left in the shared array would show up.
The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import workloads
from oracle import indexer as oidx
from gpu_util import assert_ids, gpu_cache, make_plan, oracle_cache, torch_dev, up

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def lib():
    import __graft_entry__
    import sparse_attention_block_nvfp4_gb300 as idx
    __graft_entry__.build()
    L = idx.load_library()
    P, I = ctypes.c_void_p, ctypes.c_int
    L.indexer_decode_noalloc.argtypes = [P, P, I, P, I, P, I, I, I, P, P, P]
    L.indexer_decode_noalloc.restype = I
    return L


def _call(lib, w, kv, out, status):
    import torch
    q, table, seq = up(w.q_decode), up(w.dec_page_table), up(w.dec_seq_lens)
    stream = torch.cuda.current_stream()
    rc = lib.indexer_decode_noalloc(q.data_ptr(), kv.data_ptr(), int(kv.shape[0]), table.data_ptr(),
                                    int(table.shape[1]), seq.data_ptr(), w.num_decode_reqs, w.query_len,
                                    w.num_heads, out.data_ptr(), status.data_ptr(), stream.cuda_stream)
    torch.cuda.synchronize()
    return rc


def test_noalloc_matches_indexer_decode_on_two_calls_in_a_row(lib):
    import torch
    cases = [workloads.config(2, small=True),                       # 8 heads x 4 queries, split requests
             workloads.config(1, small=True)]                       # 4 heads x 1 query
    for w in cases:
        kv = gpu_cache(w)
        plan = make_plan(w)
        want = plan.decode(up(w.q_decode), kv, up(w.dec_page_table), up(w.dec_seq_lens), w.query_len)
        torch.cuda.synchronize()
        out = torch.full((w.num_decode_rows, w.num_heads, 16), -77, dtype=torch.int32, device=torch_dev())
        status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
        assert _call(lib, w, kv, out, status) == 0, lib.indexer_last_error()
        assert int(status.item()) == 0
        got = out.cpu().numpy()
        assert np.array_equal(got, want.cpu().numpy()), f"{w.name}: differs from indexer_decode"
        ref = oidx.decode(w.q_decode, oracle_cache(w), w.dec_page_table, w.dec_seq_lens, w.query_len,
                          w.num_heads)
        assert_ids(got, ref, w.name)
        plan.close()


def _call_raw(lib, q, kv, table, seq, num_reqs, query_len, num_heads, out, status):
    import torch
    stream = torch.cuda.current_stream()
    rc = lib.indexer_decode_noalloc(q.data_ptr(), kv.data_ptr(), int(kv.shape[0]), table.data_ptr(),
                                    int(table.shape[1]), seq.data_ptr(), num_reqs, query_len, num_heads,
                                    out.data_ptr(), status.data_ptr() if status is not None else None,
                                    stream.cuda_stream)
    torch.cuda.synchronize()
    return rc


def test_noalloc_same_layout_new_data_and_null_status(lib):
    """Two calls with the same shape (so the second reuses exactly the parts
    of the array the first wrote), the second with other queries and another
    page table over the same cache, checked against the oracle; then the
    same call with status NULL."""
    import torch
    w = workloads.config(2, small=True)
    kv = gpu_cache(w)
    cache = oracle_cache(w)
    rng = np.random.Generator(np.random.PCG64(78))
    out = torch.empty((w.num_decode_rows, w.num_heads, 16), dtype=torch.int32, device=torch_dev())
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
    seq = up(w.dec_seq_lens)
    calls = [(w.q_decode, w.dec_page_table)]
    table2 = w.dec_page_table.copy()
    for r in range(table2.shape[0]):                 # another valid table: each row's pages permuted
        n = int((w.dec_seq_lens[r] + 127) // 128)
        table2[r, :n] = table2[r, :n][rng.permutation(n)]
    calls.append((workloads.random_q(w.num_decode_rows, w.num_heads, rng), table2))
    for q_np, t_np in calls:
        out.fill_(-77)
        assert _call_raw(lib, up(q_np), kv, up(t_np), seq, w.num_decode_reqs, w.query_len, w.num_heads, out,
                         status) == 0, lib.indexer_last_error()
        assert int(status.item()) == 0
        ref = oidx.decode(q_np, cache, t_np, w.dec_seq_lens, w.query_len, w.num_heads)
        assert_ids(out.cpu().numpy(), ref, "same layout, new data")
    out.fill_(-77)
    assert _call_raw(lib, up(q_np), kv, up(t_np), seq, w.num_decode_reqs, w.query_len, w.num_heads, out,
                     None) == 0, lib.indexer_last_error()
    assert_ids(out.cpu().numpy(), ref, "status NULL")


def test_noalloc_bad_page_with_null_status_gives_empty_rows(lib):
    """An unreadable page id in one request's history: with status NULL the
    call still returns its rows, -1 for that request, exact for the others."""
    import torch
    w = workloads.config(1, small=True)
    kv = gpu_cache(w)
    table = w.dec_page_table.copy()
    table[2, 1] = w.num_blocks + 5                   # request 2 reads past the cache
    ref = oidx.decode(w.q_decode, oracle_cache(w), table, w.dec_seq_lens, w.query_len, w.num_heads)
    assert ref.bad[2 * w.query_len]
    out = torch.full((w.num_decode_rows, w.num_heads, 16), -77, dtype=torch.int32, device=torch_dev())
    assert _call_raw(lib, up(w.q_decode), kv, up(table), up(w.dec_seq_lens), w.num_decode_reqs, w.query_len,
                     w.num_heads, out, None) == 0, lib.indexer_last_error()
    got = out.cpu().numpy()
    assert np.all(got[2 * w.query_len:3 * w.query_len] == -1)
    assert_ids(got, ref, "bad page, status NULL")


def test_noalloc_rejects_calls_beyond_its_fixed_scratch(lib):
    import torch
    rng = np.random.Generator(np.random.PCG64(77))
    w = workloads.make_workload(name="too_many", seed=77, rng=rng, num_heads=8,
                                dec_seq_lens=[300] * 600, query_len=8)
    kv = torch.zeros((w.num_blocks, 128, 72), dtype=torch.uint8, device=torch_dev())
    out = torch.zeros((w.num_decode_rows, 8, 16), dtype=torch.int32, device=torch_dev())
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
    import sparse_attention_block_nvfp4_gb300 as idx
    assert _call(lib, w, kv, out, status) == idx.IDX_ENOSPACE
    assert b"scratch" in lib.indexer_last_error()
