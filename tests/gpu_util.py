"""Helpers for the GPU parity tests: run a workload through the C ABI (via
the binding) and build the oracle's view of the same seeded inputs."""
from __future__ import annotations

import numpy as np

import workloads
from oracle import nvfp4 as onvfp4


def torch_dev():
    import torch
    return torch.device("cuda:0")


def up(a):
    import torch
    return torch.from_numpy(np.ascontiguousarray(a)).to(torch_dev())


def gpu_cache(w: workloads.Workload, num_blocks=None):
    """The workload's cache written by the CUDA insert kernel."""
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    nb = num_blocks or w.num_blocks
    kv = torch.zeros((nb, 128, 72), dtype=torch.uint8, device=torch_dev())
    idx.insert(up(w.k_bf16.view(np.int16)), up(w.slot_mapping), kv)
    return kv


def oracle_cache(w: workloads.Workload, reqs=None) -> np.ndarray:
    """The oracle's cache: every token (reqs None), or only the tokens of the
    listed requests (decode requests first, then prefill requests)."""
    kv = np.zeros((w.num_blocks, 128, 72), np.uint8)
    if reqs is None:
        return onvfp4.insert(w.k_bf16, w.slot_mapping, kv)
    seq = w.seq_lens.astype(np.int64)
    start = np.concatenate([[0], np.cumsum(np.maximum(seq, 0))])
    for r in reqs:
        a, b = int(start[r]), int(start[r + 1])
        onvfp4.insert(w.k_bf16[a:b], w.slot_mapping[a:b], kv)
    return kv


def make_plan(w: workloads.Workload, **kw):
    import sparse_attention_block_nvfp4_gb300 as idx
    return idx.Plan(num_heads=w.num_heads, max_reqs=max(1, w.num_decode_reqs),
                    max_query_len=max(1, w.query_len), max_pages_per_req=w.page_table.shape[1],
                    max_prefill_tokens=max(1, w.total_prefill_q), max_prefill_reqs=max(1, w.num_prefill_reqs),
                    **kw)


def run_decode(plan, w, kv, dbg=False, stream=None):
    import torch
    dbg_t = None
    if dbg:
        dbg_t = torch.full((w.num_decode_rows, w.num_heads, w.page_table.shape[1]), float("nan"),
                           dtype=torch.float32, device=torch_dev())
    out = plan.decode(up(w.q_decode), kv, up(w.dec_page_table), up(w.dec_seq_lens), w.query_len,
                      scores_dbg=dbg_t, stream=stream)
    return out.cpu().numpy(), (dbg_t.cpu().numpy() if dbg else None)


def run_prefill(plan, w, kv, dbg=False):
    import torch
    dbg_t = None
    if dbg:
        dbg_t = torch.full((w.total_prefill_q, w.num_heads, w.page_table.shape[1]), float("nan"),
                           dtype=torch.float32, device=torch_dev())
    out = plan.prefill(up(w.q_prefill), up(w.cu_seqlens_q), kv, up(w.pre_page_table), up(w.pre_seq_lens),
                       int(w.pre_query_lens.max()), scores_dbg=dbg_t)
    return out.cpu().numpy(), (dbg_t.cpu().numpy() if dbg else None)


def assert_ids(out, ref, what=""):
    from oracle import checker
    rep = checker.check_ids(out, ref)
    assert rep["fails"] == 0, f"{what}: {rep}"
    return rep


def assert_scores(dbg, ref, what=""):
    from oracle import checker
    rep = checker.check_scores(dbg, ref)
    assert rep["fails"] == 0, f"{what}: {rep}"
    return rep
