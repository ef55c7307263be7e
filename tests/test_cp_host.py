"""Decode context parallelism, host side, on CPU: two gloo ranks each hold
one page range of every request, pack their candidates in the layout
indexer_decode_partial writes, exchange them with the library's
gather_candidates (the one collective of the path), and the merge of the
gathered, rank-major tensor gives the whole-history rows (oracle merge; the
GPU merge kernel is checked against the same rows in test_gpu_cp.py)."""
import os

import numpy as np
import torch
import torch.distributed as tdist
import torch.multiprocessing as mp

import workloads
from oracle import indexer, nvfp4


def _workload():
    w = workloads.config(2, small=True)
    kv = nvfp4.insert(w.k_bf16, w.slot_mapping, np.zeros((w.num_blocks, 128, 72), np.uint8))
    res = indexer.decode(w.q_decode, kv, w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads)
    hist = (w.dec_seq_lens.astype(np.int64) - 1) // 128
    mid = (hist * np.array([1, 3, 1, 2, 0, 5])[: len(hist)]) // 5      # uneven, some empty shares
    bounds = [(np.zeros_like(hist), mid), (mid, hist)]
    return w, res, bounds


def _pack(ids, sc):
    """(score, id bits) pairs as indexer_decode_partial lays them out."""
    out = np.zeros(ids.shape + (2,), np.float32)
    out[..., 0] = np.where(ids >= 0, np.nan_to_num(sc), 0.0)
    out[..., 1] = ids.astype(np.int32).view(np.float32)
    return torch.from_numpy(out)


def _rank(rank, world, port, q):
    import sparse_attention_block_nvfp4_gb300 as idx
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    tdist.init_process_group("gloo", rank=rank, world_size=world)
    w, res, bounds = _workload()
    lo, hi = bounds[rank]
    mine = _pack(*indexer.partial_candidates(res, lo, hi, w.query_len))
    gathered = idx.gather_candidates(mine)
    q.put((rank, gathered.numpy()))
    tdist.destroy_process_group()


def test_two_gloo_ranks_gather_and_merge():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = 29600 + os.getpid() % 1000
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    got = dict(q.get(timeout=180) for _ in range(2))
    for p in procs:
        p.join(60)
        assert p.exitcode == 0
    w, res, bounds = _workload()
    want = np.stack([_pack(*indexer.partial_candidates(res, lo, hi, w.query_len)).numpy()
                     for lo, hi in bounds])
    for r in range(2):                       # rank-major, identical on every rank
        assert np.array_equal(got[r].view(np.uint32), want.view(np.uint32))
    g = got[0]
    ids = [g[k, ..., 1].view(np.int32) for k in range(2)]
    sc = [np.where(ids[k] >= 0, g[k, ..., 0].astype(np.float64), np.nan) for k in range(2)]
    assert np.array_equal(indexer.merge_candidates(ids, sc, res.L), res.out)
