"""Block-sparse attention over the selected pages: the consumer of the
indexer's [T, H, 16] id buffer.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Page vllm.models.minimax_m3.nvidia.indexer_nvfp4: the kernels write logical
block ids "straight into the shared [T, H, 16] buffer the attend reads"
(``MiniMaxM3IndexerNvfp4Impl.forward``); page
vllm.models.minimax_m3.nvidia.indexer_flashinfer: "The attend reads the
shared buffer directly" (``forward``).  The pages describe nothing of the
attend itself.  Readings (the plainest ones, the usual paged sparse
attention of vLLM):
  * the main KV cache is paged like the index cache, 128 tokens per page,
    bf16, [num_blocks, 128, H, 128] for K and for V (vLLM's "NHD" layout),
    one KV head per index head; logical page j of request r is physical
    block page_table[r][j] and holds positions 128 j .. 128 j + 127;
  * query head hq (G query heads per KV head, hq = hk * G + g) of row t
    attends over the tokens of the pages index head hk selected for row t:
    ids[t][hk][0..15], -1 entries skipped; a token is visible when its
    position is at most the row's position (causal: only the local page is
    cut), so the visible set is the union of those pages' visible tokens;
  * o[t][hq] = sum_s softmax_s(scale * q.k_s) v_s over the visible tokens
    (scale given by the caller, 1/sqrt(128) by default); a row with no
    visible token (all ids -1) gives o = 0.
Evaluated in float64 from the bf16 inputs (exact float64 values).
"""
from __future__ import annotations

import numpy as np

PAGE = 128
DIM = 128


def bf16_value(bits) -> np.ndarray:
    """bf16 bit patterns -> float64 values (exact)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def visible_tokens(ids_row, page_table_row, pos: int):
    """(physical block, slot-in-page) of every visible token of the selected
    pages, in id order then position order: ids_row [16] logical page ids
    (-1 = none), the request's page-table row, the query position.  The
    visible set is the union of the selected pages' visible tokens, so an id
    listed twice counts once (its first place)."""
    blocks, slots = [], []
    seen = set()
    for j in np.asarray(ids_row).tolist():
        if j < 0 or j in seen:
            continue
        seen.add(j)
        last = min(PAGE - 1, pos - PAGE * j)          # causal cut inside the page
        if last < 0:
            continue
        blocks.append(np.full(last + 1, int(page_table_row[j]), np.int64))
        slots.append(np.arange(last + 1, dtype=np.int64))
    if not blocks:
        return np.zeros(0, np.int64), np.zeros(0, np.int64)
    return np.concatenate(blocks), np.concatenate(slots)


def attend(q_bf16, k_cache, v_cache, page_table, row_req, row_pos, ids, G: int, scale: float):
    """Block-sparse attention, float64.

    q_bf16   bf16 bits [T, H * G, 128]
    k_cache, v_cache  bf16 bits [num_blocks, 128, H, 128]
    page_table int [num_reqs, width]; row_req, row_pos int [T]
    ids      int32 [T, H, 16] (the indexer's output)
    Returns o float64 [T, H * G, 128] and, per (t, hq), the number of
    visible tokens n [T, H * G]."""
    q = bf16_value(q_bf16)
    T, HQ, D = q.shape
    H = HQ // G
    assert HQ == H * G and D == DIM and ids.shape == (T, H, 16)
    o = np.zeros((T, HQ, DIM))
    n = np.zeros((T, HQ), np.int64)
    for t in range(T):
        r, pos = int(row_req[t]), int(row_pos[t])
        for hk in range(H):
            blk, slot = visible_tokens(ids[t, hk], page_table[r], pos)
            if blk.size == 0:
                continue
            K = bf16_value(k_cache[blk, slot, hk])                # [S, 128]
            V = bf16_value(v_cache[blk, slot, hk])
            for g in range(G):
                hq = hk * G + g
                s = scale * (K @ q[t, hq])
                p = np.exp(s - s.max())
                o[t, hq] = (p @ V) / p.sum()
                n[t, hq] = blk.size
    return o, n


def error_bound(q_bf16, k_cache, v_cache, page_table, row_req, row_pos, ids, G: int, scale: float,
                chain: int = 64, exp_rel: float = 2.0 ** -21):
    """Per element, a bound on |o32 - o| for an fp32 evaluation of the same
    attention whose longest sequential chain of additions in any sum (the
    score dot products excepted: 128 terms) is at most ``chain`` and whose
    exponentials (and the rescalings of an online softmax, at most 16) carry
    a relative error below ``exp_rel``.  With w_s = p_s / sum p the exact
    weights, m the largest score and Delta the largest score error,
      Delta = |scale| * max_s sum_d |q_d k_sd| * 130 u   (u = 2^-24),
    each computed weight is off by a relative
      rho = 2 Delta + 17 exp_rel + (2 chain + 20) u
    plus u |s - m| (the rounding of the exponent), so
      |o32 - o| <= rho * sum_s w_s |v_s| + u * sum_s w_s |s - m| |v_s| + u |o|.
    Zero where the row sees no token (the kernel writes exact zeros)."""
    q = bf16_value(q_bf16)
    T, HQ, _ = q.shape
    H = HQ // G
    u = 2.0 ** -24
    bound = np.zeros((T, HQ, DIM))
    for t in range(T):
        r, pos = int(row_req[t]), int(row_pos[t])
        for hk in range(H):
            blk, slot = visible_tokens(ids[t, hk], page_table[r], pos)
            if blk.size == 0:
                continue
            K = bf16_value(k_cache[blk, slot, hk])
            V = bf16_value(v_cache[blk, slot, hk])
            for g in range(G):
                hq = hk * G + g
                s = scale * (K @ q[t, hq])
                m = s.max()
                p = np.exp(s - m)
                w = p / p.sum()
                delta = abs(scale) * float((np.abs(K) @ np.abs(q[t, hq])).max()) * 130 * u
                rho = 2 * delta + 17 * exp_rel + (2 * chain + 20) * u
                bound[t, hq] = rho * (w @ np.abs(V)) + u * ((w * (m - s)) @ np.abs(V)) + u * np.abs(w @ V)
    return bound
