"""qk-norm and RoPE of the index key, ahead of the NVFP4 insert.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Page vllm.models.minimax_m3.nvidia.indexer_nvfp4 (module description) says
only that the index-K cache is written by "the fused qk-norm/rope insert".
Readings (the plainest ones, vLLM's RMSNorm and rotary-embedding
conventions):
  * qk-norm is RMSNorm over the key's 128 elements with a learned bf16
    weight w and an epsilon: y = x / sqrt(mean(x^2) + eps) * w;
  * RoPE rotates the first ``rotary_dim`` elements (even, at most 128) by
    the angles of the token's position, read from a caller-supplied table
    ``cos_sin_cache [max_pos, rotary_dim]`` (cosines in the first
    rotary_dim / 2 columns, sines in the rest).  Pairs are (i, i + rd/2)
    (NeoX) or (2i, 2i + 1) (GPT-J); each pair becomes
    (y1 cos - y2 sin, y2 cos + y1 sin); elements past rotary_dim pass
    through;
  * the result is rounded to bf16, the model's dtype (the unfused path hands
    bf16 keys to the insert), and then quantised by the NVFP4 insert
    (``oracle.nvfp4``).

Precision.  The pages fix none.  The arithmetic is fp32 in a fixed order,
and this oracle takes every step in that precision and order, so that the
bf16 keys, and the quantised codes they decide, can be compared bit for bit:
  * per 16-element group g (the quantiser's groups): t_g = e_g + o_g, where
    e_g and o_g run over the group's even and odd elements in order, each
    step fl(acc + x^2) with one rounding (a fused multiply-add; the square
    of a bf16 value is exact anyway unless it leaves fp32's range); then
    ss = ((t0 + t1) + (t2 + t3)) + ((t4 + t5) + (t6 + t7));
  * v = ss * (1/128) + eps (the product is exact); rs = 1 / sqrt(v), the
    square root and the division each correctly rounded;
  * y = (x * rs) * w, two fp32 roundings;
  * o1 = (y1 * c) - (y2 * s) and o2 = (y2 * c) + (y1 * s), every product and
    sum rounded to fp32 (no fused multiply-add);
  * bf16 = the fp32 value rounded to nearest, ties to even.
"""
from __future__ import annotations

import numpy as np

from . import nvfp4

DIM = 128
F32 = np.float32


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float32 values (exact)."""
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even (finite x)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    if np.any(~np.isfinite(x)):
        raise ValueError("f32_to_bf16: non-finite value")
    u = x.view(np.uint32).astype(np.uint64)
    r = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return r.astype(np.uint16)


def fma_sq(acc: np.ndarray, x: np.ndarray) -> np.ndarray:
    """fl32(acc + x^2) with a single rounding, for float32 acc and bf16-valued
    x: x^2 and the sum are exact in float64 whenever the two terms are
    within 2^29 of each other, and otherwise the smaller one is far below
    half an fp32 ulp of the larger, so rounding the float64 sum to float32
    gives the single rounding."""
    with np.errstate(over="ignore"):
        return (acc.astype(np.float64) + x.astype(np.float64) ** 2).astype(np.float32)


def rms_scale(x: np.ndarray, eps: float) -> np.ndarray:
    """1 / sqrt(mean(x^2) + eps) per row of float32 x [n, 128], in the fixed
    fp32 order: per 16-element group g, running sums e_g (even elements) and
    o_g (odd elements) of fused squares, t_g = e_g + o_g, then
    ((t0 + t1) + (t2 + t3)) + ((t4 + t5) + (t6 + t7))."""
    g = x.reshape(-1, 8, 16)
    e = np.zeros(g.shape[:2], dtype=F32)
    o = np.zeros(g.shape[:2], dtype=F32)
    for i in range(8):
        e = fma_sq(e, g[:, :, 2 * i])
        o = fma_sq(o, g[:, :, 2 * i + 1])
    t = e + o
    ss = ((t[:, 0] + t[:, 1]) + (t[:, 2] + t[:, 3])) + ((t[:, 4] + t[:, 5]) + (t[:, 6] + t[:, 7]))
    v = ss * F32(1.0 / 128.0) + F32(eps)
    return F32(1.0) / np.sqrt(v)


def rotate(y: np.ndarray, cos: np.ndarray, sin: np.ndarray, rotary_dim: int, is_neox: bool) -> np.ndarray:
    """RoPE on float32 rows y [n, 128] with per-row cos / sin [n, rd/2]."""
    out = y.copy()
    h = rotary_dim // 2
    if h == 0:
        return out
    if is_neox:
        y1, y2 = y[:, :h], y[:, h:rotary_dim]
    else:
        y1, y2 = y[:, 0:rotary_dim:2], y[:, 1:rotary_dim:2]
    o1 = (y1 * cos) - (y2 * sin)
    o2 = (y2 * cos) + (y1 * sin)
    if is_neox:
        out[:, :h], out[:, h:rotary_dim] = o1, o2
    else:
        out[:, 0:rotary_dim:2], out[:, 1:rotary_dim:2] = o1, o2
    return out


def norm_rope_f32(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox):
    """qk-norm + RoPE of bf16 keys [n, 128] at int positions [n]: float32 [n, 128]
    (before the bf16 rounding)."""
    rotary_dim = int(rotary_dim)
    if rotary_dim % 2 or not 0 <= rotary_dim <= DIM:
        raise ValueError("rotary_dim must be even and in [0, 128]")
    x = bf16_to_f32(k_bf16).reshape(-1, DIM)
    w = bf16_to_f32(weight_bf16).reshape(DIM)
    y = (x * rms_scale(x, eps)[:, None]) * w[None, :]
    if rotary_dim == 0:                     # norm only: positions and table unused
        return y
    cache = np.asarray(cos_sin_cache, dtype=F32)
    pos = np.asarray(positions, dtype=np.int64)
    if np.any(pos < 0) or np.any(pos >= cache.shape[0]):
        raise ValueError("position outside the cos/sin table")
    h = rotary_dim // 2
    rows = cache[pos]
    return rotate(y, rows[:, :h], rows[:, h:rotary_dim], rotary_dim, bool(is_neox))


def norm_rope_bf16(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox):
    """The bf16 keys [n, 128] (bit patterns) the fused insert quantises."""
    return f32_to_bf16(norm_rope_f32(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim,
                                     is_neox))


def insert(k_bf16, positions, slot_mapping, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox,
           kv_pages):
    """The fused insert: qk-norm, RoPE, bf16, NVFP4 quantise, scatter into
    ``kv_pages [num_blocks, 128, 72]`` (in place).  A negative slot is
    skipped (vLLM's padding convention), and so is a token whose position
    lies outside the cos/sin table when rotary_dim > 0 (the kernel flags it;
    with no rotation the positions are not read).  Returns kv_pages."""
    k_bf16 = np.asarray(k_bf16)
    pos = np.asarray(positions, dtype=np.int64)
    slots = np.asarray(slot_mapping, dtype=np.int64)
    keep = slots >= 0
    if int(rotary_dim) > 0:                 # a position is only read when there is a rotation
        cache = np.asarray(cos_sin_cache, dtype=F32)
        keep &= (pos >= 0) & (pos < cache.shape[0])
    if not np.any(keep):
        return kv_pages
    kb = norm_rope_bf16(k_bf16[keep], pos[keep], weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox)
    return nvfp4.insert(kb, slots[keep], kv_pages)
