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

Precision.  The pages fix none.  This oracle is the definition above
evaluated in float64 (the bf16 inputs, the fp32 eps and the fp32 table
entries are exact float64 values), rounded to bf16 once at the end, to
nearest with ties to even.  A kernel that evaluates the same formula in
fp32, in any summation order, with correctly rounded operations, lands
within ``fp32_error_bound`` of the float64 value; where that interval
contains a bf16 rounding boundary, the key element may legitimately round
to either bf16 neighbour.  ``check_rows`` therefore accepts a quantised row
if it equals the quantisation of the float64 key, or of a key in which some
of those boundary elements take their other neighbour, and reports how
many rows needed that allowance.
"""
from __future__ import annotations

import itertools

import numpy as np

from . import nvfp4

DIM = 128
F32 = np.float32
U32 = 2.0 ** -24          # unit roundoff of fp32 (round to nearest)
TINY32 = 2.0 ** -149      # smallest fp32 subnormal: absolute error of an underflowing fp32 result


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


def f64_to_bf16(x: np.ndarray) -> np.ndarray:
    """float64 -> bf16 bit patterns, ONE rounding to nearest, ties to even
    (bf16: 8 significant bits, fp32's exponent range, subnormals in steps of
    2^-133).  A value that rounds past the largest bf16 is an error."""
    x = np.asarray(x, dtype=np.float64)
    if np.any(~np.isfinite(x)):
        raise ValueError("f64_to_bf16: non-finite value")
    a = np.abs(x)
    _, e = np.frexp(a)                                  # a = m * 2^e, 0.5 <= m < 1
    step_exp = np.maximum(e - 8, -133)                  # 8 significant bits; subnormal floor
    q = np.rint(np.ldexp(a, -step_exp))                 # exact scaling; rint = ties to even
    v = np.ldexp(q, step_exp)                           # the bf16 value, exact in float64
    if np.any(v > float(bf16_to_f32(np.array([0x7F7F], np.uint16))[0])):
        raise ValueError("f64_to_bf16: value above the largest bf16")
    bits = (v.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # exact: v is a bf16 value
    return bits | (np.signbit(x).astype(np.uint16) << 15)


def rms_scale(x: np.ndarray, eps: float) -> np.ndarray:
    """1 / sqrt(mean(x^2) + eps) per row of float64 x [n, 128], in float64."""
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt((x * x).mean(axis=1) + np.float64(eps))


def rotate(y: np.ndarray, cos: np.ndarray, sin: np.ndarray, rotary_dim: int, is_neox: bool) -> np.ndarray:
    """RoPE on float64 rows y [n, 128] with per-row cos / sin [n, rd/2]."""
    out = y.copy()
    h = rotary_dim // 2
    if h == 0:
        return out
    if is_neox:
        y1, y2 = y[:, :h], y[:, h:rotary_dim]
    else:
        y1, y2 = y[:, 0:rotary_dim:2], y[:, 1:rotary_dim:2]
    o1 = y1 * cos - y2 * sin
    o2 = y2 * cos + y1 * sin
    if is_neox:
        out[:, :h], out[:, h:rotary_dim] = o1, o2
    else:
        out[:, 0:rotary_dim:2], out[:, 1:rotary_dim:2] = o1, o2
    return out


def _pairs(rotary_dim: int, is_neox: bool):
    """Element indices (i1, i2) of the rotated pairs."""
    h = rotary_dim // 2
    if is_neox:
        return np.arange(h), np.arange(h) + h
    return np.arange(0, rotary_dim, 2), np.arange(1, rotary_dim, 2)


def _table_rows(cos_sin_cache, positions, rotary_dim):
    cache = np.asarray(cos_sin_cache, dtype=F32)
    pos = np.asarray(positions, dtype=np.int64)
    if np.any(pos < 0) or np.any(pos >= cache.shape[0]):
        raise ValueError("position outside the cos/sin table")
    h = rotary_dim // 2
    rows = cache[pos].astype(np.float64)
    return rows[:, :h], rows[:, h:rotary_dim]


def _check_rd(rotary_dim):
    rotary_dim = int(rotary_dim)
    if rotary_dim % 2 or not 0 <= rotary_dim <= DIM:
        raise ValueError("rotary_dim must be even and in [0, 128]")
    return rotary_dim


def norm_rope_f64(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox):
    """qk-norm + RoPE of bf16 keys [n, 128] at int positions [n]: float64
    [n, 128] (before the bf16 rounding).  eps is taken as the fp32 value the
    C entry point receives."""
    rotary_dim = _check_rd(rotary_dim)
    x = bf16_to_f32(k_bf16).reshape(-1, DIM).astype(np.float64)
    w = bf16_to_f32(weight_bf16).reshape(DIM).astype(np.float64)
    y = x * rms_scale(x, float(np.float32(eps)))[:, None] * w[None, :]
    if rotary_dim == 0:                     # norm only: positions and table unused
        return y
    cos, sin = _table_rows(cos_sin_cache, positions, rotary_dim)
    return rotate(y, cos, sin, rotary_dim, bool(is_neox))


def norm_rope_bf16(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox):
    """The bf16 keys [n, 128] (bit patterns) of the exact qk-norm + RoPE."""
    return f64_to_bf16(norm_rope_f64(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim,
                                     is_neox))


def fp32_error_bound(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox):
    """Per element, a bound on |v32 - v| where v is the float64 value of
    ``norm_rope_f64`` and v32 the same formula evaluated in fp32 with
    correctly rounded operations (u = 2^-24), the 128 squares summed in ANY
    order, fused multiply-adds allowed:
      * sum of squares: relative error <= 127 u (positive terms, any order),
        plus 128 * 2^-149 absolute for squares that underflow;
      * v = ss / 128 + eps: + 1 u (the division by 128 is exact);
      * sqrt, then 1 / sqrt: half of v's relative error + 2 u;
      * y = (x rs) w: + 2 u                  -> rho_y, relative, per token;
      * pass-through element: |dy| <= rho_y |y| + 2 * 2^-149;
      * rotated element (y1 c - y2 s or y2 c + y1 s): the two products add
        1 u each and the sum 1 u: |do| <= (rho_y + 2 u) (|y1 c| + |y2 s|) +
        u |o| + 4 * 2^-149.
    Every relative term is inflated by 1 % for the second-order products."""
    rotary_dim = _check_rd(rotary_dim)
    x = bf16_to_f32(k_bf16).reshape(-1, DIM).astype(np.float64)
    w = bf16_to_f32(weight_bf16).reshape(DIM).astype(np.float64)
    e32 = float(np.float32(eps))
    ss = (x * x).sum(axis=1)
    with np.errstate(divide="ignore", invalid="ignore"):
        rho_ss = 127 * U32 + np.where(ss > 0, 128 * TINY32 / ss, 0.0)
    ms = ss / 128.0
    with np.errstate(divide="ignore", invalid="ignore"):
        rho_v = np.where(ms + e32 > 0, rho_ss * ms / (ms + e32), 0.0) + U32
    rho_y = (rho_v / 2 + 4 * U32) * 1.01                 # sqrt, 1/sqrt, x * rs, * w
    y = x * rms_scale(x, e32)[:, None] * w[None, :]
    bound = rho_y[:, None] * np.abs(y) + 2 * TINY32
    if rotary_dim:
        cos, sin = _table_rows(cos_sin_cache, positions, rotary_dim)
        i1, i2 = _pairs(rotary_dim, bool(is_neox))
        y1, y2 = y[:, i1], y[:, i2]
        mag = np.abs(y1 * cos) + np.abs(y2 * sin)
        o = rotate(y, cos, sin, rotary_dim, bool(is_neox))
        r = (rho_y[:, None] + 2 * U32 * 1.01) * mag + 4 * TINY32
        bound[:, i1] = r + U32 * 1.01 * np.abs(o[:, i1])
        r2 = (rho_y[:, None] + 2 * U32 * 1.01) * (np.abs(y2 * cos) + np.abs(y1 * sin)) + 4 * TINY32
        bound[:, i2] = r2 + U32 * 1.01 * np.abs(o[:, i2])
    return bound


def _bf16_neighbour(bits: np.ndarray, up: np.ndarray) -> np.ndarray:
    """The next bf16 above (up) or below (not up) the given bf16 values
    (finite; the step across zero goes to the smallest subnormal of the
    other sign)."""
    b = bits.astype(np.int32)
    neg = (b & 0x8000) != 0
    mag = b & 0x7FFF
    away = np.where(neg, ~up, up)                    # moving away from zero
    out = np.where(away, b + 1, b - 1)
    # toward zero from +-0: cross to the other sign's smallest subnormal
    zero = mag == 0
    out = np.where(zero & ~away, np.where(neg, 0x0001, 0x8001), out)
    return (out & 0xFFFF).astype(np.uint16)


def bf16_choices(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox):
    """(b0, b1, amb): b0 = the bf16 rounding of the float64 key [n, 128];
    where ``amb`` is set, the float64 value lies within ``fp32_error_bound``
    of the rounding boundary between b0 and b1, so an fp32 evaluation may
    give b1 instead."""
    v = norm_rope_f64(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox)
    d = fp32_error_bound(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox)
    b0 = f64_to_bf16(v)
    v0 = bf16_to_f32(b0).astype(np.float64)
    up = v >= v0
    b1 = _bf16_neighbour(b0, up)
    v1 = bf16_to_f32(b1).astype(np.float64)
    mid = (v0 + v1) / 2.0                             # exact in float64
    amb = np.abs(v - mid) <= d
    return b0, b1, amb


def check_rows(rows, k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox,
               max_alternatives: int = 1 << 10):
    """Parity check of quantised rows ``rows [n, 72]`` (the fused insert's
    output for keys [n]) against the oracle.  A row passes if it equals
    ``nvfp4.quantize_rows`` of the float64 key's bf16 rounding, or, group by
    group (the quantiser's 16-element groups are independent), of a key in
    which some boundary elements (``bf16_choices``) take their other bf16
    neighbour.  Returns {"rows", "exact", "allowance", "fails", "fail_rows"}."""
    rows = np.asarray(rows, dtype=np.uint8).reshape(-1, nvfp4.ROW_BYTES)
    b0, b1, amb = bf16_choices(k_bf16, positions, weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox)
    want = nvfp4.quantize_rows(b0)
    exact = np.all(rows == want, axis=1)
    fails = []
    allowance = 0
    for t in np.nonzero(~exact)[0]:
        ok_row = True
        for g in range(8):
            cols = list(range(8 * g, 8 * g + 8)) + [64 + g]
            got_g = rows[t, cols]
            if np.array_equal(got_g, want[t, cols]):
                continue
            idx = [e for e in range(16 * g, 16 * g + 16) if amb[t, e]]
            found = False
            if 0 < len(idx) and (1 << len(idx)) <= max_alternatives:
                # every non-empty subset of the boundary elements at its other
                # neighbour, quantised in one batch
                picks = np.array(list(itertools.product((0, 1), repeat=len(idx)))[1:], dtype=bool)
                keys = np.repeat(b0[t][None, :], picks.shape[0], axis=0)
                for c, e in enumerate(idx):
                    keys[picks[:, c], e] = b1[t, e]
                alt = nvfp4.quantize_rows(keys)[:, cols]
                found = bool(np.any(np.all(alt == got_g[None, :], axis=1)))
            if not found:
                ok_row = False
                break
        if ok_row:
            allowance += 1
        else:
            fails.append(int(t))
    return {"rows": int(rows.shape[0]), "exact": int(exact.sum()), "allowance": allowance,
            "fails": len(fails), "fail_rows": fails[:16]}


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
    keep = kept_tokens(pos, slots, cos_sin_cache, rotary_dim)
    if not np.any(keep):
        return kv_pages
    kb = norm_rope_bf16(k_bf16[keep], pos[keep], weight_bf16, eps, cos_sin_cache, rotary_dim, is_neox)
    return nvfp4.insert(kb, slots[keep], kv_pages)


def kept_tokens(positions, slot_mapping, cos_sin_cache, rotary_dim):
    """Tokens the fused insert writes: slot >= 0 and, when there is a
    rotation, a position inside the cos/sin table."""
    pos = np.asarray(positions, dtype=np.int64)
    keep = np.asarray(slot_mapping, dtype=np.int64) >= 0
    if int(rotary_dim) > 0:                 # a position is only read when there is a rotation
        cache = np.asarray(cos_sin_cache, dtype=F32)
        keep &= (pos >= 0) & (pos < cache.shape[0])
    return keep
