"""E2M1 and E4M3 number formats, written out from their definitions.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

E2M1 (OCP microscaling FP4): 1 sign bit, 2 exponent bits (bias 1), 1 mantissa
bit, no inf/NaN.  Magnitudes of codes 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6.

E4M3 "fn" (OCP FP8): 1 sign, 4 exponent bits (bias 7), 3 mantissa bits; the
exponent-0 encodings are subnormals m/8 * 2^-6; 0x7F / 0xFF are NaN; no inf;
largest finite 448.

E8M0 (OCP microscaling shared scale): 8 exponent bits, bias 127, no sign or
mantissa; 0xFF is NaN.

Page vllm.models.minimax_m3.nvidia.indexer_nvfp4 (module description) names
the formats: "E2M1 codes, then E4M3 block scales" for K and E4M3 for Q; page
vllm.models.minimax_m3.amd.indexer_mxfp4 (module description) names "e2m1 /
e8m0 pages" for its MXFP4 K.
"""
from __future__ import annotations

import numpy as np

E2M1_MAG = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0], dtype=np.float64)


def e2m1_value(code: np.ndarray) -> np.ndarray:
    """Value of 4-bit E2M1 codes (low 4 bits of ``code``)."""
    code = np.asarray(code).astype(np.int64) & 0xF
    mag = E2M1_MAG[code & 7]
    return np.where(code & 8, -mag, mag)


def e4m3_value(byte: np.ndarray) -> np.ndarray:
    """Value of E4M3fn bytes; NaN for 0x7F / 0xFF."""
    b = np.asarray(byte).astype(np.int64) & 0xFF
    sign = np.where(b & 0x80, -1.0, 1.0)
    e = (b >> 3) & 0xF
    m = (b & 7).astype(np.float64)
    normal = (1.0 + m / 8.0) * np.exp2(e.astype(np.float64) - 7.0)
    sub = (m / 8.0) * 2.0 ** -6
    v = np.where(e == 0, sub, normal)
    v = np.where((b & 0x7F) == 0x7F, np.nan, v)
    return sign * v


# All finite non-negative E4M3 values; byte code i has value E4M3_POS[i],
# strictly increasing in i (0x00 .. 0x7E).
E4M3_POS = e4m3_value(np.arange(0x7F))
E4M3_MAX = float(E4M3_POS[-1])  # 448


def e4m3_round_nonneg(v: np.ndarray) -> np.ndarray:
    """Round non-negative reals to E4M3 bytes: nearest value, ties to the even
    encoding (even mantissa), values above 448 saturate to 448 (0x7E)."""
    v = np.asarray(v, dtype=np.float64)
    if np.any(~np.isfinite(v)) or np.any(v < 0):
        raise ValueError("e4m3_round_nonneg: needs finite non-negative input")
    hi = np.searchsorted(E4M3_POS, v, side="left")          # first value >= v
    hi = np.minimum(hi, len(E4M3_POS) - 1)
    lo = np.maximum(hi - 1, 0)
    d_lo = np.abs(v - E4M3_POS[lo])
    d_hi = np.abs(E4M3_POS[hi] - v)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    out = np.where(pick_hi, hi, lo)
    out = np.where(v >= E4M3_MAX, len(E4M3_POS) - 1, out)
    return out.astype(np.uint8)


def e2m1_round(x: np.ndarray) -> np.ndarray:
    """Round reals to E2M1 codes: nearest magnitude, ties to the even code,
    magnitudes above 6 saturate to 6; the sign bit is the sign of x (so a
    negative value that rounds to zero keeps its sign, like -0.0)."""
    x = np.asarray(x, dtype=np.float64)
    if np.any(~np.isfinite(x)):
        raise ValueError("e2m1_round: needs finite input")
    a = np.abs(x)
    hi = np.searchsorted(E2M1_MAG, a, side="left")
    hi = np.minimum(hi, 7)
    lo = np.maximum(hi - 1, 0)
    d_lo = np.abs(a - E2M1_MAG[lo])
    d_hi = np.abs(E2M1_MAG[hi] - a)
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0))
    mag = np.where(pick_hi, hi, lo)
    mag = np.where(a >= 6.0, 7, mag)
    sign = np.signbit(x).astype(np.int64) << 3
    return (mag | sign).astype(np.uint8)


def e8m0_value(byte: np.ndarray) -> np.ndarray:
    """Value of E8M0 bytes (OCP microscaling shared scale): 2^(byte - 127), no
    sign, no mantissa; 0xFF is NaN."""
    b = np.asarray(byte).astype(np.int64) & 0xFF
    v = np.exp2(b.astype(np.float64) - 127.0)
    return np.where(b == 0xFF, np.nan, v)


def bf16_value(bits: np.ndarray) -> np.ndarray:
    """Value of bf16 bit patterns (the high half of an fp32)."""
    b = np.asarray(bits).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
