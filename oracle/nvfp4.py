"""NVFP4 index-K pages: row decoding and the quantise-insert.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Layout (page vllm.models.minimax_m3.nvidia.indexer_nvfp4, module description:
packed NVFP4 pages ``[num_blocks, 128, 72]``, E2M1 codes then E4M3 block
scales, no global scale).  Readings of what the page leaves open:
  * token-major rows of 72 bytes: bytes 0..63 hold the 128 E2M1 codes, bytes
    64..71 the 8 E4M3 scales (the shape ``[num_blocks, 128, 72]``);
  * element e sits in byte e // 2, low nibble for even e (low nibble first);
  * scale byte j covers elements 16j .. 16j+15 (one scale per 16 elements);
  * a token's value is code value * scale value (no global scale).

Quantise-insert (the step that writes the pages; the pages only say the
fused qk-norm/rope insert writes them):
  * per 16-element group g: amax = max |x|, scale byte = E4M3 round-to-
    nearest-even of amax / 6 (saturating at 448); 6 is the largest E2M1
    magnitude, so the group's largest element maps to the top code;
  * codes = E2M1 round-to-nearest-even of x / scale, saturating at +-6;
  * a zero scale (all-zero group, or amax / 6 below half the smallest E4M3
    subnormal) gives sign-only zero codes;
  * the sign of a code that rounds to zero is the sign of x;
  * ``slot_mapping[i] = page * 128 + row``; a negative slot is skipped
    (vLLM's padding convention).
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_value, e2m1_round, e2m1_value, e4m3_round_nonneg, e4m3_value

PAGE = 128
DIM = 128
ROW_BYTES = 72
PAGE_BYTES = PAGE * ROW_BYTES


def decode_rows(rows: np.ndarray) -> np.ndarray:
    """Decode NVFP4 rows ``[..., 72]`` uint8 to float64 ``[..., 128]``."""
    rows = np.asarray(rows, dtype=np.uint8)
    codes_b = rows[..., :64].astype(np.int64)
    lo = codes_b & 0xF          # even elements
    hi = codes_b >> 4           # odd elements
    codes = np.stack([lo, hi], axis=-1).reshape(*rows.shape[:-1], DIM)
    scales = e4m3_value(rows[..., 64:72])                     # [..., 8]
    scale_per_elem = np.repeat(scales, 16, axis=-1)           # element e -> scale e // 16
    return e2m1_value(codes) * scale_per_elem


def decode_pages(kv_pages: np.ndarray, phys: np.ndarray) -> np.ndarray:
    """Decode the listed physical pages: float64 ``[len(phys), 128, 128]``."""
    return decode_rows(np.asarray(kv_pages)[np.asarray(phys, dtype=np.int64)])


def quantize_rows(k_bf16: np.ndarray) -> np.ndarray:
    """Quantise bf16 keys ``[n, 128]`` (bit patterns) to NVFP4 rows ``[n, 72]``."""
    x = bf16_value(k_bf16).reshape(-1, 8, 16)                 # [n, group, 16]
    if np.any(~np.isfinite(x)):
        raise ValueError("quantize_rows: non-finite key")
    amax = np.abs(x).max(axis=-1)                             # [n, 8]
    sbyte = e4m3_round_nonneg(amax / 6.0)                     # [n, 8]
    s = e4m3_value(sbyte)[..., None]                          # [n, 8, 1]
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(s > 0, x / np.where(s > 0, s, 1.0), 0.0)
    codes = e2m1_round(ratio).astype(np.int64)
    # zero scale: sign-only codes (ratio was set to 0 above, restore the sign)
    codes = np.where(s > 0, codes, np.signbit(x).astype(np.int64) << 3)
    codes = codes.reshape(-1, DIM)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)   # [n, 64]
    return np.concatenate([packed, sbyte.astype(np.uint8)], axis=1)


def insert(k_bf16: np.ndarray, slot_mapping: np.ndarray, kv_pages: np.ndarray,
           chunk: int = 1 << 16) -> np.ndarray:
    """Write quantised rows into ``kv_pages`` ([num_blocks, 128, 72], in place)
    at ``slot_mapping``; negative slots are skipped.  Returns kv_pages."""
    k_bf16 = np.asarray(k_bf16)
    slot_mapping = np.asarray(slot_mapping, dtype=np.int64)
    flat = kv_pages.reshape(-1, ROW_BYTES)
    for a in range(0, k_bf16.shape[0], chunk):
        b = min(k_bf16.shape[0], a + chunk)
        rows = quantize_rows(k_bf16[a:b])
        sl = slot_mapping[a:b]
        keep = sl >= 0
        if np.any(sl[keep] >= flat.shape[0]):
            raise ValueError("slot out of range")
        flat[sl[keep]] = rows[keep]
    return kv_pages
