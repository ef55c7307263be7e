"""MXFP4 index-K pages: decoding and the quantise-insert.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Layout (page vllm.models.minimax_m3.amd.indexer_mxfp4: the scorers read
"e2m1 / e8m0 pages", ``mxfp4_index_topk_decode`` / ``_prefill`` take
``index_pages [pages, 8704] uint8`` and split each page with
``mxfp4_page_views`` into code data and scales).  Readings of what the page
leaves open:
  * 8704 = 128 tokens x (64 code bytes + 4 scale bytes); the first 8192 bytes
    are the codes of tokens 0..127 in order (64 bytes each), the last 512 the
    scales (4 per token, in token order): the two views of
    ``mxfp4_page_views``;
  * element e of a token sits in byte e // 2, low nibble for even e (as in
    the NVFP4 pages);
  * scale byte j of a token covers elements 32j .. 32j+31 (the 32-element
    block of the OCP microscaling formats; 4 scales x 32 = 128 elements);
  * a token's value is E2M1 code value * 2^(scale byte - 127).

Quantise-insert (the pages show no MXFP4 insert; this is the conversion of
the OCP Microscaling Formats (MX) v1.0 specification, section 6.3):
  * per 32-element block: amax = max |x|; shared exponent
    E = floor(log2(amax)) - 2, 2 being the exponent of E2M1's largest normal
    value (6 = 1.5 * 2^2); E is clamped to the E8M0 range [-127, 127]; the
    scale byte is E + 127; amax = 0 gives the byte 0 (2^-127);
  * codes = E2M1 round-to-nearest-even of x / 2^E, saturating at +-6 (the
    block's largest element lands in [4, 8) and saturates above 6);
  * the sign of a code that rounds to zero is the sign of x;
  * ``slot_mapping[i] = page * 128 + row``; a negative slot is skipped.
"""
from __future__ import annotations

import numpy as np

from .formats import bf16_value, e2m1_round, e2m1_value, e8m0_value

PAGE = 128
DIM = 128
CODE_BYTES = PAGE * 64          # 8192
PAGE_BYTES = CODE_BYTES + PAGE * 4   # 8704
BLOCK = 32


def decode_pages(pages: np.ndarray, phys: np.ndarray) -> np.ndarray:
    """Decode the listed physical pages of ``pages [num_blocks, 8704]``:
    float64 ``[len(phys), 128, 128]``."""
    pg = np.asarray(pages, dtype=np.uint8)[np.asarray(phys, dtype=np.int64)]
    codes_b = pg[:, :CODE_BYTES].reshape(-1, PAGE, 64).astype(np.int64)
    scales_b = pg[:, CODE_BYTES:].reshape(-1, PAGE, 4)
    codes = np.stack([codes_b & 0xF, codes_b >> 4], axis=-1).reshape(-1, PAGE, DIM)
    scale = np.repeat(e8m0_value(scales_b), BLOCK, axis=-1)       # element e -> scale e // 32
    return e2m1_value(codes) * scale


def scale_bytes(pages: np.ndarray, phys: np.ndarray) -> np.ndarray:
    """The E8M0 bytes of the listed pages: uint8 ``[len(phys), 128, 4]``."""
    pg = np.asarray(pages, dtype=np.uint8)[np.asarray(phys, dtype=np.int64)]
    return pg[:, CODE_BYTES:].reshape(-1, PAGE, 4)


def quantize_rows(k_bf16: np.ndarray):
    """Quantise bf16 keys ``[n, 128]`` (bit patterns): code bytes ``[n, 64]``
    and E8M0 scale bytes ``[n, 4]``."""
    x = bf16_value(k_bf16).reshape(-1, 4, BLOCK)                 # [n, block, 32]
    if np.any(~np.isfinite(x)):
        raise ValueError("quantize_rows: non-finite key")
    amax = np.abs(x).max(axis=-1)                                # [n, 4]
    _, e2 = np.frexp(amax)                                       # amax = m * 2^e2, m in [0.5, 1)
    E = np.where(amax > 0, e2.astype(np.int64) - 1 - 2, -127)    # floor(log2 amax) - 2
    E = np.clip(E, -127, 127)
    ratio = x / np.exp2(E.astype(np.float64))[..., None]         # exact: a power-of-two scale
    codes = e2m1_round(ratio).astype(np.int64).reshape(-1, DIM)
    packed = (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8)
    return packed, (E + 127).astype(np.uint8)


def insert(k_bf16: np.ndarray, slot_mapping: np.ndarray, pages: np.ndarray,
           chunk: int = 1 << 16) -> np.ndarray:
    """Write quantised tokens into ``pages [num_blocks, 8704]`` (in place) at
    ``slot_mapping``; negative slots are skipped.  Returns pages."""
    k_bf16 = np.asarray(k_bf16)
    slot_mapping = np.asarray(slot_mapping, dtype=np.int64)
    n_slots = pages.shape[0] * PAGE
    for a in range(0, k_bf16.shape[0], chunk):
        b = min(k_bf16.shape[0], a + chunk)
        codes, scales = quantize_rows(k_bf16[a:b])
        sl = slot_mapping[a:b]
        keep = sl >= 0
        if np.any(sl[keep] >= n_slots):
            raise ValueError("slot out of range")
        blk, row = sl[keep] // PAGE, sl[keep] % PAGE
        for i in range(4):
            pages[blk, CODE_BYTES + row * 4 + i] = scales[keep, i]
        cidx = (row * 64)[:, None] + np.arange(64)[None, :]
        pages[blk[:, None], cidx] = codes[keep]
    return pages
