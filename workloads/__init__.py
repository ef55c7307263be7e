"""Seeded synthetic inputs for the NVFP4 lightning indexer.

This module only DRAWS inputs: sequence lengths, page tables, slot mappings,
bf16 index keys and E4M3 index queries.  It holds none of the indexer's own
arithmetic (no NVFP4 quantisation, no scoring, no selection), so both the CPU
oracle and the CUDA path can take their inputs from here without sharing any
of the method.

The five named workloads follow the configurations the indexer is measured on
(tiny decode, decode batch, speculative decode, ragged prefill, long-context
mixed step).  Draw order for every workload is fixed: sequence lengths, page
table permutation, outlier channels, per-page scale exponents, K, Q.  The
generator is ``numpy.random.Generator(PCG64(seed))``.

Conventions (vLLM's, as used by the pages' metadata builders):
  * ``seq_lens[r]`` counts every token of request r, the new queries included;
  * the cache holds all ``seq_lens[r]`` tokens of request r, token t of
    request r lives in physical page ``page_table[r, t // 128]`` at row
    ``t % 128``; ``slot_mapping = physical_page * 128 + row``;
  * decode requests come first, then prefill requests; Q rows follow the same
    order (request-major, then query, then head);
  * unused page-table entries are 0.

Casts to bf16 (K) and E4M3 (Q) are done by torch; they prepare the inputs the
indexer receives and are not part of the indexer.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

PAGE = 128          # tokens per index-K page
DIM = 128           # index head dim


def _to_bf16_bits(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _to_e4m3_bytes(x: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy()


@dataclass
class Workload:
    """All inputs of one indexer step (one decode call and/or one prefill call)."""
    name: str
    num_heads: int
    query_len: int                      # decode query length (0 if no decode)
    dec_seq_lens: np.ndarray            # int32 [Rd]
    pre_seq_lens: np.ndarray            # int32 [Rp]
    pre_query_lens: np.ndarray          # int32 [Rp]
    page_table: np.ndarray              # int32 [Rd + Rp, width]
    num_blocks: int
    k_bf16: np.ndarray                  # uint16 [num_tokens, 128] (bf16 bit patterns)
    slot_mapping: np.ndarray            # int64 [num_tokens]
    q_e4m3: np.ndarray                  # uint8 [T, H, 128], decode rows then prefill rows
    seed: int = 0
    notes: str = ""
    meta: dict = field(default_factory=dict)

    @property
    def num_decode_reqs(self) -> int:
        return int(self.dec_seq_lens.shape[0])

    @property
    def num_prefill_reqs(self) -> int:
        return int(self.pre_seq_lens.shape[0])

    @property
    def num_decode_rows(self) -> int:
        return self.num_decode_reqs * self.query_len

    @property
    def cu_seqlens_q(self) -> np.ndarray:
        cu = np.zeros(self.num_prefill_reqs + 1, dtype=np.int32)
        cu[1:] = np.cumsum(self.pre_query_lens)
        return cu

    @property
    def total_prefill_q(self) -> int:
        return int(self.pre_query_lens.sum())

    @property
    def seq_lens(self) -> np.ndarray:
        return np.concatenate([self.dec_seq_lens, self.pre_seq_lens]).astype(np.int32)

    @property
    def dec_page_table(self) -> np.ndarray:
        return self.page_table[: self.num_decode_reqs]

    @property
    def pre_page_table(self) -> np.ndarray:
        return self.page_table[self.num_decode_reqs:]

    @property
    def q_decode(self) -> np.ndarray:
        return self.q_e4m3[: self.num_decode_rows]

    @property
    def q_prefill(self) -> np.ndarray:
        return self.q_e4m3[self.num_decode_rows:]


def make_workload(
    *,
    name: str,
    seed: int,
    num_heads: int,
    dec_seq_lens: Sequence[int] = (),
    query_len: int = 0,
    pre_seq_lens: Sequence[int] = (),
    pre_query_lens: Sequence[int] = (),
    num_blocks: Optional[int] = None,
    slack: float = 0.10,
    outlier_channels: int = 0,
    outlier_gain: float = 8.0,
    page_scale_spread: float = 0.0,
    rng: Optional[np.random.Generator] = None,
    extra_table_width: int = 0,
    poison_unused: bool = False,
    notes: str = "",
) -> Workload:
    """Draw one workload.  The caller gives the lengths; everything else is drawn.

    ``num_blocks`` defaults to ceil((1 + slack) * pages in use).  Physical pages
    are a random permutation of the cache (every request's pages are scattered).
    """
    if rng is None:
        rng = np.random.Generator(np.random.PCG64(seed))
    dec = np.asarray(dec_seq_lens, dtype=np.int64)
    pre = np.asarray(pre_seq_lens, dtype=np.int64)
    preq = np.asarray(pre_query_lens, dtype=np.int64)
    assert pre.shape == preq.shape
    assert np.all(preq <= pre) and np.all(preq >= 0)
    all_seq = np.concatenate([dec, pre])
    nreq = all_seq.shape[0]
    pages_per_req = (np.maximum(all_seq, 0) + PAGE - 1) // PAGE
    used = int(pages_per_req.sum())
    if num_blocks is None:
        num_blocks = max(1, int(np.ceil((1.0 + slack) * used)))
    assert num_blocks >= used, "cache too small for the requests"
    width = int(max(1, pages_per_req.max() if nreq else 1)) + extra_table_width

    # 2. page table: a random permutation of the physical pages
    perm = rng.permutation(num_blocks).astype(np.int32)
    page_table = np.zeros((max(nreq, 1), width), dtype=np.int32)[:nreq]
    if poison_unused:
        page_table[:] = -7  # never read by a correct indexer
    off = 0
    for r in range(nreq):
        n = int(pages_per_req[r])
        page_table[r, :n] = perm[off: off + n]
        off += n

    # 3. outlier channels, 4. per-page scale exponents
    outl = rng.choice(DIM, size=outlier_channels, replace=False) if outlier_channels else np.zeros(0, np.int64)
    page_exp = [rng.uniform(-page_scale_spread, page_scale_spread, size=int(pages_per_req[r]))
                if page_scale_spread > 0 else None for r in range(nreq)]

    # 5. K: every cached token of every request, in request order
    ntok = int(np.maximum(all_seq, 0).sum())
    k = np.empty((ntok, DIM), dtype=np.uint16)
    slots = np.empty(ntok, dtype=np.int64)
    pos = 0
    chunk = 1 << 16
    for r in range(nreq):
        n = int(max(all_seq[r], 0))
        t0 = 0
        while t0 < n:
            t1 = min(n, t0 + chunk)
            x = rng.standard_normal((t1 - t0, DIM), dtype=np.float32)
            if outlier_channels:
                x[:, outl] *= np.float32(outlier_gain)
            tok = np.arange(t0, t1)
            if page_exp[r] is not None:
                x *= np.exp2(page_exp[r][tok // PAGE]).astype(np.float32)[:, None]
            k[pos + t0: pos + t1] = _to_bf16_bits(x)
            slots[pos + t0: pos + t1] = page_table[r, tok // PAGE].astype(np.int64) * PAGE + tok % PAGE
            t0 = t1
        pos += n

    # 6. Q: decode rows (request-major, query, head) then prefill rows
    nrows = int(dec.shape[0]) * int(query_len) + int(preq.sum())
    qf = rng.standard_normal((nrows, num_heads, DIM), dtype=np.float32)
    q = _to_e4m3_bytes(qf).reshape(nrows, num_heads, DIM)

    return Workload(
        name=name, num_heads=num_heads, query_len=int(query_len),
        dec_seq_lens=dec.astype(np.int32), pre_seq_lens=pre.astype(np.int32),
        pre_query_lens=preq.astype(np.int32), page_table=page_table,
        num_blocks=int(num_blocks), k_bf16=k, slot_mapping=slots, q_e4m3=q,
        seed=seed, notes=notes,
        meta=dict(outlier_channels=[int(c) for c in outl], page_scale_spread=page_scale_spread),
    )


# --------------------------------------------------------------------------
# The five named workloads (full size) and their scaled-down parity variants.
# --------------------------------------------------------------------------

CONFIG_NAMES = [
    "tiny_decode",
    "decode_batch",
    "spec_decode",
    "ragged_prefill",
    "long_mixed",
]


def config(idx: int, small: bool = False) -> Workload:
    """Workload ``idx`` (0..4).  ``small=True`` keeps the structure (heads,
    query length, distributions, ragged tails, page-boundary crossings) at a
    size the CPU oracle finishes in seconds."""
    seed = idx
    rng = np.random.Generator(np.random.PCG64(seed))
    if idx == 0:
        # 2 requests, query_len 1, seq {700, 2500}, 1 head, 64-block cache.
        return make_workload(name="tiny_decode", seed=seed, rng=rng, num_heads=1,
                             dec_seq_lens=[700, 2500], query_len=1, num_blocks=64)
    if idx == 1:
        nreq, lo, hi = (8, 1000, 4500) if small else (64, 4096, 32768)
        seq = rng.integers(lo, hi + 1, size=nreq)
        return make_workload(name="decode_batch" + ("_small" if small else ""), seed=seed, rng=rng,
                             num_heads=4, dec_seq_lens=seq, query_len=1, outlier_channels=4)
    if idx == 2:
        nreq, lo, hi = (6, 1500, 5000) if small else (128, 8192, 65536)
        seq = rng.integers(lo, hi + 1, size=nreq)
        if small:
            seq[0] = 128 * 20 + 2   # the 4 queries straddle a page boundary
        return make_workload(name="spec_decode" + ("_small" if small else ""), seed=seed, rng=rng,
                             num_heads=8, dec_seq_lens=seq, query_len=4, outlier_channels=4)
    if idx == 3:
        lens = [300, 1000, 2100] if small else [2048, 8192, 16384, 30000]
        return make_workload(name="ragged_prefill" + ("_small" if small else ""), seed=seed, rng=rng,
                             num_heads=8, pre_seq_lens=lens, pre_query_lens=lens)
    if idx == 4:
        if small:
            dec = [128 * 30 + 5, 128 * 24]
            pre_ctx, pre_new = [128 * 10, 128 * 6 + 17], [300, 200]
        else:
            dec = [131072] * 16
            pre_ctx, pre_new = [65536, 65536], [8192, 8192]
        pre = [c + n for c, n in zip(pre_ctx, pre_new)]
        return make_workload(name="long_mixed" + ("_small" if small else ""), seed=seed, rng=rng,
                             num_heads=8, dec_seq_lens=dec, query_len=8,
                             pre_seq_lens=pre, pre_query_lens=pre_new,
                             outlier_channels=4, page_scale_spread=6.0)
    raise ValueError(idx)


def random_pages(num_blocks: int, rng: np.random.Generator, nan_free: bool = True) -> np.ndarray:
    """Arbitrary page bytes [num_blocks, 128, 72]: uniform codes, and scale
    bytes uniform over the finite E4M3 encodings (0x7F / 0xFF are NaN)."""
    pages = rng.integers(0, 256, size=(num_blocks, PAGE, 72), dtype=np.uint8)
    if nan_free:
        sc = pages[:, :, 64:]
        bad = (sc & 0x7F) == 0x7F
        sc[bad] &= 0xFE
        pages[:, :, 64:] = sc
    return pages


def random_q(rows: int, heads: int, rng: np.random.Generator) -> np.ndarray:
    return _to_e4m3_bytes(rng.standard_normal((rows, heads, DIM), dtype=np.float32)).reshape(rows, heads, DIM)


# ----------------------------------------------------------------------------- block-sparse attend inputs
# The main KV cache the attend reads: bf16 [num_blocks, 128, H, 128] for K and
# for V.  It is as large as the index cache times H x 128 bf16 per token (about
# 10 GB for the long mixed step), so its values come from a counter-based
# hash of the element's coordinates: the CPU computes only the pages it
# checks, the GPU fills the whole cache with the same bits (torch integer
# ops, in chunks).  Hash: 32-bit murmur3 finalizer of
# (element index XOR seed key); value: sign bit, exponent 124..127 and a
# 7-bit mantissa from the hash, so |value| lies in [1/8, 2).
_M32 = 0xFFFFFFFF


def _mul32(x, c: int):
    """(x * c) mod 2^32 for 0 <= x < 2^32 held in int64, without overflow."""
    lo, hi = c & 0xFFFF, c >> 16
    return (x * lo + (((x * hi) & 0xFFFF) << 16)) & _M32


def _fmix32(x):
    x = x ^ (x >> 16)
    x = _mul32(x, 0x85EBCA6B)
    x = x ^ (x >> 13)
    x = _mul32(x, 0xC2B2AE35)
    return x ^ (x >> 16)


def _kv_key(seed: int, which: int) -> int:
    return ((seed * 0x9E3779B1) ^ (which * 0x7F4A7C15) ^ 0x2545F491) & _M32


def _hash_to_bf16(h):
    return ((h >> 9) & 1) << 15 | (124 + ((h >> 7) & 3)) << 7 | (h & 0x7F)


def attend_kv_pages(seed: int, which: int, blocks, H: int) -> np.ndarray:
    """bf16 bits [len(blocks), 128, H, 128] of main-cache blocks ``blocks``
    (which = 0 for K, 1 for V), numpy."""
    b = np.asarray(blocks, dtype=np.int64).reshape(-1, 1, 1, 1)
    t = np.arange(PAGE, dtype=np.int64).reshape(1, -1, 1, 1)
    h = np.arange(H, dtype=np.int64).reshape(1, 1, -1, 1)
    d = np.arange(DIM, dtype=np.int64).reshape(1, 1, 1, -1)
    e = (((b * PAGE + t) * H + h) * DIM + d) & _M32
    return _hash_to_bf16(_fmix32(e ^ _kv_key(seed, which))).astype(np.uint16)


def attend_kv_fill(seed: int, which: int, num_blocks: int, H: int, device, chunk_blocks: int = 2048):
    """The whole main cache [num_blocks, 128, H, 128] as an int16 torch tensor
    on ``device`` (bf16 bits), the same values as ``attend_kv_pages``."""
    import torch
    out = torch.empty((num_blocks, PAGE, H, DIM), dtype=torch.int16, device=device)
    per = PAGE * H * DIM
    key = _kv_key(seed, which)
    for b0 in range(0, num_blocks, chunk_blocks):
        b1 = min(num_blocks, b0 + chunk_blocks)
        e = (torch.arange(b0 * per, b1 * per, dtype=torch.int64, device=device) & _M32) ^ key
        v = _hash_to_bf16(_fmix32(e))
        out[b0:b1] = (v - ((v >> 15) << 16)).to(torch.int16).view(b1 - b0, PAGE, H, DIM)
    return out


def attend_q(rows: int, heads: int, rng: np.random.Generator) -> np.ndarray:
    """Attention queries, bf16 bits [rows, heads, 128] from N(0, 1)."""
    return _to_bf16_bits(rng.standard_normal((rows, heads, DIM), dtype=np.float32)).reshape(rows, heads, DIM)


def attend_rows(w: "Workload"):
    """(row_req, row_pos) int32 [rows] of the workload's rows: decode rows
    first (request-major, query i at seq_len - query_len + i), then the
    prefill rows (context first)."""
    req, pos = [], []
    for r in range(w.num_decode_reqs):
        s = int(w.dec_seq_lens[r])
        for i in range(w.query_len):
            req.append(r)
            pos.append(s - w.query_len + i)
    for k in range(w.num_prefill_reqs):
        s, ql = int(w.pre_seq_lens[k]), int(w.pre_query_lens[k])
        for i in range(ql):
            req.append(w.num_decode_reqs + k)
            pos.append(s - ql + i)
    return np.array(req, np.int32), np.array(pos, np.int32)
