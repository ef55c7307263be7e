"""Page scores and top-k selection of the NVFP4 lightning indexer.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Definitions, and the passages they follow:
  * position of a query (page vllm.models.minimax_m3.nvidia.indexer_flashinfer,
    ``forward``: the default q_offset right-aligns tokens to the sequence end):
    decode row i of request r has pos = seq_len[r] - query_len + i; prefill
    token i of request r has pos = seq_len[r] - (cu[r+1] - cu[r]) + i.
  * valid pages (same page, builder ``build``): pos // 128 + 1; the local page
    is L = pos // 128; a row with pos < 0 (padding request, page
    vllm.models.minimax_m3.nvidia.indexer_nvfp4, ``forward``: padding rows are
    scored) has no valid page.
  * history pages (indexer_nvfp4, ``_build_prefill_chunks``: only pages before
    the last query's local page are scored): pages 0 .. L-1 of the row.  Every
    token of a history page lies before pos, so no token mask is needed.
  * score (indexer_nvfp4, ``__init__``: "max" scoring; indexer_flashinfer,
    ``forward``: scores are unscaled): S[j] = max over the 128 tokens t of page
    j of sum_d q[d] * k[t, d].  Heads share K and score separately
    (indexer_nvfp4 module description).
  * selection (indexer_nvfp4 module description: 15 score-ranked history
    pages plus the local page last, init_blocks=0, local_blocks=1, logical
    ids; indexer_flashinfer ``forward``: -1 tail padding): the first
    m = min(15, L) history pages ordered by (S descending, page id ascending),
    then L, then -1.
Readings: equal scores rank the lower page id first (the pages are silent);
the order inside the 16 is "score-ranked, local last" (indexer_nvfp4) rather
than indexer_flashinfer's ascending order.

Everything is float64: products of E4M3 and E2M1*E4M3 values are exact, so
S is exact up to float64 summation (<= 128 * 2^-53 relative to A).
A[j] = max_t sum_d |q[d] k[t, d]| is kept for the comparison tolerance.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import Optional, Sequence

import numpy as np

from . import mxfp4
from .formats import e4m3_value
from .nvfp4 import decode_pages

PAGE = 128
DIM = 128
TOPK = 16
HIST_TOPK = TOPK - 1


@dataclass
class Result:
    """Oracle output for a set of rows.

    out   int32 [rows, H, 16]  selected logical page ids
    S, A  float64 [rows, H, W]  page scores / tolerance scale; NaN where the
                               page is not a history page of the row
    L     int64 [rows]          local page (-1 when the row has no valid page)
    bad   bool [rows]           row's request has an unreadable page
    """
    out: np.ndarray
    S: np.ndarray
    A: np.ndarray
    L: np.ndarray
    bad: np.ndarray


def local_page(pos: np.ndarray) -> np.ndarray:
    pos = np.asarray(pos, dtype=np.int64)
    return np.where(pos >= 0, pos // PAGE, -1)


def select(S_hist: np.ndarray, L: int) -> np.ndarray:
    """Top-k row for one (row, head): ``S_hist`` holds the scores of pages
    0 .. L-1.  Ranked by (score desc, id asc); local page after; -1 tail."""
    out = np.full(TOPK, -1, dtype=np.int32)
    if L < 0:
        return out
    m = min(HIST_TOPK, L)
    ids = np.arange(L)
    order = np.lexsort((ids, -np.asarray(S_hist[:L], dtype=np.float64)))[:m]
    out[:m] = ids[order]
    out[m] = L
    return out


def page_scores(q_rows: np.ndarray, k_pages: np.ndarray):
    """q_rows float64 [n, 128]; k_pages float64 [P, 128, 128] -> S, A [n, P]."""
    P = k_pages.shape[0]
    if P == 0:
        z = np.zeros((q_rows.shape[0], 0))
        return z, z.copy()
    kf = k_pages.reshape(P * PAGE, DIM)
    dots = (q_rows @ kf.T).reshape(q_rows.shape[0], P, PAGE)
    absd = (np.abs(q_rows) @ np.abs(kf).T).reshape(q_rows.shape[0], P, PAGE)
    return dots.max(axis=2), absd.max(axis=2)


def _request_pages(kv_pages, page_table_row, n_hist, width_tokens, seq_len):
    """Physical ids of history pages 0..n_hist-1, or None if one is unreadable
    (the table is narrower than the history, or an id is outside the cache).
    The local page is output as a logical id and never looked up."""
    if n_hist * PAGE > width_tokens:
        return None
    phys = np.asarray(page_table_row[:n_hist], dtype=np.int64)
    if np.any(phys < 0) or np.any(phys >= kv_pages.shape[0]):
        return None
    return phys


def _dequant_request(kv_pages, phys, page_format="nvfp4"):
    """Decode a request's history pages once: float64 [P, 128, 128].
    ``page_format``: "nvfp4" pages [num_blocks, 128, 72] or "mxfp4" pages
    [num_blocks, 8704] (page vllm.models.minimax_m3.amd.indexer_mxfp4: the
    same scores and top-k over a different codec)."""
    if page_format == "mxfp4":
        if phys.size and np.any(mxfp4.scale_bytes(kv_pages, phys) == 0xFF):
            raise ValueError("oracle: NaN E8M0 scale byte in a scored page")
        return mxfp4.decode_pages(kv_pages, phys)
    if phys.size:
        scales = kv_pages[phys][:, :, 64:72]
        if np.any((scales & 0x7F) == 0x7F):
            raise ValueError("oracle: NaN E4M3 scale byte in a scored page")
    return decode_pages(kv_pages, phys)


def _score_rows(q_rows_bytes, K, H):
    """q_rows_bytes uint8 [n, H, 128], K float64 [P, 128, 128] -> S, A [n, H, P]."""
    n = q_rows_bytes.shape[0]
    q = e4m3_value(q_rows_bytes).reshape(n * H, DIM)
    if np.any(np.isnan(q)):
        raise ValueError("oracle: NaN E4M3 query byte")
    S, A = page_scores(q, K)
    return S.reshape(n, H, -1), A.reshape(n, H, -1)


def _run(q, kv_pages, page_table, seq_lens, qlens, H, rows_wanted, page_format="nvfp4"):
    """Shared body of decode and prefill: requests r with qlens[r] rows each, right-aligned."""
    kv_pages = np.asarray(kv_pages, dtype=np.uint8)
    page_table = np.asarray(page_table)
    seq_lens = np.asarray(seq_lens, dtype=np.int64)
    qlens = np.asarray(qlens, dtype=np.int64)
    starts = np.concatenate([[0], np.cumsum(qlens)])
    total = int(starts[-1])
    width_tokens = page_table.shape[1] * PAGE if page_table.ndim == 2 else 0
    if rows_wanted is None:
        rows_wanted = np.arange(total)
    rows_wanted = np.asarray(rows_wanted, dtype=np.int64)
    nrow = rows_wanted.size
    req_of = np.searchsorted(starts, rows_wanted, side="right") - 1
    pos_all = seq_lens[req_of] - qlens[req_of] + (rows_wanted - starts[req_of])
    L_all = local_page(pos_all)
    W = int(max(0, L_all.max())) if nrow else 0
    out = np.full((nrow, H, TOPK), -1, dtype=np.int32)
    S = np.full((nrow, H, W), np.nan)
    A = np.full((nrow, H, W), np.nan)
    bad = np.zeros(nrow, dtype=bool)
    for r in np.unique(req_of):
        sel = np.nonzero(req_of == r)[0]
        # pages the request scores: those before its last query's local page
        last_pos = int(seq_lens[r]) - 1
        n_hist = last_pos // PAGE if last_pos >= 0 else 0
        phys = _request_pages(kv_pages, page_table[r], n_hist, width_tokens, int(seq_lens[r]))
        if phys is None:
            bad[sel] = True
            continue                       # rows stay all -1
        # only the pages up to the largest wanted local page are needed
        need = int(max(0, L_all[sel].max()))
        K = _dequant_request(kv_pages, phys[:need], page_format)
        # query rows in chunks that keep the [rows*H, need*128] products small
        step = max(1, (1 << 23) // max(1, H * need * PAGE))
        for c0 in range(0, sel.size, step):
            cs = sel[c0:c0 + step]
            nc = int(max(0, L_all[cs].max()))
            if nc > 0:
                Sc, Ac = _score_rows(np.asarray(q[rows_wanted[cs]]), K[:nc], H)
                S[cs, :, :nc] = Sc
                A[cs, :, :nc] = Ac
            for row in cs:
                Lr = int(L_all[row])
                if Lr < 0:
                    continue
                S[row, :, Lr:] = np.nan
                A[row, :, Lr:] = np.nan
                for h in range(H):
                    out[row, h] = select(S[row, h, :Lr], Lr)
    return Result(out=out, S=S, A=A, L=L_all, bad=bad)


def decode(q, kv_pages, page_table, seq_lens, query_len: int, num_heads: int,
           rows: Optional[Sequence[int]] = None, page_format: str = "nvfp4") -> Result:
    """Decode indexer: every request has ``query_len`` query rows at its last
    ``query_len`` positions.  q uint8 [num_reqs * query_len, H, 128]."""
    R = len(seq_lens)
    return _run(q, kv_pages, page_table, seq_lens, np.full(R, query_len), num_heads, rows,
                page_format)


def prefill(q, cu_seqlens_q, kv_pages, page_table, seq_lens, num_heads: int,
            rows: Optional[Sequence[int]] = None, page_format: str = "nvfp4") -> Result:
    """Prefill indexer: request r owns rows cu[r] .. cu[r+1]-1, right-aligned
    to seq_lens[r] (context = seq_len - query_len tokens before them)."""
    cu = np.asarray(cu_seqlens_q, dtype=np.int64)
    return _run(q, kv_pages, page_table, seq_lens, np.diff(cu), num_heads, rows, page_format)


def partial_candidates(res: Result, page_lo, page_hi, query_len: int):
    """One context-parallel rank's candidates (page
    vllm.models.minimax_m3.nvidia.indexer_nvfp4: ``decode_cp.forward`` keeps
    each rank's best pages per row and merges them): for every decode row and
    head, the row's history pages j in [page_lo[r], page_hi[r]) ordered by
    (S descending, j ascending), the first 15, then -1.  ``res`` is the
    oracle over the whole history.  Returns ids int32 [rows, H, 15] and their
    scores float64 (NaN where the id is -1)."""
    rows, H = res.out.shape[:2]
    ids = np.full((rows, H, HIST_TOPK), -1, dtype=np.int32)
    sc = np.full((rows, H, HIST_TOPK), np.nan)
    for t in range(rows):
        r = t // query_len
        Lr = int(res.L[t])
        if Lr <= 0 or res.bad[t]:
            continue
        lo, hi = max(0, int(page_lo[r])), min(Lr, int(page_hi[r]))
        if hi <= lo:
            continue
        js = np.arange(lo, hi)
        for h in range(H):
            S = res.S[t, h, lo:hi]
            order = np.lexsort((js, -S))[:HIST_TOPK]
            ids[t, h, :order.size] = js[order]
            sc[t, h, :order.size] = S[order]
    return ids, sc


def merge_candidates(ids_list, sc_list, L):
    """Final rows [rows, H, 16] from several ranks' candidates: the first
    min(15, count) of all candidates by (score descending, id ascending),
    then the local page L[row], then -1 (all -1 where L < 0)."""
    ids = np.concatenate(ids_list, axis=2)
    sc = np.concatenate(sc_list, axis=2)
    rows, H = ids.shape[:2]
    out = np.full((rows, H, TOPK), -1, dtype=np.int32)
    for t in range(rows):
        if L[t] < 0:
            continue
        for h in range(H):
            ok = ids[t, h] >= 0
            cid, cs = ids[t, h][ok], sc[t, h][ok]
            order = np.lexsort((cid, -cs))[:HIST_TOPK]
            m = order.size
            out[t, h, :m] = cid[order]
            out[t, h, m] = L[t]
    return out
