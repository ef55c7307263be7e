"""Scalar brute force for tiny inputs: a pin for the vectorised oracle.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__``).

Written separately from ``formats`` / ``nvfp4`` / ``indexer``: formats are
decoded from their bit fields with ``math.ldexp`` (no value tables), bytes
are walked one element at a time, dot products are plain Python float
(float64) loops, and the selection is a full sort of (-score, id) pairs.
Pure Python: only for a handful of pages and heads.
"""
from __future__ import annotations

import math


def e2m1(code: int) -> float:
    """E2M1 from its fields: sign | 2-bit exponent (bias 1) | 1-bit mantissa."""
    s = -1.0 if code & 8 else 1.0
    e = (code >> 1) & 3
    m = code & 1
    if e == 0:
        return s * math.ldexp(m, -1)          # subnormal: m * 2^(1-1) * 1/2
    return s * math.ldexp(1.0 + m / 2.0, e - 1)


def e4m3(byte: int) -> float:
    """E4M3fn from its fields: sign | 4-bit exponent (bias 7) | 3-bit mantissa."""
    s = -1.0 if byte & 0x80 else 1.0
    e = (byte >> 3) & 0xF
    m = byte & 7
    if e == 15 and m == 7:
        return math.nan
    if e == 0:
        return s * math.ldexp(m, -9)           # m/8 * 2^-6
    return s * math.ldexp(8 + m, e - 10)       # (1 + m/8) * 2^(e-7)


def e8m0(byte: int) -> float:
    """E8M0 from its field: 8-bit exponent, bias 127; 0xFF is NaN."""
    return math.nan if byte == 0xFF else math.ldexp(1.0, byte - 127)


def key_element(row: bytes, e: int) -> float:
    b = row[e // 2]
    code = (b >> 4) if (e & 1) else (b & 0xF)
    return e2m1(code) * e4m3(row[64 + e // 16])


def key_element_mx(page: bytes, t: int, e: int) -> float:
    """Element e of token t of an MXFP4 page: codes of token t at bytes
    64 t .. 64 t + 63, its four E8M0 scales at 8192 + 4 t .. 8192 + 4 t + 3."""
    b = page[64 * t + e // 2]
    code = (b >> 4) if (e & 1) else (b & 0xF)
    return e2m1(code) * e8m0(page[8192 + 4 * t + e // 32])


def score_mx(q_bytes, page) -> tuple:
    """score() for one MXFP4 page (8704 bytes)."""
    q = [e4m3(int(b)) for b in q_bytes]
    page = bytes(int(x) for x in page)
    best = -math.inf
    best_abs = -math.inf
    for t in range(128):
        acc = 0.0
        acc_abs = 0.0
        for d in range(128):
            p = q[d] * key_element_mx(page, t, d)
            acc += p
            acc_abs += abs(p)
        best = max(best, acc)
        best_abs = max(best_abs, acc_abs)
    return best, best_abs


def score(q_bytes, page_rows) -> tuple:
    """(max_t q.k_t, max_t sum |q_d k_td|) over the 128 rows of one page."""
    q = [e4m3(int(b)) for b in q_bytes]
    best = -math.inf
    best_abs = -math.inf
    for row in page_rows:
        row = bytes(int(x) for x in row)
        acc = 0.0
        acc_abs = 0.0
        for d in range(128):
            p = q[d] * key_element(row, d)
            acc += p
            acc_abs += abs(p)
        best = max(best, acc)
        best_abs = max(best_abs, acc_abs)
    return best, best_abs


def indexer_rows(q, kv_pages, page_table, seq_lens, qlens, num_heads, page_format="nvfp4"):
    """Ids [rows][H][16] and scores {(row, h, page): S} by brute force
    (``page_format`` "nvfp4": pages [n, 128, 72]; "mxfp4": pages [n, 8704])."""
    page_score = score_mx if page_format == "mxfp4" else score
    out = []
    scores = {}
    row = 0
    for r, (seq, ql) in enumerate(zip(seq_lens, qlens)):
        for i in range(int(ql)):
            pos = int(seq) - int(ql) + i
            per_head = []
            for h in range(num_heads):
                if pos < 0:
                    per_head.append([-1] * 16)
                    continue
                L = pos // 128
                cand = []
                for j in range(L):
                    phys = int(page_table[r][j])
                    s, a = page_score(q[row][h], kv_pages[phys])
                    scores[(row, h, j)] = (s, a)
                    cand.append((-s, j))
                cand.sort()
                ids = [j for _, j in cand[:15]]
                ids.append(L)
                ids += [-1] * (16 - len(ids))
                per_head.append(ids)
            out.append(per_head)
            row += 1
    return out, scores


def bf16(bits: int) -> float:
    """bf16 from its fields: sign | 8-bit exponent (bias 127) | 7-bit mantissa."""
    s = -1.0 if bits & 0x8000 else 1.0
    e = (bits >> 7) & 0xFF
    m = bits & 0x7F
    if e == 0xFF:
        return math.nan if m else s * math.inf
    if e == 0:
        return s * math.ldexp(m, -133)          # m/128 * 2^-126
    return s * math.ldexp(128 + m, e - 134)     # (1 + m/128) * 2^(e-127)


def attend_one(q_bits, k_cache, v_cache, page_table_row, pos: int, ids_row, hk: int, scale: float):
    """Block-sparse attention of one query head (pure Python): walk every
    position 0 .. pos of the request, keep those whose page (position // 128)
    is among the selected ids, score q.k * scale with plain float loops,
    softmax with the maximum subtracted, weighted sum of the v rows.  Returns
    a list of 128 floats (all 0 when nothing is visible)."""
    chosen = {int(j) for j in ids_row if int(j) >= 0}
    q = [bf16(int(b)) for b in q_bits]
    toks = []
    for p in range(pos + 1):
        if p // 128 in chosen:
            blk = int(page_table_row[p // 128])
            k = [bf16(int(b)) for b in k_cache[blk][p % 128][hk]]
            v = [bf16(int(b)) for b in v_cache[blk][p % 128][hk]]
            toks.append((scale * math.fsum(a * b for a, b in zip(q, k)), v))
    if not toks:
        return [0.0] * len(q)
    m = max(s for s, _ in toks)
    w = [math.exp(s - m) for s, _ in toks]
    tot = math.fsum(w)
    return [math.fsum(wi * v[d] for wi, (_, v) in zip(w, toks)) / tot for d in range(len(q))]
