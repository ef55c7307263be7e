"""Pins for the MXFP4 part of the CPU oracle (oracle/mxfp4.py and the
page_format="mxfp4" path of oracle/indexer.py), each against something other
than the oracle itself:

* hand-worked byte examples (tests/golden/mxfp4_*.json, with citations);
* the E8M0 table against fp32 bit patterns built directly from the exponent
  field, and the field decoder of oracle/brute.py;
* the quantiser against an exhaustive nearest-code search on random blocks,
  round-trip of representable blocks, and the E8M0 range clamps;
* the scalar brute force (oracle/brute.py) on tiny MXFP4 workloads.

``test_oracle_mutations.py`` plants mistakes and checks these pins catch them.
"""
import json
import os

import numpy as np
import pytest

import workloads
from oracle import brute, checker, formats, indexer, mxfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _bf16_bits(x):
    """Round fp32 values to bf16 bit patterns (nearest even)."""
    u = np.asarray(x, np.float32).view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return u.astype(np.uint16)


def pin_mx_page_decode_golden():
    g = json.load(open(os.path.join(GOLDEN, "mxfp4_page_decode.json")))
    page = np.zeros((1, mxfp4.PAGE_BYTES), np.uint8)
    for k, v in g["page_bytes_nonzero"].items():
        page[0, int(k)] = v
    qb = np.zeros(128, np.uint8)
    for k, v in g["q_bytes_nonzero"].items():
        qb[int(k)] = v
    K = mxfp4.decode_pages(page, [0])[0]
    want = np.zeros(128)
    for i, v in g["k_nonzero"].items():
        want[int(i)] = v
    t = g["token"]
    if not np.array_equal(K[t], want) or np.count_nonzero(np.delete(K, t, axis=0)):
        return f"decoded K: token {t} {K[t][np.nonzero(K[t])]} at {np.nonzero(K[t])}"
    q = formats.e4m3_value(qb)
    S, A = indexer.page_scores(q[None], K[None])
    if S[0, 0] != g["dot"] or A[0, 0] != g["abs_dot"]:
        return f"page score {S[0, 0]} / {A[0, 0]}"
    return None


def pin_mx_quantize_golden():
    g = json.load(open(os.path.join(GOLDEN, "mxfp4_quantize.json")))
    x = np.zeros(128, np.uint16)
    for k, v in g["x_bf16_nonzero"].items():
        x[int(k)] = int(v, 16)
    want_c = np.zeros(64, np.uint8)
    for k, v in g["codes_bytes_nonzero"].items():
        want_c[int(k)] = int(v, 16)
    want_s = np.array([int(v, 16) for v in g["scale_bytes"]], np.uint8)
    c, s = mxfp4.quantize_rows(x[None])
    if not np.array_equal(c[0], want_c):
        bad = np.nonzero(c[0] != want_c)[0]
        return f"code bytes {bad.tolist()}: got {[hex(b) for b in c[0][bad]]}"
    if not np.array_equal(s[0], want_s):
        return f"scale bytes {[hex(b) for b in s[0]]}"
    return None


def pin_e8m0_table():
    b = np.arange(256)
    ours = formats.e8m0_value(b)
    # fp32 with exponent field b (b >= 1) is 2^(b - 127); b = 0 is the fp32
    # subnormal 2^-127 = mantissa bit 22
    bits = np.where(b >= 1, b.astype(np.uint32) << 23, np.uint32(1 << 22)).astype(np.uint32)
    lib = bits.view(np.float32).astype(np.float64)
    field = np.array([brute.e8m0(int(v)) for v in b])
    if not np.isnan(ours[255]) or not np.isnan(field[255]):
        return "0xFF is not NaN"
    if not np.array_equal(ours[:255], lib[:255]):
        return "E8M0 table differs from fp32 bit patterns"
    if not np.array_equal(ours[:255], field[:255]):
        return "E8M0 table differs from the field decoder"
    return None


def pin_mx_quantize_search():
    """Random blocks over many binades: every code is the nearest E2M1 value
    to x / 2^E (ties to the even code, saturating at 6), E = floor(log2 amax)
    - 2 clamped to [-127, 127], found by exhaustive search over exponents and
    codes."""
    rng = np.random.Generator(np.random.PCG64(11))
    n = 64
    mant = rng.standard_normal((n, 128)).astype(np.float32)
    spread = np.exp2(rng.integers(-140, 120, size=(n, 4)).astype(np.float32))
    x = mant * np.repeat(spread, 32, axis=1)
    x[0, :32] = 0.0
    bits = _bf16_bits(x)
    xv = formats.bf16_value(bits).reshape(n, 4, 32)
    codes, sbytes = mxfp4.quantize_rows(bits)
    cod = np.stack([codes & 0xF, codes >> 4], axis=-1).reshape(n, 4, 32).astype(np.int64)
    for i in range(n):
        for j in range(4):
            blk = xv[i, j]
            amax = float(np.abs(blk).max())
            E = -127
            if amax > 0:
                e = -200
                while 2.0 ** (e + 1) <= amax:    # largest e with 2^e <= amax
                    e += 1
                E = max(-127, min(127, e - 2))
            if int(sbytes[i, j]) != E + 127:
                return f"block {i},{j}: scale byte {sbytes[i, j]} want {E + 127}"
            for t in range(32):
                r = blk[t] / 2.0 ** E
                best = None
                for c in range(8):
                    v = brute.e2m1(c)
                    d = abs(abs(r) - v)
                    if best is None or d < best[0] or (d == best[0] and c % 2 == 0):
                        best = (d, c)
                mag = 7 if abs(r) >= 6.0 else best[1]
                want = mag | (8 if np.signbit(r) else 0)
                if cod[i, j, t] != want:
                    return f"block {i},{j} elem {t}: x/2^E={r} code {cod[i, j, t]} want {want}"
    return None


def pin_mx_round_trip():
    """A block whose values are E2M1 values times 2^E, with one element of
    magnitude 4 or 6 (so floor(log2 amax) - 2 = E), quantises to itself."""
    rng = np.random.Generator(np.random.PCG64(12))
    for trial in range(200):
        E = int(rng.integers(-120, 120))
        c = rng.integers(0, 16, size=128)
        for j in range(4):
            c[32 * j + int(rng.integers(0, 32))] = int(rng.choice([6, 7, 14, 15]))
        v = formats.e2m1_value(c) * 2.0 ** E
        bits = _bf16_bits(v.astype(np.float32))
        if not np.array_equal(formats.bf16_value(bits), v):
            continue
        pg = np.zeros((1, mxfp4.PAGE_BYTES), np.uint8)
        mxfp4.insert(bits[None], np.array([3]), pg)
        back = mxfp4.decode_pages(pg, [0])[0, 3]
        if not np.array_equal(back, v):
            return f"E={E}: round trip differs at {np.nonzero(back != v)[0][:4]}"
    return None


def pin_mx_bruteforce():
    """Tiny MXFP4 workloads: the vectorised oracle against oracle/brute.py."""
    rng = np.random.Generator(np.random.PCG64(13))
    for H, seqs, qlen in [(1, [300, 520], 2), (2, [129, 400], 1)]:
        nb = 8
        pages = rng.integers(0, 256, size=(nb, mxfp4.PAGE_BYTES), dtype=np.uint8)
        sc = pages[:, mxfp4.CODE_BYTES:]
        pages[:, mxfp4.CODE_BYTES:] = 112 + (sc % 32)          # scales 2^-15 .. 2^16
        table = np.stack([rng.permutation(nb)[:5] for _ in seqs]).astype(np.int32)
        q = workloads.random_q(len(seqs) * qlen, H, rng)
        res = indexer.decode(q, pages, table, np.array(seqs), qlen, H, page_format="mxfp4")
        out, scores = brute.indexer_rows(q, pages, table, seqs, [qlen] * len(seqs), H,
                                         page_format="mxfp4")
        if not np.array_equal(res.out, np.array(out, np.int32)):
            return f"ids differ (H={H})"
        for (row, h, j), (s, a) in scores.items():
            if abs(res.S[row, h, j] - s) > 1e-12 * max(1.0, a) or abs(res.A[row, h, j] - a) > 1e-12 * max(1.0, a):
                return f"score ({row},{h},{j}): {res.S[row, h, j]} vs {s}"
    return None


PINS = [pin_mx_page_decode_golden, pin_mx_quantize_golden, pin_e8m0_table,
        pin_mx_quantize_search, pin_mx_round_trip, pin_mx_bruteforce]


@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    msg = pin()
    assert msg is None, msg


def test_mx_insert_skips_negative_slots_and_checks_range():
    rng = np.random.Generator(np.random.PCG64(14))
    k = _bf16_bits(rng.standard_normal((3, 128)).astype(np.float32))
    pg = np.zeros((2, mxfp4.PAGE_BYTES), np.uint8)
    mxfp4.insert(k, np.array([-1, 5, 200]), pg)
    assert np.count_nonzero(pg[0, 64 * 5: 64 * 6]) > 0
    assert np.count_nonzero(pg[1]) > 0 and np.count_nonzero(pg[0, :64 * 5]) == 0
    with pytest.raises(ValueError):
        mxfp4.insert(k[:1], np.array([256]), pg)


def test_mx_invariants_small_workload():
    w = workloads.config(2, small=True)
    pg = np.zeros((w.num_blocks, mxfp4.PAGE_BYTES), np.uint8)
    mxfp4.insert(w.k_bf16, w.slot_mapping, pg)
    res = indexer.decode(w.q_decode, pg, w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads,
                         page_format="mxfp4")
    rep = checker.check_ids(res.out, res)
    assert rep["fails"] == 0 and rep["differ"] == 0
