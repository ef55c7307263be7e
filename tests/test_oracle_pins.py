"""Pins for the CPU oracle: each checks it against something other than itself.

* hand-worked byte examples (tests/golden/*.json, each with its citation);
* exhaustive format tables against library casts (torch float8_e4m3fn,
  ml_dtypes float4_e2m1fn) and a field-by-field decoder;
* the scalar brute force (oracle/brute.py) on tiny inputs;
* closed-form special cases and structural invariants.

``test_oracle_mutations.py`` plants mistakes in the oracle and checks that
these pins catch each one.
"""
import json
import os

import numpy as np
import pytest
import torch

import workloads
from oracle import brute, checker, formats, indexer, nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


# ----------------------------------------------------------------------------
# pin functions: return None when the oracle agrees, else a description
# ----------------------------------------------------------------------------

def pin_row_decode_golden():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_row_decode.json")))
    row = np.zeros(72, np.uint8)
    for k, v in g["row_bytes_nonzero"].items():
        row[int(k)] = v
    qb = np.zeros(128, np.uint8)
    for k, v in g["q_bytes_nonzero"].items():
        qb[int(k)] = v
    k = nvfp4.decode_rows(row[None])[0]
    want_k = np.zeros(128)
    for i, v in g["k_nonzero"].items():
        want_k[int(i)] = v
    if not np.array_equal(k, want_k):
        return f"decoded K {k[np.nonzero(k)]} at {np.nonzero(k)}"
    q = formats.e4m3_value(qb)
    want_q = np.zeros(128)
    for i, v in g["q_nonzero"].items():
        want_q[int(i)] = v
    if not np.array_equal(q, want_q):
        return "decoded Q differs"
    page = np.zeros((128, 72), np.uint8)
    page[5] = row                            # the example in token 5 of a page
    S, A = indexer.page_scores(q[None], nvfp4.decode_rows(page)[None])
    if S[0, 0] != g["dot"] or A[0, 0] != g["abs_dot"]:
        return f"page score {S[0, 0]} / {A[0, 0]}"
    return None


def pin_quantize_golden():
    g = json.load(open(os.path.join(GOLDEN, "nvfp4_quantize.json")))
    x = np.zeros(128, np.uint16)
    want = np.zeros(72, np.uint8)
    for gi, grp in enumerate(g["groups"]):
        for k, v in grp["x_bf16"].items():
            x[int(k)] = int(v, 16)
        for k, v in grp["codes_bytes"].items():
            want[int(k)] = int(v, 16)
        want[64 + gi] = int(grp["scale_byte"], 16)
    got = nvfp4.quantize_rows(x[None])[0]
    if not np.array_equal(got, want):
        bad = np.nonzero(got != want)[0]
        return f"bytes {bad.tolist()}: got {[hex(b) for b in got[bad]]} want {[hex(b) for b in want[bad]]}"
    return None


def pin_e4m3_table():
    allb = np.arange(256, dtype=np.uint8)
    lib = torch.from_numpy(allb).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    ours = formats.e4m3_value(allb)
    field = np.array([brute.e4m3(int(b)) for b in allb])
    same = lambda a, b: np.array_equal(np.isnan(a), np.isnan(b)) and np.array_equal(a[~np.isnan(a)], b[~np.isnan(b)])
    if not same(ours, lib):
        return "E4M3 table differs from torch.float8_e4m3fn"
    if not same(ours, field):
        return "E4M3 table differs from the field decoder"
    return None


def pin_e2m1_table():
    codes = np.arange(16, dtype=np.uint8)
    ours = formats.e2m1_value(codes)
    field = np.array([brute.e2m1(int(c)) for c in codes])
    if not np.array_equal(ours, field):
        return "E2M1 table differs from the field decoder"
    ml = pytest.importorskip("ml_dtypes")
    lib = codes.view(ml.float4_e2m1fn).astype(np.float64)
    if not np.array_equal(ours, lib):
        return "E2M1 table differs from ml_dtypes.float4_e2m1fn"
    return None


def pin_scale_rounding_exhaustive():
    """Every positive finite bf16 amax: E4M3(amax/6) against torch's RNE cast
    of fl32(amax)/6 (in range), and saturation above 448."""
    bits = np.arange(1, 0x7F80, dtype=np.uint32)           # positive finite bf16
    amax = (bits << 16).view(np.float32)
    v32 = amax / np.float32(6.0)
    ours = formats.e4m3_round_nonneg(amax.astype(np.float64) / 6.0)
    inr = v32 < 464.0
    lib = torch.from_numpy(v32[inr]).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    if not np.array_equal(ours[inr], lib):
        i = np.nonzero(ours[inr] != lib)[0][0]
        return f"scale of amax={amax[inr][i]}: ours {ours[inr][i]:#x} torch {lib[i]:#x}"
    if not np.all(ours[~inr] == 0x7E):
        return "no saturation to 448"
    return None


def pin_code_rounding():
    """E2M1 RNE against ml_dtypes' cast on a grid holding every midpoint,
    every code value, both signs, zero, and values past 6."""
    ml = pytest.importorskip("ml_dtypes")
    grid = np.arange(-8.0, 8.0 + 1e-9, 1.0 / 64)
    extra = np.array([-0.0, 0.0, 1e-30, -1e-30, 6.0000001, 100.0, -100.0])
    x = np.concatenate([grid, extra])
    ours = formats.e2m1_round(x)
    lib = x.astype(np.float32).astype(ml.float4_e2m1fn).view(np.uint8)
    if not np.array_equal(ours, lib):
        i = np.nonzero(ours != lib)[0][0]
        return f"x={x[i]}: ours {ours[i]:#x} ml_dtypes {lib[i]:#x}"
    return None


def _tiny_case(seed=11):
    """A few pages of arbitrary bytes, 2 heads, query_len 3 straddling page
    boundaries, one padding request (seq_len < query_len)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    kv = workloads.random_pages(8, rng)
    seq = np.array([2 * 128 + 1, 3 * 128 + 2, 2, 130], np.int32)
    table = np.array([[3, 5, 1, 0], [6, 2, 7, 4], [0, 0, 0, 0], [1, 3, 0, 0]], np.int32)
    qlen, H = 3, 2
    q = workloads.random_q(len(seq) * qlen, H, rng)
    return q, kv, table, seq, qlen, H


def pin_bruteforce():
    q, kv, table, seq, qlen, H = _tiny_case()
    res = indexer.decode(q, kv, table, seq, qlen, H)
    ids, scores = brute.indexer_rows(q, kv, table, seq, [qlen] * len(seq), H)
    if not np.array_equal(res.out, np.array(ids, np.int32)):
        return f"ids differ from brute force:\n{res.out}\n{np.array(ids)}"
    for (row, h, j), (s, a) in scores.items():
        if abs(res.S[row, h, j] - s) > 1e-12 * a or abs(res.A[row, h, j] - a) > 1e-12 * a:
            return f"score ({row},{h},{j}) {res.S[row, h, j]} vs brute {s}"
    n_scored = np.count_nonzero(~np.isnan(res.S))
    if n_scored != len(scores):
        return f"oracle scored {n_scored} (row, head, page) triples, brute force {len(scores)}"
    # the same rows through the prefill entry point (ragged query lengths)
    cu = np.concatenate([[0], np.cumsum([qlen] * len(seq))])
    resp = indexer.prefill(q, cu, kv, table, seq, H)
    if not np.array_equal(resp.out, res.out):
        return "prefill entry point differs from decode on the same rows"
    return None


def pin_closed_forms():
    rng = np.random.Generator(np.random.PCG64(5))
    nb = 40
    # (a) q = 0 or identical pages: all scores tie -> ids 0..14 then local
    kv = workloads.random_pages(nb, rng)
    seq = np.array([37 * 128 + 5], np.int32)
    table = rng.permutation(nb)[None, :38].astype(np.int32)
    q0 = np.zeros((1, 1, 128), np.uint8)
    r = indexer.decode(q0, kv, table, seq, 1, 1)
    want = np.array(list(range(15)) + [37], np.int32)
    if not np.array_equal(r.out[0, 0], want):
        return f"q=0: {r.out[0, 0]}"
    kv_same = np.repeat(kv[:1], nb, axis=0)
    qr = workloads.random_q(1, 1, rng)
    r = indexer.decode(qr, kv_same, table, seq, 1, 1)
    if not np.array_equal(r.out[0, 0], want):
        return f"identical pages: {r.out[0, 0]}"
    # (b) one-hot power-of-two q: score = 2^a * max_t k[t, c], exact
    c, a_byte = 77, 0x48                                  # 0x48 = 4.0
    q1 = np.zeros((1, 1, 128), np.uint8)
    q1[0, 0, c] = a_byte
    r = indexer.decode(q1, kv, table, seq, 1, 1)
    K = nvfp4.decode_rows(kv[table[0, :37]])              # [37, 128, 128]
    if not np.array_equal(r.S[0, 0, :37], 4.0 * K[:, :, c].max(axis=1)):
        return "one-hot query score"
    # (c) fewer than 16 valid pages: every history page, then the local page
    seq2 = np.array([9 * 128 + 100], np.int32)
    r = indexer.decode(qr, kv, table, seq2, 1, 1)
    o = r.out[0, 0]
    if sorted(o[:9].tolist()) != list(range(9)) or o[9] != 9 or np.any(o[10:] != -1):
        return f"V<=16: {o}"
    if np.any(np.diff(r.S[0, 0, o[:9]]) > 0):
        return "V<=16 ids not in score order"
    # (d) the tiny-decode workload's 700-token request: V = 6
    w = workloads.config(0)
    kvw = np.zeros((w.num_blocks, 128, 72), np.uint8)
    nvfp4.insert(w.k_bf16, w.slot_mapping, kvw)
    rw = indexer.decode(w.q_decode, kvw, w.dec_page_table, w.dec_seq_lens, 1, 1)
    o = rw.out[0, 0]
    if sorted(o[:5].tolist()) != list(range(5)) or o[5] != 5 or np.any(o[6:] != -1):
        return f"700-token request: {o}"
    if rw.L[1] != 2499 // 128 or rw.out[1, 0, 15] != rw.L[1]:
        return "2500-token request local page"
    return None


def pin_invariants(res) -> str:
    """Structure of every oracle row (see oracle.checker)."""
    rep = checker.check_ids(res.out, res)
    if rep["fails"]:
        return f"invariants: {rep['examples']}"
    if rep["differ"]:
        return "oracle differs from itself"
    return None


PINS = [pin_row_decode_golden, pin_quantize_golden, pin_e4m3_table, pin_e2m1_table,
        pin_scale_rounding_exhaustive, pin_code_rounding, pin_bruteforce, pin_closed_forms]


# ----------------------------------------------------------------------------
# tests
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_pin(pin):
    msg = pin()
    assert msg is None, msg


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_invariants_small_workloads(idx):
    w = workloads.config(idx, small=True)
    kv = np.zeros((w.num_blocks, 128, 72), np.uint8)
    nvfp4.insert(w.k_bf16, w.slot_mapping, kv)
    if w.num_decode_reqs:
        r = indexer.decode(w.q_decode, kv, w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads)
        assert pin_invariants(r) is None
    if w.num_prefill_reqs:
        r = indexer.prefill(w.q_prefill, w.cu_seqlens_q, kv, w.pre_page_table, w.pre_seq_lens, w.num_heads)
        assert pin_invariants(r) is None


def test_insert_skips_negative_slots_and_checks_range():
    rng = np.random.Generator(np.random.PCG64(3))
    k = workloads._to_bf16_bits(rng.standard_normal((4, 128), dtype=np.float32))
    kv = np.full((2, 128, 72), 0xAB, np.uint8)
    nvfp4.insert(k, np.array([-1, 3, 129, -5]), kv)
    assert np.all(kv[0, 0] == 0xAB) and np.all(kv[1, 2] == 0xAB)
    assert np.array_equal(kv[0, 3], nvfp4.quantize_rows(k[1:2])[0])
    assert np.array_equal(kv[1, 1], nvfp4.quantize_rows(k[2:3])[0])
    with pytest.raises(ValueError):
        nvfp4.insert(k[:1], np.array([256]), kv)


def test_unreadable_request_rows_are_minus_one():
    rng = np.random.Generator(np.random.PCG64(4))
    kv = workloads.random_pages(4, rng)
    seq = np.array([3 * 128 + 1, 2 * 128 + 1], np.int32)
    table = np.array([[0, 9, 1, 2], [2, 3, 0, 0]], np.int32)   # 9 is outside the cache
    q = workloads.random_q(2, 1, rng)
    r = indexer.decode(q, kv, table, seq, 1, 1)
    assert r.bad.tolist() == [True, False]
    assert np.all(r.out[0] == -1) and r.out[1, 0, 2] == 2
    # a table narrower than the history is unreadable too
    r2 = indexer.decode(q[1:], kv, table[1:, :1], seq[1:], 1, 1)
    assert r2.bad.tolist() == [True]


def test_checker_accepts_near_ties_and_rejects_errors():
    rng = np.random.Generator(np.random.PCG64(8))
    q, kv, table, seq, qlen, H = _tiny_case(8)
    res = indexer.decode(q, kv, table, seq, qlen, H)
    assert checker.check_ids(res.out, res)["fails"] == 0
    # swap two ranked ids whose scores are far apart -> rejected
    bad = res.out.copy()
    r, h = 3, 0                                  # a row with >= 2 history pages
    assert res.L[r] >= 2
    bad[r, h, [0, 1]] = bad[r, h, [1, 0]]
    far = abs(res.S[r, h, bad[r, h, 0]] - res.S[r, h, bad[r, h, 1]]) > 1e-3 * res.A[r, h, 0]
    if far:
        assert checker.check_ids(bad, res)["fails"] == 1
    # make the two scores tie within tolerance -> the swap is accepted
    res.S[r, h, bad[r, h, 0]] = res.S[r, h, bad[r, h, 1]]
    assert checker.check_ids(bad, res)["fails"] == 0
    # wrong local page / missing -1 tail -> rejected
    bad2 = res.out.copy()
    bad2[r, h, 15] = 0
    assert checker.check_ids(bad2, res)["fails"] == 1
    bad3 = res.out.copy()
    m = min(15, int(res.L[r]))
    bad3[r, h, m] = -1
    assert checker.check_ids(bad3, res)["fails"] == 1


def test_cp_merge_of_any_split_is_the_full_selection():
    """Decode context parallelism: merging the per-rank candidates of any
    split of the history into page ranges gives the whole-history selection
    (the top-15 of a union is the top-15 of the parts' top-15s)."""
    rng = np.random.Generator(np.random.PCG64(77))
    w = workloads.config(2, small=True)
    kv = nvfp4.insert(w.k_bf16, w.slot_mapping, np.zeros((w.num_blocks, 128, 72), np.uint8))
    res = indexer.decode(w.q_decode, kv, w.dec_page_table, w.dec_seq_lens, w.query_len, w.num_heads)
    hist = (w.dec_seq_lens.astype(np.int64) - 1) // 128
    for world in (1, 2, 3, 5):
        cuts = np.sort(rng.integers(0, hist[:, None] + 1, size=(len(hist), world - 1)), axis=1)
        bounds = np.concatenate([np.zeros((len(hist), 1), np.int64), cuts, hist[:, None]], axis=1)
        parts = [indexer.partial_candidates(res, bounds[:, k], bounds[:, k + 1], w.query_len)
                 for k in range(world)]
        out = indexer.merge_candidates([p[0] for p in parts], [p[1] for p in parts], res.L)
        assert np.array_equal(out, res.out), world
