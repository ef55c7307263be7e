"""Planted mistakes: each plausible oracle bug must be caught by a pin.

Every mistake is planted in the CPU oracle (never in the CUDA path) with
monkeypatch, and the test asserts that at least one pin of
test_oracle_pins.py now reports a failure.
"""
import numpy as np
import pytest

from oracle import formats, indexer, nvfp4
import test_oracle_pins as pins


def _any_pin_fails(names):
    for n in names:
        try:
            if getattr(pins, n)() is not None:
                return True
        except Exception:
            return True
    return False


def _decode_rows_swapped(rows):
    rows = np.asarray(rows, dtype=np.uint8)
    b = rows[..., :64].astype(np.int64)
    codes = np.stack([b >> 4, b & 0xF], axis=-1).reshape(*rows.shape[:-1], 128)   # high nibble first
    sc = np.repeat(formats.e4m3_value(rows[..., 64:72]), 16, axis=-1)
    return formats.e2m1_value(codes) * sc


def _decode_rows_scale8(rows):
    rows = np.asarray(rows, dtype=np.uint8)
    b = rows[..., :64].astype(np.int64)
    codes = np.stack([b & 0xF, b >> 4], axis=-1).reshape(*rows.shape[:-1], 128)
    sc = formats.e4m3_value(rows[..., 64:72])
    per = np.repeat(sc, 8, axis=-1)
    per = np.concatenate([per, per], axis=-1)                # one scale per 8 elements
    return formats.e2m1_value(codes) * per


def _e4m3_round_ties_up(v):
    v = np.asarray(v, dtype=np.float64)
    P = formats.E4M3_POS
    hi = np.minimum(np.searchsorted(P, v, side="left"), len(P) - 1)
    lo = np.maximum(hi - 1, 0)
    pick_hi = (P[hi] - v) <= (v - P[lo])
    out = np.where(pick_hi, hi, lo)
    return np.where(v >= formats.E4M3_MAX, len(P) - 1, out).astype(np.uint8)


def _e2m1_round_ties_away(x):
    x = np.asarray(x, dtype=np.float64)
    a = np.abs(x)
    M = formats.E2M1_MAG
    hi = np.minimum(np.searchsorted(M, a, side="left"), 7)
    lo = np.maximum(hi - 1, 0)
    mag = np.where((M[hi] - a) <= (a - M[lo]), hi, lo)
    mag = np.where(a >= 6, 7, mag)
    return (mag | (np.signbit(x).astype(np.int64) << 3)).astype(np.uint8)


_ORIG_E2M1 = formats.e2m1_round


def _e2m1_round_unsigned_zero(x):
    c = _ORIG_E2M1(x)
    return np.where((c & 7) == 0, 0, c).astype(np.uint8)


_ORIG_SELECT = indexer.select
_ORIG_LOCAL = indexer.local_page
_ORIG_SCORES = indexer.page_scores


def _select_ties_high_id(S_hist, L):
    out = np.full(16, -1, dtype=np.int32)
    if L < 0:
        return out
    m = min(15, L)
    ids = np.arange(L)
    order = np.lexsort((-ids, -np.asarray(S_hist[:L])))[:m]
    out[:m] = ids[order]
    out[m] = L
    return out


def _select_no_local(S_hist, L):
    out = _ORIG_SELECT(S_hist, L)
    if L >= 0:
        out[min(15, L)] = -1
    return out


def _select_ascending(S_hist, L):
    out = _ORIG_SELECT(S_hist, L)
    if L >= 0:
        m = min(15, L)
        out[:m] = np.sort(out[:m])
    return out


def _local_page_off_by_one(pos):
    pos = np.asarray(pos, dtype=np.int64)
    return np.where(pos >= 0, (pos + 1) // 128, -1)


def _scores_sum(q_rows, k_pages):
    P = k_pages.shape[0]
    if P == 0:
        z = np.zeros((q_rows.shape[0], 0))
        return z, z.copy()
    kf = k_pages.reshape(P * 128, 128)
    dots = (q_rows @ kf.T).reshape(q_rows.shape[0], P, 128)
    absd = (np.abs(q_rows) @ np.abs(kf).T).reshape(q_rows.shape[0], P, 128)
    return dots.sum(axis=2), absd.max(axis=2)


def _scores_transposed_q(q_rows, k_pages):
    return _ORIG_SCORES(q_rows[:, ::-1].copy(), k_pages)


MUTATIONS = [
    ("nibble order swapped", nvfp4, "decode_rows", _decode_rows_swapped, ["pin_row_decode_golden"]),
    ("one scale per 8 elements", nvfp4, "decode_rows", _decode_rows_scale8, ["pin_row_decode_golden"]),
    ("E4M3 ties rounded up", formats, "e4m3_round_nonneg", _e4m3_round_ties_up,
     ["pin_scale_rounding_exhaustive", "pin_quantize_golden"]),
    ("E2M1 ties away from zero", formats, "e2m1_round", _e2m1_round_ties_away,
     ["pin_code_rounding", "pin_quantize_golden"]),
    ("zero codes lose their sign", formats, "e2m1_round", _e2m1_round_unsigned_zero,
     ["pin_code_rounding", "pin_quantize_golden"]),
    ("equal scores rank the higher id first", indexer, "select", _select_ties_high_id, ["pin_closed_forms"]),
    ("local page not written", indexer, "select", _select_no_local, ["pin_closed_forms", "pin_bruteforce"]),
    ("ids sorted ascending instead of by score", indexer, "select", _select_ascending,
     ["pin_closed_forms", "pin_bruteforce"]),
    ("local page off by one position", indexer, "local_page", _local_page_off_by_one, ["pin_bruteforce"]),
    ("page score = sum instead of max", indexer, "page_scores", _scores_sum,
     ["pin_row_decode_golden", "pin_bruteforce", "pin_closed_forms"]),
    ("query dims reversed", indexer, "page_scores", _scores_transposed_q,
     ["pin_row_decode_golden", "pin_bruteforce"]),
]


@pytest.mark.parametrize("name,mod,attr,bad,pin_names", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, mod, attr, bad, pin_names):
    for n in pin_names:                      # the pins hold before planting
        assert getattr(pins, n)() is None, n
    monkeypatch.setattr(mod, attr, bad)
    if mod is formats:                       # nvfp4 imported these names directly
        monkeypatch.setattr(nvfp4, attr, bad, raising=False)
    if mod is nvfp4 and attr == "decode_rows":
        monkeypatch.setattr(nvfp4, "decode_pages", lambda kv, phys: bad(np.asarray(kv)[np.asarray(phys, dtype=np.int64)]))
        monkeypatch.setattr(indexer, "decode_pages", lambda kv, phys: bad(np.asarray(kv)[np.asarray(phys, dtype=np.int64)]))
    assert _any_pin_fails(pin_names), f"planted mistake not caught: {name}"


# ---------------------------------------------------------------- MXFP4 pages
import test_oracle_mxfp4 as mxpins   # noqa: E402
from oracle import mxfp4             # noqa: E402

_ORIG_MX_DECODE = mxfp4.decode_pages
_ORIG_MX_QUANT = mxfp4.quantize_rows


def _mx_decode(pages, phys, swap=False, per=32, bias=127, interleaved=False):
    pg = np.asarray(pages, dtype=np.uint8)[np.asarray(phys, dtype=np.int64)]
    if interleaved:                         # 68-byte token rows instead of the split page
        rows = pg.reshape(-1, 128, 68)
        cb, sb = rows[..., :64].astype(np.int64), rows[..., 64:]
    else:
        cb = pg[:, :8192].reshape(-1, 128, 64).astype(np.int64)
        sb = pg[:, 8192:].reshape(-1, 128, 4)
    lo, hi = (cb >> 4, cb & 0xF) if swap else (cb & 0xF, cb >> 4)
    codes = np.stack([lo, hi], axis=-1).reshape(-1, 128, 128)
    sc = np.exp2(sb.astype(np.float64) - bias)
    if per == 32:
        scale = np.repeat(sc, 32, axis=-1)
    else:                                   # one scale per 16 elements, repeated
        scale = np.concatenate([np.repeat(sc, 16, axis=-1)] * 2, axis=-1)
    return formats.e2m1_value(codes) * scale


def _mx_quant_exponent(bits, shift):
    x = formats.bf16_value(bits).reshape(-1, 4, 32)
    amax = np.abs(x).max(axis=-1)
    _, e2 = np.frexp(amax)
    E = np.clip(np.where(amax > 0, e2.astype(np.int64) - 1 - shift, -127), -127, 127)
    codes = formats.e2m1_round(x / np.exp2(E.astype(np.float64))[..., None]).astype(np.int64).reshape(-1, 128)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), (E + 127).astype(np.uint8)


def _mx_quant_no_clamp(bits):
    x = formats.bf16_value(bits).reshape(-1, 4, 32)
    amax = np.abs(x).max(axis=-1)
    _, e2 = np.frexp(amax)
    E = np.where(amax > 0, e2.astype(np.int64) - 3, -127)
    codes = formats.e2m1_round(x / np.exp2(E.astype(np.float64))[..., None]).astype(np.int64).reshape(-1, 128)
    return (codes[:, 0::2] | (codes[:, 1::2] << 4)).astype(np.uint8), ((E + 127) & 0xFF).astype(np.uint8)


MX_MUTATIONS = [
    ("MXFP4 nibble order swapped", "decode_pages", lambda p, f: _mx_decode(p, f, swap=True),
     ["pin_mx_page_decode_golden", "pin_mx_round_trip"]),
    ("MXFP4 one scale per 16 elements", "decode_pages", lambda p, f: _mx_decode(p, f, per=16),
     ["pin_mx_page_decode_golden", "pin_mx_round_trip"]),
    ("MXFP4 E8M0 bias 128", "decode_pages", lambda p, f: _mx_decode(p, f, bias=128),
     ["pin_mx_page_decode_golden", "pin_mx_round_trip"]),
    ("MXFP4 interleaved 68-byte rows", "decode_pages", lambda p, f: _mx_decode(p, f, interleaved=True),
     ["pin_mx_page_decode_golden", "pin_mx_round_trip"]),
    ("MXFP4 shared exponent floor(log2 amax) - 1", "quantize_rows", lambda b: _mx_quant_exponent(b, 1),
     ["pin_mx_quantize_golden", "pin_mx_quantize_search", "pin_mx_round_trip"]),
    ("MXFP4 shared exponent not clamped", "quantize_rows", _mx_quant_no_clamp,
     ["pin_mx_quantize_golden", "pin_mx_quantize_search"]),
]


@pytest.mark.parametrize("name,attr,bad,pin_names", MX_MUTATIONS, ids=[m[0] for m in MX_MUTATIONS])
def test_planted_mxfp4_mistake_is_caught(monkeypatch, name, attr, bad, pin_names):
    for n in pin_names:
        assert getattr(mxpins, n)() is None, n
    monkeypatch.setattr(mxfp4, attr, bad)
    assert any(_fails(getattr(mxpins, n)) for n in pin_names), f"planted mistake not caught: {name}"


def _fails(pin):
    try:
        return pin() is not None
    except Exception:
        return True
