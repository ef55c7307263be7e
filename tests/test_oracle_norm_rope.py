"""Pins of the qk-norm + RoPE oracle (oracle/norm_rope.py), and planted
mistakes each caught by one of them.

The pins: a hand-worked one-hot key (tests/golden/norm_rope_onehot.json)
fixes the rotation's sign, the pairing, the cos / sin column order and the
pass-through past rotary_dim; closed forms fix the RMS scale (unit mean
square for eps = 0, ms / (ms + eps) otherwise) and the weight; the mean
square equals the exact rational mean of tiny keys; the rotation keeps every
claimed pair's norm and is the identity at angle 0; the single float64 ->
bf16 rounding agrees with torch where the value is an fp32 number and
rounds exact midpoints to even and near-midpoints the right way; the fp32
error bound covers fp32 evaluations of the formula in several orders, and
the row check accepts their quantised rows and rejects a planted wrong one.
"""
import json
import os

import numpy as np
import pytest

from oracle import norm_rope as nr
from oracle import nvfp4 as onvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "norm_rope_onehot.json")


def _bf16(x):
    return nr.f32_to_bf16(np.asarray(x, np.float32))


def _table(angles_rad, rd):
    """cos / sin table rows [len(angles), rd] for one angle per row, the same
    angle on every pair (enough for the pins)."""
    a = np.asarray(angles_rad, np.float64)[:, None]
    h = rd // 2
    return np.concatenate([np.repeat(np.cos(a), h, 1), np.repeat(np.sin(a), h, 1)], 1).astype(np.float32)


def _rand_keys(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    return _bf16(rng.standard_normal((n, 128)) * np.exp2(rng.integers(-4, 5, size=(n, 1))))


def pin_onehot_golden():
    g = json.load(open(GOLDEN))
    for c in g["cases"]:
        rd = c["rotary_dim"]
        k = np.zeros((1, 128), np.uint16)
        k[0, c["hot"]] = _bf16([2.0])[0]
        table = np.zeros((1, rd), np.float32)
        table[0, : rd // 2] = np.float32(g["cos"])
        table[0, rd // 2:] = np.float32(g["sin"])
        out = nr.bf16_to_f32(nr.norm_rope_bf16(k, [0], _bf16(np.ones(128)), 0.0, table, rd,
                                               c["style"] == "neox"))[0].astype(np.float64)
        want = np.zeros(128)
        for i, v in c["expect"].items():
            want[int(i)] = v
        if np.any(np.abs(out - want) > 2.0 ** -8 * np.abs(want) + 1e-30):
            return f"{c}: got {out[np.nonzero(out)[0]]} at {np.nonzero(out)[0]}"
    return None


def pin_angle_zero_is_identity():
    k = _rand_keys(64, 1)
    w = _bf16(np.linspace(0.5, 2.0, 128))
    for neox in (True, False):
        for rd in (128, 64, 32):
            a = nr.norm_rope_f64(k, np.zeros(64, np.int64), w, 1e-6, _table([0.0], rd), rd, neox)
            b = nr.norm_rope_f64(k, np.zeros(64, np.int64), w, 1e-6, _table([0.0], 0), 0, neox)
            if not np.array_equal(a, b):
                return f"angle 0 changed the key (neox={neox}, rd={rd})"
    return None


def pin_pair_norms_kept():
    k = _rand_keys(64, 2)
    w = _bf16(np.ones(128))
    ang = np.random.Generator(np.random.PCG64(3)).uniform(-np.pi, np.pi, 64)
    for neox in (True, False):
        for rd in (128, 64):
            y = nr.norm_rope_f64(k, np.zeros(64, np.int64), w, 1e-6, _table([0.0], 0), 0, neox)
            o = nr.norm_rope_f64(k, np.arange(64), w, 1e-6, _table(ang, rd), rd, neox)
            h = rd // 2
            i1 = np.arange(h) if neox else np.arange(0, rd, 2)
            i2 = i1 + h if neox else i1 + 1
            n_y = y[:, i1].astype(np.float64) ** 2 + y[:, i2].astype(np.float64) ** 2
            n_o = o[:, i1].astype(np.float64) ** 2 + o[:, i2].astype(np.float64) ** 2
            if np.any(np.abs(n_o - n_y) > 1e-5 * n_y + 1e-30):
                return f"pair norms changed (neox={neox}, rd={rd})"
            if not np.array_equal(o[:, rd:], y[:, rd:]):
                return f"elements past rotary_dim changed (neox={neox}, rd={rd})"
    return None


def pin_rms_closed_form():
    """mean(y^2) of the normed key (weight 1, no rotation) is ms / (ms + eps),
    ms = mean(x^2): 1 for eps = 0, 2/3 and 1/2 for eps = ms/2 and ms."""
    k = _rand_keys(16, 4)
    x = nr.bf16_to_f32(k).astype(np.float64)
    ms = (x * x).mean(1)
    w = _bf16(np.ones(128))
    for r in range(16):
        for eps in (0.0, float(np.float32(ms[r] / 2)), float(np.float32(ms[r]))):
            y = nr.norm_rope_f64(k[r:r + 1], [0], w, eps, _table([0.0], 0), 0, True).astype(np.float64)
            got, want = (y * y).mean(), ms[r] / (ms[r] + eps)
            if abs(got - want) > 1e-12 * want:
                return f"mean square of the normed key {got} != {want} (eps {eps})"
    return None


def pin_weight_elementwise():
    k = _rand_keys(32, 5)
    rng = np.random.Generator(np.random.PCG64(6))
    wv = np.exp2(rng.integers(-3, 4, 128)).astype(np.float32)       # powers of two: exact scaling
    y1 = nr.norm_rope_f64(k, np.zeros(32, np.int64), _bf16(np.ones(128)), 1e-6, _table([0.0], 0), 0, True)
    yw = nr.norm_rope_f64(k, np.zeros(32, np.int64), _bf16(wv), 1e-6, _table([0.0], 0), 0, True)
    if not np.array_equal(yw, y1 * wv[None, :]):
        return "weight not applied element by element"
    return None


def pin_mean_square_exact():
    """On keys whose squares sum exactly in float64 (a few binades), the
    oracle's scale is 1 / sqrt of the exact rational mean of the squares
    plus eps, to float64 rounding."""
    from fractions import Fraction
    rng = np.random.Generator(np.random.PCG64(7))
    k = _bf16(rng.standard_normal((24, 128)) * np.exp2(rng.integers(-3, 4, size=(24, 128))))
    x = nr.bf16_to_f32(k).astype(np.float64)
    eps = float(np.float32(1e-6))
    got = nr.rms_scale(x, eps)
    for r in range(24):
        ms = sum(Fraction(float(v)) ** 2 for v in x[r]) / 128 + Fraction(eps)
        want = 1.0 / np.sqrt(float(ms))
        if abs(got[r] - want) > 4 * 2.0 ** -53 * want:
            return f"row {r}: rms scale {got[r]} != exact {want}"
    return None


def _fp32_eval(k, pos, w, eps, table, rd, neox, order):
    """The formula in fp32 (numpy float32 arithmetic, each operation rounded),
    summing the squares in the given order: 'seq', 'rev', 'pairwise' or
    'groups' (per 16-element group, then a tree)."""
    x = nr.bf16_to_f32(k).reshape(-1, 128)
    sq = x * x
    if order == "seq":
        ss = np.zeros(x.shape[0], np.float32)
        for i in range(128):
            ss = ss + sq[:, i]
    elif order == "rev":
        ss = np.zeros(x.shape[0], np.float32)
        for i in range(127, -1, -1):
            ss = ss + sq[:, i]
    elif order == "pairwise":
        t = sq
        while t.shape[1] > 1:
            t = t[:, 0::2] + t[:, 1::2]
        ss = t[:, 0]
    else:
        g = np.zeros((x.shape[0], 8), np.float32)
        for i in range(16):
            g = g + sq[:, i::16][:, :8] if False else g + sq.reshape(-1, 8, 16)[:, :, i]
        ss = ((g[:, 0] + g[:, 1]) + (g[:, 2] + g[:, 3])) + ((g[:, 4] + g[:, 5]) + (g[:, 6] + g[:, 7]))
    v = ss * np.float32(1.0 / 128.0) + np.float32(eps)
    rs = np.float32(1.0) / np.sqrt(v)
    y = (x * rs[:, None]) * nr.bf16_to_f32(w)[None, :]
    if rd == 0:
        return y
    cache = np.asarray(table, np.float32)[np.asarray(pos)]
    h = rd // 2
    c, s = cache[:, :h], cache[:, h:rd]
    i1, i2 = (np.arange(h), np.arange(h) + h) if neox else (np.arange(0, rd, 2), np.arange(1, rd, 2))
    y1, y2 = y[:, i1].copy(), y[:, i2].copy()
    y[:, i1] = y1 * c - y2 * s
    y[:, i2] = y2 * c + y1 * s
    return y


def _rope_case(n, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    x = rng.standard_normal((n, 128)) * np.exp2(rng.integers(-6, 7, size=(n, 1)))
    x[:, rng.integers(0, 128, 4)] *= 8.0
    k = _bf16(x)
    w = _bf16(rng.uniform(0.25, 2.0, 128))
    ang = np.arange(512)[:, None] * 10000.0 ** (-np.arange(64) / 64.0)[None, :]
    table = np.concatenate([np.cos(ang), np.sin(ang)], 1).astype(np.float32)
    pos = rng.integers(0, 512, n)
    return k, w, pos, table


def pin_fp32_bound_covers_fp32_orders():
    """An fp32 evaluation of the formula, the squares summed in any of four
    orders, stays within fp32_error_bound of the float64 value."""
    k, w, pos, table = _rope_case(2000, 11)
    for rd, neox in ((128, True), (64, False), (0, True)):
        tb = table if rd == 128 else (table[:, np.r_[0:32, 64:96]] if rd == 64 else None)
        v = nr.norm_rope_f64(k, pos, w, 1e-6, tb, rd, neox)
        d = nr.fp32_error_bound(k, pos, w, 1e-6, tb, rd, neox)
        for order in ("seq", "rev", "pairwise", "groups"):
            v32 = _fp32_eval(k, pos, w, 1e-6, tb, rd, neox, order).astype(np.float64)
            if np.any(np.abs(v32 - v) > d):
                return f"rd {rd} neox {neox} order {order}: fp32 value outside the bound"
    return None


def pin_row_check_accepts_fp32_and_rejects_wrong():
    """check_rows accepts the quantised rows of every fp32 evaluation order;
    accepts a row quantised from a key with one boundary element at its
    other bf16 neighbour (a row that differs from the float64 key's) and
    rejects the same flip of an element that is not near a boundary; rejects
    a row with one code changed, and keys truncated to bf16 instead of
    rounded."""
    k, w, pos, table = _rope_case(4000, 12)
    for order in ("seq", "rev", "pairwise", "groups"):
        v32 = _fp32_eval(k, pos, w, 1e-6, table, 128, True, order)
        rows = onvfp4.quantize_rows(nr.f32_to_bf16(v32))
        rep = nr.check_rows(rows, k, pos, w, 1e-6, table, 128, True)
        if rep["fails"]:
            return f"order {order}: {rep}"
    b0, b1, amb = nr.bf16_choices(k, pos, w, 1e-6, table, 128, True)
    base = onvfp4.quantize_rows(b0)
    flipped_amb = flipped_far = 0
    for t in range(k.shape[0]):
        for e in np.nonzero(amb[t])[0][:2].tolist() + [int(np.argmax(np.abs(nr.bf16_to_f32(b0[t]))))]:
            key = b0[t].copy()
            key[e] = b1[t, e]
            row = onvfp4.quantize_rows(key[None, :])
            if np.array_equal(row[0], base[t]):
                continue                                  # the flip does not change the row
            rep = nr.check_rows(row, k[t:t + 1], pos[t:t + 1], w, 1e-6, table, 128, True)
            if amb[t, e]:
                if rep["fails"] or rep["allowance"] != 1:
                    return f"token {t}: a boundary element at its other neighbour was rejected"
                flipped_amb += 1
            else:
                if rep["fails"] != 1:
                    return f"token {t}: an element far from a boundary was accepted at its other neighbour"
                flipped_far += 1
    if flipped_amb == 0 or flipped_far == 0:
        return f"allowance not exercised ({flipped_amb} boundary flips, {flipped_far} far flips)"
    rows = onvfp4.quantize_rows(nr.norm_rope_bf16(k, pos, w, 1e-6, table, 128, True))
    bad = rows.copy()
    bad[5, 3] ^= 0x11
    if nr.check_rows(bad, k, pos, w, 1e-6, table, 128, True)["fail_rows"] != [5]:
        return "a changed code byte was accepted"
    trunc = (nr.norm_rope_f64(k, pos, w, 1e-6, table, 128, True).astype(np.float32).view(np.uint32) >> 16)
    rows_t = onvfp4.quantize_rows(trunc.astype(np.uint16))
    if nr.check_rows(rows_t, k, pos, w, 1e-6, table, 128, True)["fails"] < 100:
        return "keys truncated to bf16 were accepted"
    return None


def pin_f64_bf16_single_rounding():
    """float64 -> bf16 is ONE rounding: exact midpoints go to the even
    neighbour, a value a hair above (below) a midpoint goes up (down) --
    where rounding through fp32 first would tie wrongly -- and signed zeros
    and subnormals keep their sign."""
    one = 1.0
    ulp = 2.0 ** -7                                    # bf16 spacing in [1, 2)
    cases = [
        (one + ulp / 2, 0x3F80),                       # tie -> even (1.0)
        (one + 3 * ulp / 2, 0x3F82),                   # tie -> even (1 + 2 ulp)
        (one + ulp / 2 + 2.0 ** -40, 0x3F81),          # above the tie: fp32 would round to the tie
        (one + ulp / 2 - 2.0 ** -40, 0x3F80),
        (-(one + ulp / 2 + 2.0 ** -40), 0xBF81),
        (-0.0, 0x8000), (0.0, 0x0000),
        (2.0 ** -133, 0x0001), (-(2.0 ** -133), 0x8001),   # smallest subnormal
        (2.0 ** -134, 0x0000),                         # half of it: tie -> even (zero)
        (2.0 ** -134 + 2.0 ** -160, 0x0001),
    ]
    x = np.array([c[0] for c in cases])
    want = np.array([c[1] for c in cases], np.uint16)
    got = nr.f64_to_bf16(x)
    if not np.array_equal(got, want):
        return f"got {[hex(v) for v in got]}, want {[hex(v) for v in want]}"
    return None


def pin_bf16_rounding_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.Generator(np.random.PCG64(8))
    u = rng.integers(0, 1 << 32, 200000, dtype=np.uint64).astype(np.uint32)
    u = u[(u & 0x7F800000) != 0x7F800000]
    ties = (rng.integers(0, 1 << 16, 1000, dtype=np.uint32) << 16) | 0x8000   # exact ties
    ties = ties[(ties & 0x7F800000) != 0x7F800000]
    x = np.concatenate([u, ties]).view(np.float32)
    want = torch.from_numpy(x.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = nr.f32_to_bf16(x)
    if not np.array_equal(got, want):
        return f"{np.count_nonzero(got != want)} bf16 roundings differ from torch"
    big = np.abs(x.astype(np.float64)) < 3.38e38           # f64_to_bf16 refuses values past bf16's range
    got64 = nr.f64_to_bf16(x.astype(np.float64)[big])
    if not np.array_equal(got64, want[big]):
        return f"{np.count_nonzero(got64 != want[big])} float64 -> bf16 roundings differ from torch"
    return None


def pin_insert_skips():
    k = _rand_keys(4, 9)
    pages = np.full((1, 128, 72), 0xAB, np.uint8)
    table = _table([0.1, 0.2], 64)
    nr.insert(k, [0, 1, 5, -1], [3, -1, 4, 6], _bf16(np.ones(128)), 1e-6, table, 64, True, pages)
    if not np.array_equal(pages[0, 3], onvfp4.quantize_rows(nr.norm_rope_bf16(k[:1], [0], _bf16(np.ones(128)),
                                                                               1e-6, table, 64, True))[0]):
        return "inserted row differs from quantising the normed, rotated key"
    untouched = [r for r in range(128) if r != 3]
    if np.any(pages[0, untouched] != 0xAB):
        return "a skipped token (negative slot or position outside the table) was written"
    return None


PINS = [pin_onehot_golden, pin_angle_zero_is_identity, pin_pair_norms_kept, pin_rms_closed_form,
        pin_weight_elementwise, pin_mean_square_exact, pin_bf16_rounding_matches_torch,
        pin_f64_bf16_single_rounding, pin_fp32_bound_covers_fp32_orders,
        pin_row_check_accepts_fp32_and_rejects_wrong, pin_insert_skips]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    assert pin() is None


# ---------------------------------------------------------------- planted mistakes
_orig_rotate = nr.rotate
_orig_f64 = nr.norm_rope_f64
_orig_bound = nr.fp32_error_bound
_orig_check = nr.check_rows


def _rotate_sign_flipped(y, cos, sin, rd, neox):
    return _orig_rotate(y, cos, -sin, rd, neox)


def _rotate_pairs_swapped(y, cos, sin, rd, neox):
    return _orig_rotate(y, cos, sin, rd, not neox)


def _rotate_cos_sin_swapped(y, cos, sin, rd, neox):
    return _orig_rotate(y, sin, cos, rd, neox)


def _rotate_whole_key(y, cos, sin, rd, neox):
    if rd == 0:
        return y.copy()
    h = rd // 2
    reps = 64 // h
    return _orig_rotate(y, np.tile(cos, reps), np.tile(sin, reps), 128, neox)


def _rms_eps_after_sqrt(x, eps):
    sq = (x * x).astype(np.float64).mean(1)
    return (1.0 / (np.sqrt(sq) + eps)).astype(np.float32)


def _rms_mean_over_64(x, eps):
    sq = (x * x).astype(np.float64).sum(1) / 64.0
    return (1.0 / np.sqrt(sq + eps)).astype(np.float32)


def _rms_no_sqrt(x, eps):
    sq = (x * x).astype(np.float64).mean(1)
    return (1.0 / (sq + eps)).astype(np.float32)


def _bf16_truncate(x):
    x = np.ascontiguousarray(x, dtype=np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _bf16_truncate64(x):
    x = np.asarray(x, dtype=np.float64).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


def _bound_without_sum_error(k, positions, w, eps, cache, rd, neox):
    v = _orig_f64(k, positions, w, eps, cache, rd, neox)
    return 3 * 2.0 ** -24 * np.abs(v)


def _check_accepts_all(rows, *a, **kw):
    rep = _orig_check(rows, *a, **kw)
    return dict(rep, fails=0, fail_rows=[])


def _f32_weight_reversed(k, positions, w, eps, cache, rd, neox):
    return _orig_f64(k, positions, np.asarray(w)[::-1].copy(), eps, cache, rd, neox)


def _f32_weight_ignored(k, positions, w, eps, cache, rd, neox):
    return _orig_f64(k, positions, _bf16(np.ones(128)), eps, cache, rd, neox)


MUTATIONS = [
    ("rotation sign flipped", "rotate", _rotate_sign_flipped, ["pin_onehot_golden"]),
    ("NeoX / GPT-J pairing swapped", "rotate", _rotate_pairs_swapped,
     ["pin_onehot_golden", "pin_pair_norms_kept"]),
    ("cos / sin columns swapped", "rotate", _rotate_cos_sin_swapped, ["pin_onehot_golden"]),
    ("elements past rotary_dim rotated", "rotate", _rotate_whole_key,
     ["pin_onehot_golden", "pin_pair_norms_kept"]),
    ("eps added after the square root", "rms_scale", _rms_eps_after_sqrt, ["pin_rms_closed_form"]),
    ("mean over 64 elements", "rms_scale", _rms_mean_over_64, ["pin_onehot_golden", "pin_rms_closed_form"]),
    ("no square root", "rms_scale", _rms_no_sqrt, ["pin_onehot_golden", "pin_rms_closed_form"]),
    ("bf16 by truncation (fp32 path)", "f32_to_bf16", _bf16_truncate, ["pin_bf16_rounding_matches_torch"]),
    ("bf16 by truncation (float64 path)", "f64_to_bf16", _bf16_truncate64,
     ["pin_bf16_rounding_matches_torch", "pin_f64_bf16_single_rounding"]),
    ("weight reversed", "norm_rope_f64", _f32_weight_reversed, ["pin_weight_elementwise"]),
    ("weight ignored", "norm_rope_f64", _f32_weight_ignored, ["pin_weight_elementwise"]),
    ("error bound without the summation term", "fp32_error_bound", _bound_without_sum_error,
     ["pin_fp32_bound_covers_fp32_orders"]),
    ("row check accepts any row", "check_rows", _check_accepts_all,
     ["pin_row_check_accepts_fp32_and_rejects_wrong"]),
]


def _fails(pin):
    try:
        return pin() is not None
    except Exception:
        return True


@pytest.mark.parametrize("name,attr,bad,pins", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(monkeypatch, name, attr, bad, pins):
    by_name = {p.__name__: p for p in PINS}
    for n in pins:
        assert by_name[n]() is None, n
    monkeypatch.setattr(nr, attr, bad)
    assert any(_fails(by_name[n]) for n in pins), f"planted mistake not caught: {name}"
