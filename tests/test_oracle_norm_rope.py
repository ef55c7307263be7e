"""Pins of the qk-norm + RoPE oracle (oracle/norm_rope.py), and planted
mistakes each caught by one of them.

The pins: a hand-worked one-hot key (tests/golden/norm_rope_onehot.json)
fixes the rotation's sign, the pairing, the cos / sin column order and the
pass-through past rotary_dim; closed forms fix the RMS scale (unit mean
square for eps = 0, ms / (ms + eps) otherwise) and the weight; the
rotation keeps every claimed pair's norm and is the identity at angle 0;
the fp32 sum order stays within fp32 error of a float64 evaluation; the
bf16 rounding equals torch's float32 -> bfloat16 conversion.
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
            a = nr.norm_rope_f32(k, np.zeros(64, np.int64), w, 1e-6, _table([0.0], rd), rd, neox)
            b = nr.norm_rope_f32(k, np.zeros(64, np.int64), w, 1e-6, _table([0.0], 0), 0, neox)
            if not np.array_equal(a, b):
                return f"angle 0 changed the key (neox={neox}, rd={rd})"
    return None


def pin_pair_norms_kept():
    k = _rand_keys(64, 2)
    w = _bf16(np.ones(128))
    ang = np.random.Generator(np.random.PCG64(3)).uniform(-np.pi, np.pi, 64)
    for neox in (True, False):
        for rd in (128, 64):
            y = nr.norm_rope_f32(k, np.zeros(64, np.int64), w, 1e-6, _table([0.0], 0), 0, neox)
            o = nr.norm_rope_f32(k, np.arange(64), w, 1e-6, _table(ang, rd), rd, neox)
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
            y = nr.norm_rope_f32(k[r:r + 1], [0], w, eps, _table([0.0], 0), 0, True).astype(np.float64)
            got, want = (y * y).mean(), ms[r] / (ms[r] + eps)
            if abs(got - want) > 1e-5 * want:
                return f"mean square of the normed key {got} != {want} (eps {eps})"
    return None


def pin_weight_elementwise():
    k = _rand_keys(32, 5)
    rng = np.random.Generator(np.random.PCG64(6))
    wv = np.exp2(rng.integers(-3, 4, 128)).astype(np.float32)       # powers of two: exact scaling
    y1 = nr.norm_rope_f32(k, np.zeros(32, np.int64), _bf16(np.ones(128)), 1e-6, _table([0.0], 0), 0, True)
    yw = nr.norm_rope_f32(k, np.zeros(32, np.int64), _bf16(wv), 1e-6, _table([0.0], 0), 0, True)
    if not np.array_equal(yw, y1 * wv[None, :]):
        return "weight not applied element by element"
    return None


def pin_sum_order_within_fp32_error():
    k = _rand_keys(256, 7)
    x = nr.bf16_to_f32(k).astype(np.float64)
    exact = 1.0 / np.sqrt((x * x).mean(1) + np.float64(np.float32(1e-6)))
    got = nr.rms_scale(nr.bf16_to_f32(k), 1e-6).astype(np.float64)
    if np.any(np.abs(got - exact) > 2.0 ** -20 * exact):
        return "rms scale off by more than fp32 error"
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
        pin_weight_elementwise, pin_sum_order_within_fp32_error, pin_bf16_rounding_matches_torch,
        pin_insert_skips]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    assert pin() is None


# ---------------------------------------------------------------- planted mistakes
_orig_rotate = nr.rotate
_orig_f32 = nr.norm_rope_f32


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


def _f32_weight_reversed(k, positions, w, eps, cache, rd, neox):
    return _orig_f32(k, positions, np.asarray(w)[::-1].copy(), eps, cache, rd, neox)


def _f32_weight_ignored(k, positions, w, eps, cache, rd, neox):
    return _orig_f32(k, positions, _bf16(np.ones(128)), eps, cache, rd, neox)


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
    ("bf16 by truncation", "f32_to_bf16", _bf16_truncate, ["pin_bf16_rounding_matches_torch"]),
    ("weight reversed", "norm_rope_f32", _f32_weight_reversed, ["pin_weight_elementwise"]),
    ("weight ignored", "norm_rope_f32", _f32_weight_ignored, ["pin_weight_elementwise"]),
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
