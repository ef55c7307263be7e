"""NVFP4 insert kernel: bytes bit-exact against the oracle."""
import json
import os

import numpy as np
import pytest

import workloads
from oracle import nvfp4 as onvfp4
from gpu_util import gpu_cache, oracle_cache, torch_dev, up

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("idx", [0, 1, 2, 3, 4])
def test_insert_bit_exact_small_workloads(idx):
    w = workloads.config(idx, small=True)
    got = gpu_cache(w).cpu().numpy()
    want = oracle_cache(w)
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} bytes differ"


def _edge_rows():
    """Rows that exercise every rounding rule: the hand-worked token, scale
    ties / saturation / subnormals, code ties, signed zeros, and arbitrary
    finite bf16 bit patterns."""
    g = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "nvfp4_quantize.json")))
    row = np.zeros(128, np.uint16)
    for grp in g["groups"]:
        for k, v in grp["x_bf16"].items():
            row[int(k)] = int(v, 16)
    rows = [row]
    rng = np.random.Generator(np.random.PCG64(21))
    # arbitrary finite bf16 patterns (exponent field != 0xFF)
    r = rng.integers(0, 1 << 16, size=(2048, 128), dtype=np.uint32).astype(np.uint16)
    r[(r & 0x7F80) == 0x7F80] &= 0xBFFF
    rows.append(r)
    # every midpoint of every scale: x = m * s for m in the E2M1 midpoints
    x = np.zeros((256, 128), np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.0], np.float32)
    sc = np.exp2(rng.integers(-9, 8, size=256)).astype(np.float32)
    for i in range(256):
        for gi in range(8):
            vals = mids * sc[i]
            x[i, gi * 16: gi * 16 + 8] = vals
            x[i, gi * 16 + 8: gi * 16 + 16] = -vals
    rows.append(workloads._to_bf16_bits(x))
    # amax exactly 6 * (E4M3 midpoints): scale ties
    from oracle.formats import E4M3_POS
    mid = (E4M3_POS[1:] + E4M3_POS[:-1]) / 2 * 6
    y = np.zeros((len(mid) // 8 + 1, 128), np.float32)
    for i, m in enumerate(mid):
        y[i // 8, (i % 8) * 16] = m
    rows.append(workloads._to_bf16_bits(y))
    # tiny, huge, signed zeros
    z = np.zeros((4, 128), np.float32)
    z[0, :16] = 1e-4
    z[0, 16:32] = -1e-4
    z[1, :] = -0.0
    z[2, :16] = 5000.0
    z[2, 16:32] = np.linspace(-3000, 3000, 16)
    z[3, ::3] = 2.0 ** -20
    rows.append(workloads._to_bf16_bits(z))
    return np.concatenate([np.atleast_2d(a) for a in rows], axis=0)


def test_insert_edge_values_bit_exact():
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    k = _edge_rows()
    n = k.shape[0]
    nb = (n + 127) // 128 + 1
    rng = np.random.Generator(np.random.PCG64(22))
    slots = rng.permutation(nb * 128)[:n].astype(np.int64)
    slots[::7] = -1                                   # skipped
    kv = torch.full((nb, 128, 72), 0x5A, dtype=torch.uint8, device=torch_dev())
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
    idx.insert(up(k.view(np.int16)), up(slots), kv, status=status)
    want = np.full((nb, 128, 72), 0x5A, np.uint8)
    onvfp4.insert(k, slots, want)
    got = kv.cpu().numpy()
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} bytes differ"
    assert int(status.item()) == 0


def _finite_bf16():
    from oracle.formats import bf16_value
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]             # exponent field 0xFF: inf / NaN
    return bits, bf16_value(bits)


def _bf16_floor(v):
    """Bits of the largest bf16 value below the positive real v (v < 2^128)."""
    from oracle.formats import bf16_value
    b = np.uint16(np.float32(v).view(np.uint32) >> 16)
    while bf16_value(np.array([b]))[0] >= v:
        b = np.uint16(b - 1)
    return b


def _pack_groups(groups, width):
    g = np.concatenate(groups)
    per_row = 128 // width
    pad = (-g.shape[0]) % per_row
    g = np.concatenate([g, np.zeros((pad, width), np.uint16)])
    return g.reshape(-1, 128)


def _every_value_every_scale():
    """Groups that pair every finite bf16 value with every positive E4M3
    scale it can meet.  For each scale s two kinds of group: element 0 is
    6 s (the group's scale is then exactly s) and the other 15 run over every
    x with |x| <= 6 s; or element 0 is the largest bf16 amax still rounding to
    s (just under 6 times the midpoint above s; the largest finite bf16 for
    s = 448) and the others run over every x with 6 s < |x| <= amax, where the
    quotient saturates or sits just under 6."""
    from oracle.formats import E4M3_POS, bf16_value, e4m3_round_nonneg
    bits, val = _finite_bf16()
    pos = E4M3_POS[E4M3_POS > 0]
    groups = []
    for i, s in enumerate(pos):
        a = 6.0 * s
        a_bits = np.uint16(np.float32(a).view(np.uint32) >> 16)
        assert bf16_value(np.array([a_bits]))[0] == a
        top = _bf16_floor(3 * (s + pos[i + 1])) if i + 1 < pos.size else np.uint16(0x7F7F)
        top_v = bf16_value(np.array([top]))[0]
        assert e4m3_round_nonneg(np.array([top_v / 6.0]))[0] == i + 1     # byte i+1 holds pos[i]
        for amax_bits, sel in ((a_bits, np.abs(val) <= a),
                               (top, (np.abs(val) > a) & (np.abs(val) <= top_v))):
            xs = bits[sel]
            xs = np.concatenate([xs, np.zeros((-xs.size) % 15, np.uint16)]).reshape(-1, 15)
            groups.append(np.concatenate([np.full((xs.shape[0], 1), amax_bits, np.uint16), xs], 1))
    return _pack_groups(groups, 16)


def _every_amax():
    """One group per finite non-zero bf16 value, alone in its group: every
    amax the scale rounding can see."""
    bits, val = _finite_bf16()
    bits = bits[val != 0]
    g = np.zeros((bits.size, 16), np.uint16)
    g[:, 0] = bits
    return _pack_groups([g], 16)


@pytest.mark.parametrize("kind", ["every_value_every_scale", "every_amax"])
def test_insert_exhaustive_bit_exact(kind):
    """Every finite bf16 key value against every E4M3 scale, and every
    amax: the kernel's bytes equal the oracle's exact rounding."""
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    k = _every_value_every_scale() if kind == "every_value_every_scale" else _every_amax()
    n = k.shape[0]
    nb = (n + 127) // 128
    slots = np.arange(n, dtype=np.int64)
    kv = torch.zeros((nb, 128, 72), dtype=torch.uint8, device=torch_dev())
    idx.insert(up(k.view(np.int16)), up(slots), kv)
    want = onvfp4.insert(k, slots, np.zeros((nb, 128, 72), np.uint8))
    got = kv.cpu().numpy()
    assert np.array_equal(got, want), f"{np.count_nonzero(got != want)} bytes differ"


def test_insert_out_of_range_slot_sets_status_and_skips():
    import torch
    import sparse_attention_block_nvfp4_gb300 as idx
    rng = np.random.Generator(np.random.PCG64(23))
    k = workloads._to_bf16_bits(rng.standard_normal((3, 128), dtype=np.float32))
    kv = torch.zeros((2, 128, 72), dtype=torch.uint8, device=torch_dev())
    status = torch.zeros(1, dtype=torch.int32, device=torch_dev())
    idx.insert(up(k.view(np.int16)), up(np.array([5, 256, 300], np.int64)), kv, status=status)
    got = kv.cpu().numpy()
    assert int(status.item()) == idx.STATUS_BAD_SLOT
    assert np.array_equal(got[0, 5], onvfp4.quantize_rows(k[:1])[0])
    assert np.count_nonzero(got) == np.count_nonzero(got[0, 5])


def test_insert_full_size_cache_sampled():
    """The long mixed step's full cache (2.24 M tokens): every token inserted
    by the kernel; a random sample of 16384 rows checked against the oracle."""
    w = workloads.config(4)
    got = gpu_cache(w).cpu().numpy().reshape(-1, 72)
    rng = np.random.Generator(np.random.PCG64(24))
    pick = rng.choice(w.k_bf16.shape[0], size=16384, replace=False)
    want = onvfp4.quantize_rows(w.k_bf16[pick])
    assert np.array_equal(got[w.slot_mapping[pick]], want)
