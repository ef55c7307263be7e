"""The insert kernels' rounding shortcuts, replayed in fp32 emulation over
every input they can meet, against the oracle's exact rounding.

The NVFP4 insert does not divide: it rounds |x| * rcp(s) to a multiple of
2^-12 with one fused multiply-add (adding 3 * 2^10) before the hardware
E2M1 conversion, and it rounds amax * fl(1/6) to 12 significant bits
(Veltkamp's split with 2^12 + 1) before the hardware E4M3 conversion.  The
argument that both equal the exact round-to-nearest-even is in
csrc/codec.cuh; this test checks the claim itself, with no GPU: every
finite bf16 value against every positive E4M3 scale, with reciprocals one
ulp off either way (rcp.approx is within one ulp), and every bf16 amax.
The fp32 steps are emulated exactly (float64 holds each product, the sum
with 3072 and the split exactly before the final float32 rounding).
"""
import numpy as np

from oracle.formats import E4M3_POS, bf16_value, e2m1_round, e4m3_round_nonneg


def _finite_bf16():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    bits = bits[(bits & 0x7F80) != 0x7F80]
    return bf16_value(bits).astype(np.float32)


def _rn32(v):
    return np.asarray(v, np.float64).astype(np.float32)


def test_code_shortcut_equals_exact_rounding():
    x = _finite_bf16()
    ax = np.abs(x).astype(np.float64)
    bad = 0
    for s in E4M3_POS[E4M3_POS > 0]:
        r0 = np.float64(np.float32(1.0) / np.float32(s))
        for r in (np.nextafter(np.float32(r0), np.float32(0)), np.float32(r0),
                  np.nextafter(np.float32(r0), np.float32(np.inf))):
            with np.errstate(over="ignore"):
                t = _rn32(ax * np.float64(r) + 3072.0).astype(np.float64) - 3072.0   # one FMA, then exact
            t = np.where(np.isinf(t), 7.0, t)                                          # saturates either way
            got = e2m1_round(np.copysign(t, x.astype(np.float64)))
            want = e2m1_round(x.astype(np.float64) / s)
            bad += int(np.count_nonzero(got != want))
    assert bad == 0


def test_scale_shortcut_equals_exact_rounding():
    x = _finite_bf16()
    amax = np.unique(np.abs(x)).astype(np.float32)
    v = np.minimum(_rn32(amax.astype(np.float64) * np.float64(np.float32(1.0) / np.float32(6.0))),
                   np.float32(1024.0))
    c = _rn32(v.astype(np.float64) * 4097.0)
    hi = _rn32(c.astype(np.float64) + _rn32(v.astype(np.float64) - c.astype(np.float64)).astype(np.float64))
    got = e4m3_round_nonneg(hi.astype(np.float64))
    want = e4m3_round_nonneg(amax.astype(np.float64) / 6.0)
    assert np.array_equal(got, want)
