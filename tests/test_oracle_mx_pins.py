"""Pins for the oracle's power-of-two-scale FP8 quantization (no GPU).

"02 · DeepSeek-V3" (PaperTrace) §2 groups activations in 1 x 128 tiles and
weights in 128 x 128 blocks, each with a scale from the group's own max
|value|, and likens this to the microscaling formats that Blackwell's tensor
cores scale natively, where a scale is a power of two held as an 8-bit
exponent.  The exponent rule is pinned by exact rational arithmetic, the
quantizers by their defining properties, by the special case where they
coincide with the fp32-scale quantizers (already pinned by brute force), and
the FFN variant by explicit loops on a tiny input.
"""
import math
from fractions import Fraction

import numpy as np
import pytest

from oracle import moe_oracle as O

F32 = np.float32


def _least_exponent(amax: float) -> int:
    """min{e : 448 * 2^e >= amax} by exact rationals, clamped at -127."""
    a = Fraction(float(amax))
    if a == 0:
        return 0
    e = 0
    while Fraction(448) * Fraction(2) ** e < a:
        e += 1
    while Fraction(448) * Fraction(2) ** (e - 1) >= a:
        e -= 1
    return max(e, -127)


def test_exponent_worked_values():
    cases = {448.0: 0, 449.0: 1, 224.0: -1, 896.0: 1, 1.0: -8, 1.75: -8,
             0.0: 0, 3.0e38: 120}
    for a, e in cases.items():
        assert O.group_exponent_pow2(np.array([a], F32))[0] == e, a
    # one ulp above a boundary moves to the next exponent
    a = np.nextafter(F32(224.0), F32(1e9))
    assert O.group_exponent_pow2(np.array([a]))[0] == 0
    # subnormal amax: the exact exponent is below -127, so it is clamped
    tiny = np.array([2.0 ** -140, 2.0 ** -126, 2.0 ** -118], F32)
    assert O.group_exponent_pow2(tiny).tolist() == [-127, -127, -126]


def test_exponent_against_exact_rationals():
    rng = np.random.default_rng(11)
    mant = rng.uniform(1.0, 2.0, 3000)
    expo = rng.integers(-149, 128, 3000)
    a = (mant * np.exp2(expo.astype(float))).astype(F32)
    a = a[np.isfinite(a)]
    bounds = (448.0 * np.exp2(np.arange(-130, 120))).astype(F32)
    a = np.concatenate([a, bounds, np.nextafter(bounds, F32(np.inf)),
                        np.nextafter(bounds, F32(0))])
    got = O.group_exponent_pow2(a)
    want = np.array([_least_exponent(v) for v in a])
    np.testing.assert_array_equal(got, want)


def test_ue8m0_codec():
    e = np.arange(-127, 128)
    b = O.ue8m0_encode(e)
    assert b.dtype == np.uint8 and b[0] == 0 and b[127] == 127
    np.testing.assert_array_equal(O.ue8m0_decode(b),
                                  np.ldexp(1.0, e).astype(F32))


def test_quantize_1x128_pow2_properties():
    """Scales are powers of two with each tile's largest code magnitude in
    (224, 448]; each code is the E4M3 rounding of the exact quotient, so
    every element is within half a step of its value."""
    rng = np.random.default_rng(12)
    x = (rng.standard_normal((8, 512)) * np.exp(rng.uniform(-10, 10, (8, 1)))
         ).astype(F32)
    x[3, 128:256] = 0.0
    q, s = O.quantize_1x128_pow2(x)
    assert q.shape == x.shape and s.shape == (8, 4) and s.dtype == F32
    m, ex = np.frexp(s.astype(np.float64))
    assert np.all(m == 0.5)
    v = O.e4m3_decode(q).reshape(8, 4, 128)
    vmax = np.abs(v).max(axis=2)
    live = np.abs(x.reshape(8, 4, 128)).max(axis=2) > 0
    assert np.all((vmax[live] > 224.0) & (vmax[live] <= 448.0))
    assert s[3, 1] == 1.0 and np.all(q[3, 128:256] == 0)
    for r in range(8):
        for t in range(4):
            xs = x[r, 128 * t:128 * (t + 1)].astype(np.float64) / s[r, t]
            np.testing.assert_array_equal(
                q[r, 128 * t:128 * (t + 1)], O.e4m3_encode(xs.astype(F32)))
    deq = O.dequantize(q, s, 1)
    sc = np.repeat(s.astype(np.float64), 128, axis=1)
    err = np.abs(deq - x)
    normal = np.abs(x) >= sc * 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]))
    assert np.all(err[~normal] <= 2.0 ** -10 * sc[~normal])


def test_pow2_equals_fp32_quantizer_when_amax_is_448_times_a_power_of_two():
    """With amax = 448 * 2^k the fp32 scale amax / 448 is itself 2^k, so
    both quantizers must give the same codes and scales."""
    rng = np.random.default_rng(13)
    x = rng.uniform(-1, 1, (4, 384)).astype(F32)
    k = rng.integers(-20, 20, size=(4, 3))
    t = x.reshape(4, 3, 128)
    t[:, :, 0] = 1.0
    x = (t * (448.0 * np.exp2(k.astype(float)))[:, :, None]).reshape(4, 384)
    x = x.astype(F32)
    q1, s1 = O.quantize_1x128(x)
    q2, s2 = O.quantize_1x128_pow2(x)
    np.testing.assert_array_equal(s1, s2)
    np.testing.assert_array_equal(q1, q2)
    w = np.tile(x, (128, 1))[:256]
    b1, c1 = O.quantize_128x128(w)
    b2, c2 = O.quantize_128x128_pow2(w)
    np.testing.assert_array_equal(c1, c2)
    np.testing.assert_array_equal(b1, b2)


def test_quantize_128x128_pow2_blocks_are_independent():
    rng = np.random.default_rng(14)
    w = (rng.standard_normal((256, 384)) * 0.02).astype(F32)
    q, s = O.quantize_128x128_pow2(w)
    assert s.shape == (2, 3)
    w2 = w.copy()
    w2[5, 200] = 50.0
    q2, s2 = O.quantize_128x128_pow2(w2)
    mask = np.ones_like(q, bool)
    mask[:128, 128:256] = False
    np.testing.assert_array_equal(q2[mask], q[mask])
    assert s2[0, 1] > s[0, 1] and np.sum(s2 != s) == 1
    blk = np.abs(w[:128, 128:256]).max()
    e = _least_exponent(float(blk))
    assert s[0, 1] == F32(2.0 ** e)


def test_pow2_ffn_brute_force_on_tiny_input():
    """Two tokens, H = I = 128, power-of-two scales throughout (inputs,
    weights and the re-quantized intermediate): p, q, m and y by explicit
    loops over the dequantized values."""
    rng = np.random.default_rng(15)
    H = I = 128
    x = rng.standard_normal((2, H)).astype(F32)
    ws = [(rng.standard_normal((I, H)) * 0.05).astype(F32),
          (rng.standard_normal((I, H)) * 0.05).astype(F32),
          (rng.standard_normal((H, I)) * 0.05).astype(F32)]
    a_q, a_s = O.quantize_1x128_pow2(x)
    wq = [O.quantize_128x128_pow2(w) for w in ws]
    y, (m_q, m_s) = O.fp8_swiglu_ffn(a_q, a_s, *wq,
                                     requant=O.quantize_1x128_pow2)
    av = O.e4m3_decode(a_q)
    wv = [O.e4m3_decode(q) * float(s[0, 0]) for q, s in wq]
    for t in range(2):
        a = [float(av[t, h]) * float(a_s[t, 0]) for h in range(H)]
        m = []
        for i in range(I):
            p = math.fsum(a[h] * wv[0][i, h] for h in range(H))
            q = math.fsum(a[h] * wv[1][i, h] for h in range(H))
            m.append(float(F32(p / (1 + math.exp(-p)) * q)))
        e = _least_exponent(max(abs(v) for v in m))
        assert m_s[t, 0] == F32(2.0 ** e)
        codes = O.e4m3_encode((np.array(m, np.float64) / 2.0 ** e)
                              .astype(F32))
        np.testing.assert_array_equal(m_q[t], codes)
        mv = O.e4m3_decode(codes) * 2.0 ** e
        for j in range(0, H, 17):
            yj = math.fsum(mv[i] * wv[2][j, i] for i in range(I))
            assert y[t, j] == pytest.approx(yj, rel=1e-12, abs=1e-15)


def test_pow2_ffn_close_to_full_precision_ffn():
    """Power-of-two scales keep the FP8 expert within 10% (RMS) of the fp64
    SwiGLU expert, like the fp32 scales: a scale at most twice the fp32 one
    moves a group's values down at most one binade, where E4M3 keeps the
    same 3-bit relative step."""
    rng = np.random.default_rng(16)
    H, I = 256, 384
    x = rng.standard_normal((16, H)).astype(F32)
    w1, w3 = [(rng.standard_normal((I, H)) * 0.05).astype(F32)
              for _ in range(2)]
    w2 = (rng.standard_normal((H, I)) * 0.05).astype(F32)
    y, _ = O.fp8_swiglu_ffn(*O.quantize_1x128_pow2(x),
                            O.quantize_128x128_pow2(w1),
                            O.quantize_128x128_pow2(w3),
                            O.quantize_128x128_pow2(w2),
                            requant=O.quantize_1x128_pow2)
    ref = O.swiglu_ffn(x, w1, w3, w2)
    rel = np.sqrt(np.mean((y - ref) ** 2) / np.mean(ref ** 2))
    assert 1e-2 < rel < 1e-1
