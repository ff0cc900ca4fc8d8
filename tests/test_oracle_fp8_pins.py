"""Pins for the oracle's FP8 (E4M3) quantization (no GPU).

"02 · DeepSeek-V3" (PaperTrace) §2, mixed precision: every tensor in E4M3
(4 exponent bits, 3 mantissa bits); activations scaled per 1 x 128 tile
(one token, 128 channels), weights per 128 x 128 block, each scale from the
group's own max |value|.  The codec is pinned to published facts of the
format and to brute force over its value table; the quantizers to the
properties the pages give for fine-grained groups (an outlier only affects
its own group) and to exact round trips.
"""
import math

import numpy as np
import pytest

from oracle import moe_oracle as O

F32 = np.float32
CODES = np.arange(256, dtype=np.uint8)


def _table():
    v = O.e4m3_decode(CODES[:0x7F])        # the non-negative finite codes
    return v


def test_e4m3_published_constants():
    """Largest finite 448, smallest normal 2^-6, smallest subnormal 2^-9,
    1.0 = 0x38 (exponent bias 7), NaN only at 0x7F / 0xFF, no infinity."""
    v = O.e4m3_decode(CODES)
    assert v[0x7E] == 448.0 and v[0xFE] == -448.0
    assert v[0x08] == 2.0 ** -6 and v[0x01] == 2.0 ** -9
    assert v[0x38] == 1.0 and v[0x40] == 2.0 and v[0x30] == 0.5
    assert set(np.nonzero(np.isnan(v))[0].tolist()) == {0x7F, 0xFF}
    assert not np.any(np.isinf(v))
    assert np.all(np.diff(_table()) > 0)          # increasing in code order
    assert len(_table()) == 127                    # +0 and 126 magnitudes
    np.testing.assert_array_equal(v[0x80:0xFF], -v[0x00:0x7F])


def _nearest_even(x, table):
    """Brute force: the table entry nearest |x|, ties to the even code."""
    a = abs(float(x))
    if a >= 448.0:
        return 0x7E
    d = np.abs(table - a)
    best = np.nonzero(d == d.min())[0]
    return int(best[0] if len(best) == 1 else best[best % 2 == 0][0])


def test_encode_is_nearest_value_ties_to_even():
    t = _table()
    rng = np.random.default_rng(0)
    xs = np.concatenate([
        rng.uniform(-460, 460, 4000), rng.uniform(-1, 1, 4000),
        rng.uniform(-0.02, 0.02, 4000),
        (t[:-1] + t[1:]) / 2,                      # every midpoint
        -(t[:-1] + t[1:]) / 2,
        t, [447.9, 448.0, 449.0, 463.99, 464.0, 1e6, -1e6]]).astype(F32)
    got = O.e4m3_encode(xs)
    for x, c in zip(xs, got):
        want = _nearest_even(x, t) | (0x80 if np.signbit(x) else 0)
        assert c == want, (float(x), int(c), want)


def test_encode_subnormal_ties_and_signed_zero():
    assert O.e4m3_encode(np.array([2.0 ** -10], F32))[0] == 0x00   # tie -> 0
    assert O.e4m3_encode(np.array([3 * 2.0 ** -10], F32))[0] == 0x02
    assert O.e4m3_encode(np.array([-1e-30], F32))[0] == 0x80       # -0
    assert O.e4m3_encode(np.array([0.0], F32))[0] == 0x00


def test_quantize_1x128_scale_and_error_bound():
    """Each tile's largest magnitude maps to +-448; every element is within
    half a step: 2^-4 relative in the normal range, 2^-10 s below it."""
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((6, 512)) * np.exp(rng.uniform(-8, 8, (6, 1)))
         ).astype(F32)
    q, s = O.quantize_1x128(x)
    assert q.shape == x.shape and s.shape == (6, 4) and s.dtype == F32
    v = O.e4m3_decode(q)
    assert np.all(np.abs(v).reshape(6, 4, 128).max(axis=2) == 448.0)
    deq = O.dequantize(q, s, 1)
    sc = np.repeat(s.astype(np.float64), 128, axis=1)
    err = np.abs(deq - x)
    normal = np.abs(x) >= sc * 2.0 ** -6
    assert np.all(err[normal] <= 2.0 ** -4 * np.abs(x[normal]) * (1 + 1e-6))
    assert np.all(err[~normal] <= 2.0 ** -10 * sc[~normal] * (1 + 1e-6))


def test_outlier_stays_in_its_tile():
    """The pages' reason for small groups: one outlier sets the scale of its
    own 1x128 tile only.  Raising one element of tile 0 leaves the other
    tiles' codes unchanged, while a single per-tensor scale (the practice
    the pages contrast) loses them to underflow."""
    rng = np.random.default_rng(2)
    x = rng.standard_normal((2, 512)).astype(F32)
    q0, _ = O.quantize_1x128(x)
    y = x.copy()
    y[0, 5] = 1e5
    q1, s1 = O.quantize_1x128(y)
    np.testing.assert_array_equal(q1[:, 128:], q0[:, 128:])
    np.testing.assert_array_equal(q1[1], q0[1])
    s_tensor = F32(np.abs(y).max() / 448.0)
    qw = O.e4m3_encode((y / s_tensor).astype(F32))
    whole = O.e4m3_decode(qw) * s_tensor
    err_tile = np.abs(O.dequantize(q1, s1, 1) - y)[:, 128:].mean()
    err_whole = np.abs(whole - y)[:, 128:].mean()
    assert err_whole > 4 * err_tile
    zero = lambda q: np.mean((q[:, 128:] & 0x7F) == 0)   # noqa: E731
    assert zero(qw) > 0.1 and zero(q1) < 0.01


def test_quantize_128x128_blocks_are_independent_and_exact_on_grid():
    """Values already on the E4M3 grid times a power of two, with 448 in
    every block, come back exactly; changing one block changes only its
    own codes and scale."""
    rng = np.random.default_rng(3)
    t = _table()
    codes = rng.choice(t, size=(256, 384)) * rng.choice([-1.0, 1.0],
                                                       size=(256, 384))
    codes[::128, ::128] = 448.0
    k = rng.integers(-6, 6, size=(2, 3)).astype(float)
    w = (codes * np.exp2(np.repeat(np.repeat(k, 128, 0), 128, 1))).astype(F32)
    q, s = O.quantize_128x128(w)
    assert s.shape == (2, 3)
    np.testing.assert_array_equal(s, np.exp2(k).astype(F32))
    np.testing.assert_array_equal(O.dequantize(q, s, 128), w)
    w2 = w.copy()
    w2[130, 300] = 1e4
    q2, s2 = O.quantize_128x128(w2)
    mask = np.ones_like(q, bool)
    mask[128:, 256:] = False
    np.testing.assert_array_equal(q2[mask], q[mask])
    assert s2[1, 2] != s[1, 2] and np.sum(s2 != s) == 1


def test_all_zero_group_has_unit_scale_and_zero_codes():
    q, s = O.quantize_1x128(np.zeros((1, 256), F32))
    assert np.all(s == 1.0) and np.all(q == 0)


def test_fp8_ffn_brute_force_on_tiny_input():
    """Two tokens, H = I = 128: p, q, m and y by explicit loops over the
    dequantized values, against the matrix form."""
    rng = np.random.default_rng(4)
    H = I = 128
    x = rng.standard_normal((2, H)).astype(F32)
    ws = [(rng.standard_normal((I, H)) * 0.05).astype(F32),
          (rng.standard_normal((I, H)) * 0.05).astype(F32),
          (rng.standard_normal((H, I)) * 0.05).astype(F32)]
    a_q, a_s = O.quantize_1x128(x)
    wq = [O.quantize_128x128(w) for w in ws]
    y, (m_q, m_s) = O.fp8_swiglu_ffn(a_q, a_s, *wq)
    av = O.e4m3_decode(a_q)
    wv = [O.e4m3_decode(q) * float(s[0, 0]) for q, s in wq]
    for t in range(2):
        a = [float(av[t, h]) * float(a_s[t, 0]) for h in range(H)]
        m = []
        for i in range(I):
            p = math.fsum(a[h] * wv[0][i, h] for h in range(H))
            q = math.fsum(a[h] * wv[1][i, h] for h in range(H))
            m.append(float(F32(p / (1 + math.exp(-p)) * q)))
        amax = max(abs(v) for v in m)
        sc = float(F32(F32(amax) / F32(448.0)))
        assert m_s[t, 0] == F32(sc)
        mv = O.e4m3_decode(O.e4m3_encode(
            (np.array(m, F32) / F32(sc)).astype(F32))) * sc
        for j in range(0, H, 17):
            yj = math.fsum(mv[i] * wv[2][j, i] for i in range(I))
            assert y[t, j] == pytest.approx(yj, rel=1e-12, abs=1e-15)


def test_fp8_ffn_close_to_full_precision_ffn():
    """On Gaussian data the FP8 expert stays within 10% (RMS) of the fp64
    SwiGLU expert: a 3-bit mantissa rounds each operand with about
    2^-4/sqrt(3) = 3.6% relative RMS error, and x, W1/W3, m and W2 are
    rounded in series (measured here: 6.4%); and it is not exact."""
    rng = np.random.default_rng(5)
    H, I = 256, 384
    x = rng.standard_normal((16, H)).astype(F32)
    w1, w3 = [(rng.standard_normal((I, H)) * 0.05).astype(F32)
              for _ in range(2)]
    w2 = (rng.standard_normal((H, I)) * 0.05).astype(F32)
    y, _ = O.fp8_swiglu_ffn(*O.quantize_1x128(x), O.quantize_128x128(w1),
                            O.quantize_128x128(w3), O.quantize_128x128(w2))
    ref = O.swiglu_ffn(x, w1, w3, w2)
    rel = np.sqrt(np.mean((y - ref) ** 2) / np.mean(ref ** 2))
    assert 1e-2 < rel < 1e-1
