"""Shared helpers of the GPU parity tests (device tensors, calls through
the C ABI, tolerance checks)."""
import numpy as np
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O


def dev(a):
    """numpy -> CUDA tensor (uint16 bf16 bits travel as int16)."""
    a = np.ascontiguousarray(a)
    if a.dtype == np.uint16:
        a = a.view(np.int16)
    return torch.from_numpy(a).cuda()


def host(t, dtype=None):
    a = t.cpu().numpy()
    if dtype is not None:
        a = a.view(dtype)
    return a


def bf16_dev_to_f32(t):
    return inputs.bf16_bits_to_f32(host(t, np.uint16))


def f32_bits(a):
    return np.ascontiguousarray(a, np.float32).view(np.uint32)


def route_gpu(d, logits, bias):
    T, E, K = d.T, d.E, d.topk
    idx = torch.full((T, K), -7, dtype=torch.int32, device="cuda")
    gate = torch.full((T, K), -7.0, dtype=torch.float32, device="cuda")
    counts = torch.full((E,), -7, dtype=torch.int32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_ROUTE)
    ops.moe_route(d, dev(logits), dev(bias), idx, gate, counts, ws)
    assert ops.moe_get_device_error(ws) == 0
    return host(idx), host(gate), host(counts)


def assert_route_bit_exact(d, logits, bias):
    r = O.route(logits, bias, d.n_group, d.topk_group, d.topk)
    idx, gate, counts = route_gpu(d, logits, bias)
    bad = np.nonzero(np.any(idx != r["idx"], axis=1))[0]
    assert bad.size == 0, (bad[:5], idx[bad[:2]], r["idx"][bad[:2]])
    assert np.array_equal(f32_bits(gate), f32_bits(r["gate"]))
    assert np.array_equal(counts, O.expert_counts(r["idx"], d.E))
    return r


def rms_tolerance_check(got, ref, rows=None, frac=2e-2):
    """max |got - ref| <= frac * RMS(ref) over the compared rows."""
    g = np.asarray(got, np.float64)
    f = np.asarray(ref, np.float64)
    if rows is not None:
        g, f = g[rows], f[rows]
    rms = np.sqrt(np.mean(f * f))
    err = np.max(np.abs(g - f)) if g.size else 0.0
    assert err <= frac * rms, (err, rms, err / rms)
    return err / rms


U_BF16 = 2.0 ** -8   # unit roundoff of bf16 (8-bit significand)


def ffn_bound_check(got, a, w1, w3, w2):
    """Elementwise bound for one expert FFN whose intermediate h and output
    y are stored in bf16 with fp32 accumulation:
        |y_gpu - y| <= u*|y| + u*sum_i |m_i| |W2_ji|  (+ fp32 slack)
    with u = 2^-8 and m = silu(W1 a) * (W3 a) in fp64 -- the first term is
    the output rounding, the second the rounding of every h_i.  Returns the
    largest error / bound ratio (must be <= 1)."""
    from oracle import moe_oracle as O
    a = np.asarray(a, np.float64)
    p = a @ np.asarray(w1, np.float64).T
    q = a @ np.asarray(w3, np.float64).T
    m = O.silu(p) * q
    w2 = np.asarray(w2, np.float64)
    y = m @ w2.T
    bound = 1.01 * U_BF16 * np.abs(y) + 1.1 * U_BF16 * (np.abs(m) @ np.abs(w2).T)
    bound += 1e-5 * np.sqrt(np.mean(y * y)) + 1e-30
    ratio = np.abs(np.asarray(got, np.float64) - y) / bound
    assert ratio.max() <= 1.0, ratio.max()
    return ratio.max()


_TABLE = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
# spacing of the E4M3 grid around each magnitude code (the wider side)
_STEP = np.maximum(np.diff(_TABLE, append=_TABLE[-1] + 32.0),
                   np.diff(_TABLE, prepend=0.0))


def _flip_bound(m, w2):
    """2 max_i step_i(t) |W2_ji| for the oracle's intermediate m = (codes,
    scales) of each token and the dequantized W2 [H, I]."""
    mq, ms = m
    step = _STEP[mq & 0x7F] * np.repeat(ms.astype(np.float64), 128, axis=1)
    aw = np.abs(w2)
    out = np.empty((mq.shape[0], aw.shape[0]))
    for t in range(mq.shape[0]):
        out[t] = 2.0 * (aw * step[t][None, :]).max(axis=1)
    return out


def fp8_ffn_check(got, ref, what, m=None, w2=None):
    """The FP8 expert bar (see test_gpu_fp8_ffn.py's module docstring):
    |y_gpu - y| <= 2^-8 |y| + 1e-3 RMS(y) + the one-step code flips of the
    intermediate, and RMS error <= 5e-3 RMS(y)."""
    got = np.asarray(got, np.float64)
    rms = np.sqrt(np.mean(ref * ref))
    err = np.abs(got - ref)
    bound = 2.0 ** -8 * np.abs(ref) + 1e-3 * rms
    if m is not None:
        bound = bound + _flip_bound(m, w2)
    # on failure, say how the two relate: a scale slip shows as a clean
    # fit with the wrong factor, a layout slip as low correlation
    g, r = got.ravel(), ref.ravel()
    diag = dict(what=what, max_err=float(err.max() / rms),
                rms_err=float(np.sqrt(np.mean(err * err)) / rms),
                corr=float(np.corrcoef(g, r)[0, 1]) if g.std() > 0 else 0.0,
                fit=float(g @ r / (r @ r)), got_rms=float(np.sqrt(np.mean(
                    g * g)) / rms), finite=bool(np.isfinite(g).all()),
                over=int(np.sum(err > bound)))
    assert np.all(err <= bound), diag
    assert np.sqrt(np.mean(err * err)) <= 5e-3 * rms, diag
