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
