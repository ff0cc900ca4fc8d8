"""Routing backward on the GPU against the oracle: the gates' and the
sequence-wise balance loss's gradients to the router logits (the top-K
choices and indicator counts carry no gradient; the bias takes no part).

Both sides start from the same fp32 sigmoid values, the oracle continuing
in fp64.  The bounds follow the kernels' fixed fp32 order (u = 2^-24,
doubled for margin), per element:
  gates:   c = s(1-s)/D (dg - dot): D a 5-level butterfly of positive
           terms, dot a 5-level butterfly of dg_k g_k ->
           |dc| <= 2 [P (14u A + u(|dg| + |dot|)) + 10u |c|]
           with P = s(1-s)/D, A = sum_k |dg_k g_k|
  balance: g = pre s(1-s)/S (f - dot): S and dot from EPL lane-local terms
           plus a 5-level butterfly ->
           |dg| <= 2 [Q (3u f + (2 EPL + 15) u dot) + 12u |g|]
           with Q = |pre| s(1-s)/S
plus u |result| when accumulating."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def _logits(cfg, T, seed):
    g = np.random.default_rng(seed)
    z = (g.standard_normal((T, cfg.E)) * 1.5).astype(np.float32)
    z[g.random((T, cfg.E)) < 0.01] *= 12            # some saturated
    return z


def _cfg(E, K, G=None):
    G = G or min(8, E // 2)
    return inputs.custom_config("bwd", 600 + E + K, T=1, H=64, E=E,
                                n_group=G, topk_group=G, topk=K, I=64,
                                I_shared=64)


def _route_bound(z, idx, dg):
    s = O.sig32(z).astype(np.float64)
    sk = np.take_along_axis(s, idx, axis=1)
    D = sk.sum(1, keepdims=True)
    gk = sk / D
    dot = (dg * gk).sum(1, keepdims=True)
    A = np.abs(dg * gk).sum(1, keepdims=True)
    P = sk * (1 - sk) / D
    c = P * (dg - dot)
    b = 2 * (P * (14 * U * A + U * (np.abs(dg) + np.abs(dot))) +
             10 * U * np.abs(c))
    out = np.zeros_like(s)
    np.put_along_axis(out, idx, b, axis=1)
    return out


@pytest.mark.parametrize("E,K,T", [(256, 8, 4096), (16, 4, 300),
                                   (1024, 8, 200), (32, 32, 100),
                                   (64, 6, 777)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_route_backward(E, K, T, accumulate):
    cfg = _cfg(E, K)
    d = ops.dims_of(cfg, T=T)
    z = _logits(cfg, T, E + K)
    idx = O.route(z, np.zeros(E, np.float32), cfg.n_group, cfg.topk_group,
                  K)["idx"]
    dg = np.random.default_rng(7).standard_normal((T, K)).astype(np.float32)
    prev = np.random.default_rng(8).standard_normal((T, E)).astype(
        np.float32)
    out = dev(prev) if accumulate else torch.full(
        (T, E), 7.0, dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_ROUTE)
    ops.moe_route_backward(d, dev(z), dev(idx), dev(dg), out, ws,
                           accumulate=accumulate)
    assert ops.moe_get_device_error(ws) == 0
    ref = O.route_backward(z, idx, dg.astype(np.float64))
    bound = _route_bound(z, idx, dg.astype(np.float64))
    if accumulate:
        ref = ref + prev
        bound = bound + U * np.abs(ref)
    got = host(out).astype(np.float64)
    over = np.abs(got - ref) > bound
    assert not over.any(), (int(over.sum()), np.abs(got - ref)[over][:4],
                            bound[over][:4])


def test_route_backward_bad_index_is_reported_and_skipped():
    cfg = _cfg(16, 4)
    T = 64
    d = ops.dims_of(cfg, T=T)
    z = _logits(cfg, T, 3)
    idx = O.route(z, np.zeros(16, np.float32), cfg.n_group, cfg.topk_group,
                  4)["idx"]
    # a non-uniform upstream gradient: with equal dgate the exact gradient
    # is identically zero (sum_k g_k = 1) and only rounding would remain
    dg = np.random.default_rng(4).standard_normal((T, 4)).astype(np.float32)
    bad = idx.copy()
    bad[9, 2] = 99
    out = torch.zeros((T, 16), dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_ROUTE)
    ops.moe_route_backward(d, dev(z), dev(bad), dev(dg), out, ws)
    assert ops.moe_get_device_error(ws) == ops.STATUS_CODES[
        "MOE_ERR_DEVICE_BOUNDS"]
    got = host(out).astype(np.float64)
    dg64 = dg.astype(np.float64)
    ref = O.route_backward(z, idx, dg64)
    bound = _route_bound(z, idx, dg64)
    ok = np.ones(T, bool)
    ok[9] = False
    assert np.all(np.abs(got[ok] - ref[ok]) <= bound[ok])
    # the bad slot is skipped: row 9 is finite and zero off its 3 valid
    # experts (their D then omits the skipped slot)
    valid = [e for e in bad[9].tolist() if 0 <= e < 16]
    assert len(valid) == 3 and np.all(np.isfinite(got[9]))
    assert np.all(np.delete(got[9], valid) == 0)


def _balance_bound(z, seq_len, K, alpha, dloss, E):
    fw = O.seq_balance_loss(z, seq_len, K, alpha)
    s = O.sig32(z).astype(np.float64)
    S = s.sum(1, keepdims=True)
    T = z.shape[0]
    epl = max(1, E // 32)
    b = np.zeros((T, E))
    for q in range(fw["loss"].shape[0]):
        a, e = q * seq_len, min(T, (q + 1) * seq_len)
        f = fw["f"][q]
        sp = s[a:e] / S[a:e]
        dot = (sp @ f)[:, None]
        Q = abs(dloss[q]) * alpha / (e - a) * s[a:e] * (1 - s[a:e]) / S[a:e]
        g = Q * (f[None, :] - dot)
        b[a:e] = 2 * (Q * (3 * U * f[None, :] + (2 * epl + 15) * U * dot) +
                      12 * U * np.abs(g))
    return fw, b


@pytest.mark.parametrize("E,K,T,S", [(256, 8, 4096, 4096), (256, 8, 4096, 1000),
                                     (16, 4, 300, 64), (1024, 8, 200, 77),
                                     (64, 6, 500, 1)])
@pytest.mark.parametrize("accumulate", [False, True])
def test_seq_balance_loss_backward(E, K, T, S, accumulate):
    cfg = _cfg(E, K)
    d = ops.dims_of(cfg, T=T)
    z = _logits(cfg, T, 11 + E)
    alpha = 1e-4
    n_seq = -(-T // S)
    dloss = np.random.default_rng(5).standard_normal(n_seq).astype(
        np.float32)
    fw, bound = _balance_bound(z, S, K, alpha, dloss.astype(np.float64), E)
    prev = np.random.default_rng(6).standard_normal((T, E)).astype(
        np.float32) * 1e-6
    out = dev(prev) if accumulate else torch.full(
        (T, E), 7.0, dtype=torch.float32, device="cuda")
    ops.moe_seq_balance_loss_backward(d, dev(z), S, alpha,
                                      dev(fw["counts"]), out,
                                      dloss=dev(dloss), accumulate=accumulate)
    torch.cuda.synchronize()
    ref = O.seq_balance_loss_backward(z, S, K, alpha,
                                      dloss.astype(np.float64))
    if accumulate:
        ref = ref + prev
        bound = bound + U * np.abs(ref)
    got = host(out).astype(np.float64)
    over = np.abs(got - ref) > bound
    assert not over.any(), (int(over.sum()), np.abs(got - ref)[over][:4],
                            bound[over][:4])


def test_seq_balance_loss_backward_default_upstream_is_one():
    cfg = _cfg(256, 8)
    T = 512
    d = ops.dims_of(cfg, T=T)
    z = _logits(cfg, T, 2)
    fw = O.seq_balance_loss(z, 256, 8)
    out = torch.empty((T, 256), dtype=torch.float32, device="cuda")
    ops.moe_seq_balance_loss_backward(d, dev(z), 256, 1e-4,
                                      dev(fw["counts"]), out)
    torch.cuda.synchronize()
    ref = O.seq_balance_loss_backward(z, 256, 8)
    np.testing.assert_allclose(host(out), ref, rtol=1e-4,
                               atol=1e-6 * np.abs(ref).max())


@pytest.mark.parametrize("E,K,T,S", [(256, 8, 4096, 1000), (16, 4, 300, 64),
                                     (1024, 8, 200, 77), (32, 32, 100, 100),
                                     (64, 6, 777, 1)])
@pytest.mark.parametrize("accumulate", [False, True])
@pytest.mark.parametrize("with_dloss", [False, True])
def test_route_balance_backward_equals_the_two_calls(E, K, T, S, accumulate,
                                                     with_dloss):
    """moe_route_balance_backward gives moe_route_backward followed by
    moe_seq_balance_loss_backward (accumulate set) bit for bit, and both
    gradients' sum within the two bounds of the oracle's."""
    cfg = _cfg(E, K)
    d = ops.dims_of(cfg, T=T)
    z = _logits(cfg, T, 31 + E + K)
    idx = O.route(z, np.zeros(E, np.float32), cfg.n_group, cfg.topk_group,
                  K)["idx"]
    dg = np.random.default_rng(9).standard_normal((T, K)).astype(np.float32)
    alpha = 1e-4
    n_seq = -(-T // S)
    dloss = (np.random.default_rng(10).standard_normal(n_seq).astype(
        np.float32) if with_dloss else None)
    dl64 = (dloss.astype(np.float64) if with_dloss else np.ones(n_seq))
    fw, bbound = _balance_bound(z, S, K, alpha, dl64, E)
    prev = np.random.default_rng(12).standard_normal((T, E)).astype(
        np.float32) * 1e-6
    ws = ops.workspace(d, ops.MOE_WS_ROUTE)
    two = dev(prev) if accumulate else torch.full(
        (T, E), 7.0, dtype=torch.float32, device="cuda")
    ops.moe_route_backward(d, dev(z), dev(idx), dev(dg), two, ws,
                           accumulate=accumulate)
    ops.moe_seq_balance_loss_backward(
        d, dev(z), S, alpha, dev(fw["counts"]), two,
        dloss=dev(dloss) if with_dloss else None, accumulate=True)
    one = dev(prev) if accumulate else torch.full(
        (T, E), 7.0, dtype=torch.float32, device="cuda")
    ops.moe_route_balance_backward(
        d, dev(z), dev(idx), dev(dg), S, alpha, dev(fw["counts"]), one, ws,
        dloss=dev(dloss) if with_dloss else None, accumulate=accumulate)
    assert ops.moe_get_device_error(ws) == 0
    a, b = host(two), host(one)
    assert np.array_equal(a.view(np.uint32), b.view(np.uint32))
    ref = (O.route_backward(z, idx, dg.astype(np.float64)) +
           O.seq_balance_loss_backward(z, S, K, alpha, dl64))
    bound = _route_bound(z, idx, dg.astype(np.float64)) + bbound + \
        U * np.abs(ref)
    if accumulate:
        ref = ref + prev
        bound = bound + U * np.abs(ref)
    over = np.abs(b.astype(np.float64) - ref) > bound
    assert not over.any(), (int(over.sum()), np.abs(b - ref)[over][:4],
                            bound[over][:4])


def test_route_balance_backward_bad_index_is_reported_and_skipped():
    cfg = _cfg(16, 4)
    T, S = 64, 32
    d = ops.dims_of(cfg, T=T)
    z = _logits(cfg, T, 5)
    idx = O.route(z, np.zeros(16, np.float32), cfg.n_group, cfg.topk_group,
                  4)["idx"]
    dg = np.random.default_rng(4).standard_normal((T, 4)).astype(np.float32)
    bad = idx.copy()
    bad[9, 2] = 99
    fw = O.seq_balance_loss(z, S, 4, 1e-4)
    ws = ops.workspace(d, ops.MOE_WS_ROUTE)
    two = torch.zeros((T, 16), dtype=torch.float32, device="cuda")
    ops.moe_route_backward(d, dev(z), dev(bad), dev(dg), two, ws)
    ops.moe_seq_balance_loss_backward(d, dev(z), S, 1e-4, dev(fw["counts"]),
                                      two, accumulate=True)
    ws2 = ops.workspace(d, ops.MOE_WS_ROUTE)
    one = torch.zeros((T, 16), dtype=torch.float32, device="cuda")
    ops.moe_route_balance_backward(d, dev(z), dev(bad), dev(dg), S, 1e-4,
                                   dev(fw["counts"]), one, ws2)
    for w in (ws, ws2):
        assert ops.moe_get_device_error(w) == ops.STATUS_CODES[
            "MOE_ERR_DEVICE_BOUNDS"]
    assert np.array_equal(host(two).view(np.uint32), host(one).view(np.uint32))
