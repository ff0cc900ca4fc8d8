"""Pins for the oracle's routing backward (no GPU): the analytic gradients
against central finite differences of an fp64 restatement of the forward
(sigmoid from math, the top-K choice and the balance loss's indicator held
fixed, as they are piecewise constant), plus closed-form special cases."""
import numpy as np
import pytest
from scipy.special import expit

from oracle import moe_oracle as O

F32 = np.float32


def _gates64(z, idx):
    s = expit(z)
    sk = np.take_along_axis(s, idx, axis=1)
    return sk / sk.sum(axis=1, keepdims=True)


def test_route_backward_matches_finite_differences():
    g = np.random.default_rng(1)
    T, E, K = 5, 16, 4
    z = g.normal(0, 1, (T, E)).astype(F32)
    idx = np.argsort(-z, axis=1)[:, :K].astype(np.int32)
    dg = g.normal(0, 1, (T, K))
    grad = O.route_backward(z, idx, dg)
    z64 = z.astype(np.float64)
    h = 1e-6
    num = np.zeros((T, E))
    for t in range(T):
        for e in range(E):
            zp, zm = z64.copy(), z64.copy()
            zp[t, e] += h
            zm[t, e] -= h
            num[t, e] = ((_gates64(zp, idx) - _gates64(zm, idx))[t] *
                         dg[t]).sum() / (2 * h)
    np.testing.assert_allclose(grad, num, rtol=1e-5, atol=1e-8)
    chosen = np.zeros((T, E), bool)
    np.put_along_axis(chosen, idx, True, axis=1)
    assert np.all(grad[~chosen] == 0)


def test_route_backward_uniform_upstream_gives_zero():
    """sum_k g_k = 1, so an upstream gradient equal on every gate moves
    nothing: dgate_m - sum_k dgate_k g_k = 0."""
    z = np.random.default_rng(2).normal(0, 1, (3, 32)).astype(F32)
    idx = np.argsort(-z, axis=1)[:, :8].astype(np.int32)
    grad = O.route_backward(z, idx, np.full((3, 8), 2.5))
    assert np.abs(grad).max() < 1e-15


def _balance64(z, seq_len, topk, alpha, counts):
    """L per sequence with the counts (indicator) held fixed."""
    T, E = z.shape
    s = expit(z)
    sp = s / s.sum(axis=1, keepdims=True)
    out = []
    for q in range(counts.shape[0]):
        a, b = q * seq_len, min(T, (q + 1) * seq_len)
        f = E * counts[q] / (topk * (b - a))
        out.append(alpha * f @ sp[a:b].mean(axis=0))
    return np.array(out)


def test_balance_backward_matches_finite_differences():
    g = np.random.default_rng(3)
    T, E, K, S = 7, 16, 3, 3
    z = g.normal(0, 1, (T, E)).astype(F32)
    alpha = 0.01
    fw = O.seq_balance_loss(z, S, K, alpha)
    dl = g.normal(0, 1, fw["loss"].shape[0])
    grad = O.seq_balance_loss_backward(z, S, K, alpha, dl)
    z64 = z.astype(np.float64)
    h = 1e-6
    num = np.zeros((T, E))
    for t in range(T):
        for e in range(E):
            zp, zm = z64.copy(), z64.copy()
            zp[t, e] += h
            zm[t, e] -= h
            num[t, e] = ((_balance64(zp, S, K, alpha, fw["counts"]) -
                          _balance64(zm, S, K, alpha, fw["counts"])) @ dl
                         ) / (2 * h)
    np.testing.assert_allclose(grad, num, rtol=1e-5, atol=1e-12)


def test_balance_backward_vanishes_for_uniform_f():
    """f_i = 1 for every expert (an evenly spread selection) makes
    f_i - sum_j f_j s'_j = 1 - 1 = 0: the loss is flat in z there."""
    E, K = 64, 4
    nb = E // K
    T = 2 * nb
    g = np.random.default_rng(4)
    z = g.uniform(-3, -1, (T, E)).astype(F32)
    for t in range(T):
        z[t, (t % nb) * K:(t % nb + 1) * K] = g.uniform(1, 3, K)
    fw = O.seq_balance_loss(z, T, K)
    assert np.all(fw["f"] == 1.0)
    assert np.abs(O.seq_balance_loss_backward(z, T, K)).max() < 1e-18


def test_balance_backward_pushes_hot_experts_down():
    """A token's gradient is positive on experts with f above the
    token's f-weighted mean and negative below it (descent lowers the
    affinity of over-selected experts)."""
    g = np.random.default_rng(5)
    z = g.normal(0, 1, (40, 16)).astype(F32)
    z[:, 2] += 2.0                              # expert 2 over-selected
    fw = O.seq_balance_loss(z, 40, 2)
    grad = O.seq_balance_loss_backward(z, 40, 2)
    s = O.sig32(z).astype(np.float64)
    dot = (s / s.sum(1, keepdims=True)) @ fw["f"][0]
    sign = np.sign(fw["f"][0][None, :] - dot[:, None])
    assert np.all(np.sign(grad) == sign)
    assert np.all(grad[:, 2] > 0)
