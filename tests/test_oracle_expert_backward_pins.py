"""Pins for the oracle's expert and combine backward (no GPU): central
finite differences of the pinned forward functions (swiglu_ffn, moe_output)
and the chain from the layer output to the router logits through the gates
(combine_backward's dgate into route_backward); and the composed
layer_backward (all token, gate and weight gradients of eq. 12 with fixed
routing) against finite differences, an unchosen expert, and the zero
routed-weights reduction to the dense SwiGLU backward."""
import numpy as np

from oracle import moe_oracle as O

F32 = np.float32


def _fd(f, x, h=1e-6):
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        xp, xm = x.copy(), x.copy()
        xp[i] += h
        xm[i] -= h
        g[i] = (f(xp) - f(xm)) / (2 * h)
    return g


def test_swiglu_backward_matches_finite_differences():
    g = np.random.default_rng(0)
    n, H, I = 3, 6, 5
    a = g.normal(0, 1, (n, H))
    w1, w3 = g.normal(0, 0.5, (I, H)), g.normal(0, 0.5, (I, H))
    w2 = g.normal(0, 0.5, (H, I))
    dy = g.normal(0, 1, (n, H))
    da, dw1, dw3, dw2 = O.swiglu_ffn_backward(a, w1, w3, w2, dy)
    L = lambda A, W1, W3, W2: float((O.swiglu_ffn(A, W1, W3, W2) * dy).sum())  # noqa: E731
    np.testing.assert_allclose(da, _fd(lambda v: L(v, w1, w3, w2), a),
                               rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(dw1, _fd(lambda v: L(a, v, w3, w2), w1),
                               rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(dw3, _fd(lambda v: L(a, w1, v, w2), w3),
                               rtol=1e-6, atol=1e-9)
    np.testing.assert_allclose(dw2, _fd(lambda v: L(a, w1, w3, v), w2),
                               rtol=1e-6, atol=1e-9)


def test_swiglu_backward_linear_in_dy_and_zero_for_zero_weights():
    g = np.random.default_rng(1)
    a = g.normal(0, 1, (2, 4))
    w1, w3, w2 = (g.normal(0, 1, s) for s in ((3, 4), (3, 4), (4, 3)))
    d1, d2 = g.normal(0, 1, (2, 4)), g.normal(0, 1, (2, 4))
    r1 = O.swiglu_ffn_backward(a, w1, w3, w2, d1)
    r2 = O.swiglu_ffn_backward(a, w1, w3, w2, d2)
    r12 = O.swiglu_ffn_backward(a, w1, w3, w2, d1 + 2 * d2)
    for x, y, z in zip(r1, r2, r12):
        np.testing.assert_allclose(z, x + 2 * y, rtol=1e-12, atol=1e-12)
    # W3 = 0: m = 0, so dW2 = 0 and dW1 = 0 (dp carries the factor q = 0)
    da, dw1, dw3, dw2 = O.swiglu_ffn_backward(a, w1, 0 * w3, w2, d1)
    assert np.all(dw2 == 0) and np.all(dw1 == 0)


def test_combine_backward_matches_finite_differences():
    g = np.random.default_rng(2)
    T, K, H = 3, 2, 4
    x, ys = g.normal(0, 1, (T, H)), g.normal(0, 1, (T, H))
    y = g.normal(0, 1, (T, K, H))
    gate = g.uniform(0.1, 1, (T, K))
    dout = g.normal(0, 1, (T, H))
    dx, dys, dy, dg = O.combine_backward(dout, y, gate)
    L = lambda X, YS, Y, G: float((O.moe_output(X, YS, Y, G) * dout).sum())  # noqa: E731
    np.testing.assert_allclose(dx, _fd(lambda v: L(v, ys, y, gate), x),
                               rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(dys, _fd(lambda v: L(x, v, y, gate), ys),
                               rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(dy, _fd(lambda v: L(x, ys, v, gate), y),
                               rtol=1e-7, atol=1e-9)
    np.testing.assert_allclose(dg, _fd(lambda v: L(x, ys, y, v), gate),
                               rtol=1e-7, atol=1e-9)


def test_output_to_logits_chain_through_the_gates():
    """d(loss)/dz along the gate path: combine_backward's dgate fed to
    route_backward equals finite differences of the output in z, with the
    expert outputs and the top-K choice held fixed (gates from scipy's
    sigmoid of z, the forward's definition)."""
    from scipy.special import expit
    g = np.random.default_rng(3)
    T, E, K, H = 2, 8, 3, 5
    z = g.normal(0, 1, (T, E)).astype(F32)
    idx = np.argsort(-z, axis=1)[:, :K].astype(np.int32)
    y = g.normal(0, 1, (T, K, H))
    x, ys = np.zeros((T, H)), np.zeros((T, H))
    dout = g.normal(0, 1, (T, H))

    def out_of(zz):
        s = np.take_along_axis(expit(zz), idx, axis=1)
        return float((O.moe_output(x, ys, y, s / s.sum(1, keepdims=True))
                      * dout).sum())
    dg = O.combine_backward(dout, y, np.ones((T, K)))[3]
    grad = O.route_backward(z, idx, dg)
    num = _fd(out_of, z.astype(np.float64))
    np.testing.assert_allclose(grad, num, rtol=1e-5, atol=1e-8)


def _tiny_layer(seed, T=5, H=6, E=4, I=3, Is=4, K=2):
    g = np.random.default_rng(seed)
    x = g.normal(0, 1, (T, H))
    w1, w3 = g.normal(0, 0.5, (E, I, H)), g.normal(0, 0.5, (E, I, H))
    w2 = g.normal(0, 0.5, (E, H, I))
    ws1, ws3 = g.normal(0, 0.5, (Is, H)), g.normal(0, 0.5, (Is, H))
    ws2 = g.normal(0, 0.5, (H, Is))
    idx = np.stack([g.choice(E, K, replace=False) for _ in range(T)])
    gate = g.uniform(0.1, 1.0, (T, K))
    dout = g.normal(0, 1, (T, H))
    return x, dout, idx, gate, [w1, w3, w2, ws1, ws3, ws2]


def _out_fixed_routing(x, idx, gate, w):
    """eq. 12 with the routing and the gates held fixed, straight from the
    forward pieces (moe_output of the per-slot swiglu_ffn values)."""
    w1, w3, w2, ws1, ws3, ws2 = w
    T, K = idx.shape
    ys = O.swiglu_ffn(x, ws1, ws3, ws2)
    y = np.zeros((T, K, x.shape[1]))
    for t in range(T):
        for k in range(K):
            e = idx[t, k]
            y[t, k] = O.swiglu_ffn(x[t:t + 1], w1[e], w3[e], w2[e])[0]
    return O.moe_output(x, ys, y, gate)


def test_layer_backward_matches_finite_differences():
    """Every gradient of layer_backward against central differences of
    <dout, out> with the routing and gates fixed: the token gradient (the
    residual, shared and routed terms together), the routed experts' and
    the shared expert's three weight gradients, and the gates."""
    x, dout, idx, gate, w = _tiny_layer(4)
    r = O.layer_backward(x, dout, idx, gate, *w)
    L = lambda X, G, W: float((_out_fixed_routing(X, idx, G, W) * dout).sum())  # noqa: E731
    np.testing.assert_allclose(r["dx"], _fd(lambda v: L(v, gate, w), x),
                               rtol=1e-6, atol=1e-8)
    np.testing.assert_allclose(r["dgate"], _fd(lambda v: L(x, v, w), gate),
                               rtol=1e-6, atol=1e-8)
    names = ["dw1", "dw3", "dw2", "dws1", "dws3", "dws2"]
    for i, n in enumerate(names):
        def Lw(v, i=i):
            ww = list(w)
            ww[i] = v
            return L(x, gate, ww)
        np.testing.assert_allclose(r[n], _fd(Lw, w[i]), rtol=1e-6,
                                   atol=1e-8, err_msg=n)


def test_layer_backward_unchosen_expert_has_zero_gradient():
    x, dout, idx, gate, w = _tiny_layer(5)
    idx = np.array([[0, 1], [1, 2], [2, 0], [0, 2], [1, 0]])   # never 3
    assert not np.any(idx == 3)
    r = O.layer_backward(x, dout, idx, gate, *w)
    assert np.all(r["dw1"][3] == 0) and np.all(r["dw2"][3] == 0)
    assert np.all(r["dw3"][3] == 0)


def test_layer_backward_zero_routed_weights_is_dense_swiglu_backward():
    """Routed experts all zero: dx = dout + the dense shared-expert token
    gradient, and the gates' gradient is 0 (every routed output is 0)."""
    x, dout, idx, gate, w = _tiny_layer(6)
    w = [0 * w[0], 0 * w[1], 0 * w[2]] + w[3:]
    r = O.layer_backward(x, dout, idx, gate, *w)
    da = O.swiglu_ffn_backward(x, w[3], w[4], w[5], dout)[0]
    np.testing.assert_allclose(r["dx"], dout + da, rtol=1e-12, atol=1e-12)
    assert np.all(r["dgate"] == 0)
