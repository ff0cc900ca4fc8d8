"""The experts' backward (moe_expert_backward: recompute, dgrad and wgrad
GEMMs on the tensor cores) against the oracle's fp64 ``layer_backward``
("02 · DeepSeek-V3" §1.1 SwiGLU experts, eq. 12 combine, fixed routing).

Tolerance, per element, derived from where the GPU rounds (u = 2^-8 for a
bf16 store, v = 2^-24 for fp32 arithmetic, n the length of a sum):
* p, q, D = W2^T dout: fp32 sums of exact bf16 products, error
  e_p <= n v sum |a w| (likewise e_q, e_D);
* dq = dm silu(p), dp = dm q silu'(p) with dm = g D, stored as bf16:
  e_dq = u|dq| + |g silu(p)| e_D + |dm silu'(p)| e_p,
  e_dp = u|dp| + |g q silu'(p)| e_D + |dm silu'(p)| e_q + |dm q silu''(p)| e_p
         + 8v |dm q| (1 + |p|)  (silu'(p) cancels near its root);
* dW1 = sum_r dp a^T: sum_r e_dp |a| + n v sum_r |dp a| (dW3 with dq);
  dW2 = sum_r dout (g m)^T with g m stored as bf16:
  sum_r |dout| (u |g m| + |g| e_m) + n v sum_r |dout| |g m|;
* dx: each routed / shared row's W1 dp + W3 dq is stored as bf16, then
  dout + shared + routed rows are summed in fp32 and stored as bf16:
  u |dx| + sum over the rows of (u |row| + sum_i (e_dp |W1| + e_dq |W3|)
  + n v sum_i (|dp W1| + |dq W3|)) + (K + 2) v sum |terms|;
* dgate = <D, h> in fp32: n v sum_i (|D| |h| + |D| e_h + e_D |h|).
Every bound is an upper bound of the first-order error terms; the tests also
require the worst ratio to be a visible fraction of it (the bound is not
vacuous) on the full comparisons."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import bf16_dev_to_f32, dev, host

pytestmark = pytest.mark.gpu

f32 = inputs.bf16_bits_to_f32
U = 2.0 ** -8
V = 2.0 ** -24


def _silu_parts(p):
    sg = 1.0 / (1.0 + np.exp(-np.clip(p, -700, 700)))
    d1 = sg * (1.0 + p * (1.0 - sg))
    d2 = sg * (1.0 - sg) * (2.0 + p * (1.0 - 2.0 * sg))
    return sg, p * sg, d1, d2


def expert_terms(a, dy, g, w1, w3, w2):
    """fp64 intermediates of one expert's backward on rows a [n, H] with
    upstream rows dy = g * dout [n, H] and gates g [n], plus the error
    allowances of the module docstring.  Returns a dict."""
    a = np.asarray(a, np.float64)
    w1, w3, w2 = (np.asarray(w, np.float64) for w in (w1, w3, w2))
    dy = np.asarray(dy, np.float64)
    g = np.asarray(g, np.float64)[:, None]
    H = a.shape[1]
    aa = np.abs(a)
    p, q = a @ w1.T, a @ w3.T
    e_p = H * V * (aa @ np.abs(w1).T)
    e_q = H * V * (aa @ np.abs(w3).T)
    sg, sl, d1, d2 = _silu_parts(p)
    m = sl * q
    dout = np.where(g != 0, dy / np.where(g != 0, g, 1.0), 0.0)
    D = dout @ w2                                   # W2^T dout per row
    e_D = H * V * (np.abs(dout) @ np.abs(w2))
    dm = g * D
    dq = dm * sl
    dp = dm * q * d1
    e_dq = U * np.abs(dq) + np.abs(g * sl) * e_D + np.abs(dm * d1) * e_p
    e_dp = (U * np.abs(dp) + np.abs(g * q * d1) * e_D + np.abs(dm * d1) * e_q
            + np.abs(dm * q * d2) * e_p + 8 * V * np.abs(dm * q) * (1 + np.abs(p)))
    e_m = np.abs(d1 * q) * e_p + np.abs(sl) * e_q
    return dict(p=p, q=q, m=m, D=D, dm=dm, dp=dp, dq=dq, e_dp=e_dp,
                e_dq=e_dq, e_m=e_m, e_D=e_D, dout=dout, g=g)


def wgrad_bounds(tm, a, n_rows):
    """Bounds of dW1, dW3, dW2 for one expert from expert_terms()."""
    aa = np.abs(np.asarray(a, np.float64))
    n = max(1, n_rows)
    b1 = tm["e_dp"].T @ aa + n * V * (np.abs(tm["dp"]).T @ aa)
    b3 = tm["e_dq"].T @ aa + n * V * (np.abs(tm["dq"]).T @ aa)
    # the GPU multiplies the ungated dout rows by the stored g m rows
    do = np.abs(tm["dout"])
    gm = np.abs(tm["g"] * tm["m"])
    b2 = do.T @ (U * gm + np.abs(tm["g"]) * tm["e_m"]) + n * V * (do.T @ gm)
    return b1, b3, b2


def row_grad_terms(tm, w1, w3):
    """A routed row's input gradient W1^T dp + W3^T dq, its stored (bf16)
    error allowance, and the absolute sum of its terms."""
    w1, w3 = np.asarray(w1, np.float64), np.asarray(w3, np.float64)
    I = w1.shape[0]
    val = tm["dp"] @ w1 + tm["dq"] @ w3
    absum = np.abs(tm["dp"]) @ np.abs(w1) + np.abs(tm["dq"]) @ np.abs(w3)
    err = (U * np.abs(val) + tm["e_dp"] @ np.abs(w1) + tm["e_dq"] @ np.abs(w3)
           + I * V * absum)
    return val, err


def check(got, ref, bound, what, min_ratio=0.0):
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all(), what
    ratio = np.abs(got - ref) / (bound + 1e-30)
    worst = float(ratio.max()) if ratio.size else 0.0
    assert worst <= 1.0, (what, worst, np.unravel_index(np.argmax(ratio),
                                                        ratio.shape))
    assert worst >= min_ratio, (what, worst)
    return worst


def run_backward(d, W, x, dout, idx, gate, accumulate=False, grads=None):
    T, K, H = d.T, d.topk, d.H
    dx = torch.full((T, H), 0x7FC0, dtype=torch.int16, device="cuda")
    dg = torch.full((T, K), float("nan"), dtype=torch.float32, device="cuda")
    if grads is None:
        grads = ops.WeightGrads.empty(d)
        for t in grads.tensors():
            t.fill_(float("nan"))
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_BWD)
    ops.moe_expert_backward(d, W, x, dout, idx, gate, dx, dg, grads, ws,
                            accumulate=accumulate)
    assert ops.moe_get_device_error(ws) == 0
    return dx, dg, grads


def _dout(cfg, T, sigma=1.0):
    key = (cfg.config_id * 104729 + 77) & 0xFFFFFFFF
    return inputs.normal_bf16(key, (T, cfg.H), sigma)


def _small_case(cfg, idx=None):
    """Full comparison on a small layer: every element of dx, dgate and all
    six weight gradients."""
    d = ops.dims_of(cfg)
    T, K, E = cfg.T, cfg.topk, cfg.E
    w = inputs.layer_inputs(cfg)
    xf = f32(w["x"])
    if idx is None:
        z = O.router_logits(xf, w["w_router"])
        r = O.route(z, w["bias"], cfg.n_group, cfg.topk_group, K)
        idx, gate = r["idx"], r["gate"]
    else:
        rng = np.random.default_rng(cfg.config_id)
        gate = rng.uniform(0.05, 0.6, idx.shape).astype(np.float32)
    dout = _dout(cfg, T)
    W = ops.Weights(torch.zeros(E, cfg.H, dtype=torch.float32, device="cuda"),
                    dev(w["w1"]), dev(w["w3"]), dev(w["w2"]), dev(w["ws1"]),
                    dev(w["ws3"]), dev(w["ws2"]))
    dx, dg, grads = run_backward(d, W, dev(w["x"]), dev(dout), dev(idx),
                                 dev(gate))
    F = {n: f32(w[n]) for n in ("w1", "w3", "w2", "ws1", "ws3", "ws2")}
    ref = O.layer_backward(xf, f32(dout), idx, gate, F["w1"], F["w3"],
                           F["w2"], F["ws1"], F["ws3"], F["ws2"])
    do = f32(dout).astype(np.float64)
    # shared expert: every token, g = 1
    ts = expert_terms(xf, do, np.ones(T), F["ws1"], F["ws3"], F["ws2"])
    bs1, bs3, bs2 = wgrad_bounds(ts, xf, T)
    sv, se = row_grad_terms(ts, F["ws1"], F["ws3"])
    dx_err = se.copy()
    dx_abs = np.abs(do) + np.abs(sv)
    gw = {n: host(getattr(grads, n)) for n in ops.WeightGrads.NAMES}
    worst = []
    dg_h = host(dg)
    for e in range(E):
        t, k = np.nonzero(idx == e)
        if t.size == 0:
            for n in ("dw1", "dw3", "dw2"):
                assert np.all(gw[n][e] == 0), (n, e)
            continue
        gk = gate[t, k].astype(np.float64)
        tm = expert_terms(xf[t], gk[:, None] * do[t], gk, F["w1"][e],
                          F["w3"][e], F["w2"][e])
        b1, b3, b2 = wgrad_bounds(tm, xf[t], t.size)
        worst.append(check(gw["dw1"][e], ref["dw1"][e], b1, f"dw1[{e}]"))
        worst.append(check(gw["dw3"][e], ref["dw3"][e], b3, f"dw3[{e}]"))
        worst.append(check(gw["dw2"][e], ref["dw2"][e], b2, f"dw2[{e}]"))
        rv, re_ = row_grad_terms(tm, F["w1"][e], F["w3"][e])
        dx_err[t] += re_
        dx_abs[t] += np.abs(rv)
        h = tm["m"]
        bnd = (F["w2"].shape[2]) * V * (np.abs(tm["D"]) * np.abs(h)).sum(1) \
            + (np.abs(tm["D"]) * tm["e_m"] + tm["e_D"] * np.abs(h)).sum(1)
        worst.append(check(dg_h[t, k], ref["dgate"][t, k], bnd + 1e-30,
                           f"dgate[{e}]"))
    worst.append(check(gw["dws1"], ref["dws1"], bs1, "dws1"))
    worst.append(check(gw["dws3"], ref["dws3"], bs3, "dws3"))
    worst.append(check(gw["dws2"], ref["dws2"], bs2, "dws2"))
    dx_bound = U * (np.abs(ref["dx"]) + dx_err) + dx_err + \
        (K + 2) * V * dx_abs
    worst.append(check(bf16_dev_to_f32(dx), ref["dx"], dx_bound, "dx"))
    # the bounds are not vacuous: some element uses a visible part of one
    assert max(worst) > 0.02, worst
    return d, W, (dev(w["x"]), dev(dout), dev(idx), dev(gate)), grads


def test_backward_tiny_config():
    _small_case(inputs.CONFIGS["tiny"])


def test_backward_ragged_features_and_rows():
    """I = 192 (a 256-feature block with 64 valid features in the dgrad
    of the down projection, a partial 128-row block of dW1 / dW3), I_s =
    128, H = 320 (a partial 256-column block of dW1 / dW3), T = 77 (the
    shared expert's reduction ends inside a 16-row step)."""
    cfg = inputs.custom_config("bwd_r", 800, T=77, H=320, E=8, n_group=4,
                               topk_group=2, topk=2, I=192, I_shared=128,
                               router_sigma=0.05)
    _small_case(cfg)


def test_backward_unused_expert_single_row_expert_and_full_segments():
    """Expert 5 gets no rows (zero gradient), expert 2 exactly one row,
    expert 0 exactly 16 (no padding), expert 1 a long segment of several
    64-row reduction blocks."""
    cfg = inputs.custom_config("bwd_u", 801, T=150, H=256, E=8, n_group=4,
                               topk_group=2, topk=2, I=128, I_shared=64)
    T = cfg.T
    idx = np.zeros((T, 2), np.int32)
    idx[:, 0] = 1
    idx[:, 1] = np.array([3, 4, 6, 7] * 38)[:T]
    idx[:16, 1] = 0
    idx[16, 1] = 2
    _small_case(cfg, idx)


def test_backward_resident_and_streamed_segments_and_row_block_groups():
    """The weight-gradient GEMM keeps a segment's B operand in shared
    memory when the segment has at most 192 rows and streams it otherwise:
    expert 1 gets 210 rows (224 padded: streamed, four reduction blocks),
    expert 3 150 (160: resident, a 32-row tail), expert 0 16, expert 2
    none, the shared expert 260 (streamed, a 4-row tail past which the map
    ends).  H = 2176 gives dW2 17 row blocks (a group of 16 and one more)
    and dW1 / dW3 a partial 256-column block."""
    cfg = inputs.custom_config("bwd_g", 803, T=260, H=2176, E=8, n_group=4,
                               topk_group=2, topk=2, I=128, I_shared=64)
    T = cfg.T
    idx = np.zeros((T, 2), np.int32)
    idx[:210, 0] = 1
    idx[210:, 0] = 3
    idx[:100, 1] = 3
    idx[100:116, 1] = 0
    idx[116:, 1] = np.array([4, 5, 6, 7] * 36)
    counts = np.bincount(idx.ravel(), minlength=8)
    assert counts.tolist() == [16, 210, 0, 150, 36, 36, 36, 36]
    _small_case(cfg, idx)


def test_backward_largest_hidden_size():
    """H = 16384 (the backward's limit): the token gather and the finalize
    at their widest rows, dW1 / dW3 with 64 256-column blocks, dW2 with 128
    row blocks (groups of 16)."""
    cfg = inputs.custom_config("bwd_h16k", 806, T=40, H=16384, E=8,
                               n_group=4, topk_group=2, topk=2, I=128,
                               I_shared=64, router_sigma=0.01)
    _small_case(cfg)


def test_backward_1024_experts_mostly_empty():
    """E = 1024 (the largest expert count): ~2 rows per chosen expert and
    most experts without a token, so the weight-gradient GEMM's task table
    has 3 x 1025 (matrix, segment) pairs and most of its tasks zero-fill a
    whole group of row blocks."""
    cfg = inputs.custom_config("bwd_e1k", 805, T=300, H=256, E=1024,
                               n_group=8, topk_group=4, topk=8, I=128,
                               I_shared=64, router_sigma=0.05)
    _small_case(cfg)


def test_backward_repeats_bit_exactly_on_one_workspace():
    """Calls on one workspace give the same results bit for bit: the
    weight-gradient GEMM's task counter lives in the workspace and every
    call resets it, also when the call is replayed from a CUDA graph (no
    host step between the replays)."""
    import torch
    cfg = inputs.custom_config("bwd_rep", 804, T=96, H=256, E=8, n_group=4,
                               topk_group=2, topk=2, I=128, I_shared=64,
                               router_sigma=0.05)
    d = ops.dims_of(cfg)
    T, K, E = cfg.T, cfg.topk, cfg.E
    w = inputs.layer_inputs(cfg)
    z = O.router_logits(f32(w["x"]), w["w_router"])
    r = O.route(z, w["bias"], cfg.n_group, cfg.topk_group, K)
    W = ops.Weights(torch.zeros(E, cfg.H, dtype=torch.float32, device="cuda"),
                    dev(w["w1"]), dev(w["w3"]), dev(w["w2"]), dev(w["ws1"]),
                    dev(w["ws3"]), dev(w["ws2"]))
    args = (dev(w["x"]), dev(_dout(cfg, T)), dev(r["idx"]), dev(r["gate"]))
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_BWD)
    outs = []
    for _ in range(3):
        dx = torch.empty((T, cfg.H), dtype=torch.int16, device="cuda")
        dg = torch.empty((T, K), dtype=torch.float32, device="cuda")
        grads = ops.WeightGrads.empty(d)
        for t in grads.tensors():
            t.fill_(float("nan"))
        outs.append((dx, dg, grads))
    for dx, dg, grads in outs[:2]:
        ops.moe_expert_backward(d, W, *args, dx, dg, grads, ws)
    dx, dg, grads = outs[2]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            ops.moe_expert_backward(d, W, *args, dx, dg, grads, ws)
    torch.cuda.current_stream().wait_stream(side)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert ops.moe_get_device_error(ws) == 0
    ref = [host(t) for t in (outs[0][0], outs[0][1], *outs[0][2].tensors())]
    assert all(np.isfinite(a).all() for a in ref[1:])
    for dx_, dg_, gr_ in outs[1:]:
        got = [host(t) for t in (dx_, dg_, *gr_.tensors())]
        for a, b in zip(ref, got):
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))


def test_backward_accumulates_into_the_weight_gradients():
    """accumulate != 0 adds to the arrays: a second call on the same inputs
    doubles every weight gradient exactly (x + x is exact in fp32)."""
    cfg = inputs.custom_config("bwd_acc", 802, T=64, H=256, E=8, n_group=4,
                               topk_group=2, topk=2, I=128, I_shared=128,
                               router_sigma=0.05)
    d, W, args, grads = _small_case(cfg)
    first = [host(t).copy() for t in grads.tensors()]
    run_backward(d, W, *args, accumulate=True, grads=grads)
    for a, b in zip(first, grads.tensors()):
        assert np.array_equal(2 * a, host(b))


def test_backward_v3_prefill_sampled(v3_weights):
    """The V3 prefill size (T = 4096, 256 experts of 7168 x 2048, top-8):
    the busiest expert's three weight gradients and its rows' gate
    gradients in full, the smallest segment's, the shared expert's three
    weight gradients in full, and dx of sampled tokens (each with its 8
    experts and the shared expert)."""
    cfg = inputs.CONFIGS["prefill_v3"]
    d = ops.dims_of(cfg)
    T, K, E = cfg.T, cfg.topk, cfg.E
    x = inputs.x_tokens(cfg)
    xf = f32(x)
    z = O.router_logits(xf, inputs.router_weight(cfg))
    r = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group, K)
    idx, gate = r["idx"], r["gate"]
    dout = _dout(cfg, T)
    do = f32(dout).astype(np.float64)
    dx, dg, grads = run_backward(d, v3_weights, dev(x), dev(dout), dev(idx),
                                 dev(gate))
    counts = O.expert_counts(idx, E)
    busy = int(np.argmax(counts))
    nz = np.nonzero(counts)[0]
    small = int(nz[np.argmin(counts[nz])])
    dg_h = host(dg)
    for e in (busy, small):
        t, k = np.nonzero(idx == e)
        w1, w3, w2 = (f32(m) for m in inputs.expert_weights(cfg, e))
        gk = gate[t, k].astype(np.float64)
        tm = expert_terms(xf[t], gk[:, None] * do[t], gk, w1, w3, w2)
        b1, b3, b2 = wgrad_bounds(tm, xf[t], t.size)
        _, r1, r3, r2 = O.swiglu_ffn_backward(xf[t], w1, w3, w2,
                                              gk[:, None] * do[t])
        check(host(grads.dw1[e]), r1, b1, f"dw1[{e}]")
        check(host(grads.dw3[e]), r3, b3, f"dw3[{e}]")
        check(host(grads.dw2[e]), r2, b2, f"dw2[{e}]")
        y = O.swiglu_ffn(xf[t], w1, w3, w2)
        ref_g = np.einsum("nh,nh->n", do[t], y)
        bnd = w2.shape[1] * V * (np.abs(tm["D"]) * np.abs(tm["m"])).sum(1) \
            + (np.abs(tm["D"]) * tm["e_m"] + tm["e_D"] * np.abs(tm["m"])).sum(1)
        check(dg_h[t, k], ref_g, bnd, f"dgate[{e}]")
    s1, s3, s2 = (f32(m) for m in inputs.shared_weights(cfg))
    ts = expert_terms(xf, do, np.ones(T), s1, s3, s2)
    bs1, bs3, bs2 = wgrad_bounds(ts, xf, T)
    _, q1, q3, q2 = O.swiglu_ffn_backward(xf, s1, s3, s2, do)
    check(host(grads.dws1), q1, bs1, "dws1")
    check(host(grads.dws3), q3, bs3, "dws3")
    check(host(grads.dws2), q2, bs2, "dws2")
    # dx of sampled tokens: residual + shared + their 8 experts
    rows = np.arange(0, T, 1023)
    sv, se = row_grad_terms(
        expert_terms(xf[rows], do[rows], np.ones(rows.size), s1, s3, s2),
        s1, s3)
    ref = do[rows] + sv
    err = se.copy()
    absum = np.abs(do[rows]) + np.abs(sv)
    for i, t in enumerate(rows):
        for k in range(K):
            e = int(idx[t, k])
            w1, w3, w2 = (f32(m) for m in inputs.expert_weights(cfg, e))
            gk = np.array([float(gate[t, k])])
            tm = expert_terms(xf[t:t + 1], gk[:, None] * do[t:t + 1], gk, w1,
                              w3, w2)
            v, ev = row_grad_terms(tm, w1, w3)
            ref[i] += v[0]
            err[i] += ev[0]
            absum[i] += np.abs(v[0])
    bound = U * (np.abs(ref) + err) + err + (K + 2) * V * absum
    check(bf16_dev_to_f32(dx)[rows], ref, bound, "dx")
    # nothing left unwritten
    assert bool(torch.isfinite(dg).all())
    assert bool(torch.isfinite(dx.view(torch.bfloat16)).all())
    for t in grads.tensors():
        assert bool(torch.isfinite(t).all())
