"""FP8 expert FFNs on the GPU against the oracle ("02 · DeepSeek-V3" §2:
E4M3 operands, 1 x 128 activation / 128 x 128 weight scales, promotion of
every 128-element slice of the reduction into fp32).

The oracle's codes and scales -- its own quantization of the same bf16
tokens and weights -- are the GPU's inputs, so both sides multiply the same
E4M3 values.  They differ by fp32 accumulation order and the fp32 SwiGLU
(~1e-6 relative), and so, rarely, in an intermediate code: the GPU's m and
the oracle's (fp64) m can fall on the two sides of a rounding midpoint, and
one E4M3 step is up to 1/8 of the value, carried into y through a column
of W2.  Bar, per element of y (token t, feature j):
  |y_gpu - y| <= 2^-8 |y| + 1e-3 RMS(y) + 2 max_i step_i(t) |W2_ji|
(bf16 rounding of y, accumulation noise, and up to two one-step code
differences per token, step_i(t) = the E4M3 spacing at the oracle's code
of m_i(t) times its scale); and RMS error <= 5e-3 RMS(y)."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import bf16_dev_to_f32, dev, fp8_ffn_check

pytestmark = pytest.mark.gpu

f32 = inputs.bf16_bits_to_f32


def _host_weights(cfg, e):
    w1, w3, w2 = (f32(m) for m in inputs.expert_weights(cfg, e))
    return [O.quantize_128x128(w) for w in (w1, w3, w2)]


def _run(cfg, idx, qw_routed, qw_shared, T=None):
    """GPU FP8 FFN for routing idx; the oracle's quantized tokens and the
    given (codes, scales) weights.  Returns yp, ys (fp32) and the oracle
    permutation."""
    T = cfg.T if T is None else T
    K, E, H = cfg.topk, cfg.E, cfg.H
    d = ops.dims_of(cfg, T=T)
    p = O.permutation(idx, E)
    xq, xs = O.quantize_1x128(f32(inputs.x_tokens(cfg, T=T)))
    tok = p["src_row"] // K
    W = ops.WeightsFp8(**{n: (dev(q), dev(s)) for n, (q, s) in
                          {**qw_routed, **qw_shared}.items()})
    yp = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
    ys = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN_FP8)
    ops.moe_expert_ffn_fp8(d, W, dev(xq[tok]), dev(xs[tok]), dev(xq), dev(xs),
                           dev(p["offsets"]), yp, ys, ws)
    assert ops.moe_get_device_error(ws) == 0
    return bf16_dev_to_f32(yp), bf16_dev_to_f32(ys), p, (xq, xs)


def _stack(cfg, experts):
    per = [_host_weights(cfg, e) for e in range(cfg.E)]
    out = {}
    for i, n in enumerate(("w1", "w3", "w2")):
        out[n] = (np.concatenate([per[e][i][0] for e in range(cfg.E)]),
                  np.concatenate([per[e][i][1] for e in range(cfg.E)]))
    return out, per


def _shared(cfg):
    s1, s3, s2 = (f32(m) for m in inputs.shared_weights(cfg))
    return {"ws1": O.quantize_128x128(s1), "ws3": O.quantize_128x128(s3),
            "ws2": O.quantize_128x128(s2)}


def _small_cfg():
    return inputs.custom_config("fp8", 970, T=300, H=512, E=8, n_group=4,
                                topk_group=2, topk=2, I=256, I_shared=256,
                                router_sigma=0.05)


def _assert_layer(cfg, idx, T=None, experts=None, shared_rows=None):
    routed, per = _stack(cfg, None)
    sh = _shared(cfg)
    yp, ys, p, (xq, xs) = _run(cfg, idx, routed, sh, T)
    off = p["offsets"]
    for e in (range(cfg.E) if experts is None else experts):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        rows = p["src_row"][a:b] // cfg.topk
        ref, m = O.fp8_swiglu_ffn(xq[rows], xs[rows], *per[e])
        fp8_ffn_check(yp[a:b], ref, f"expert {e}", m,
                      O.dequantize(*per[e][2], 128))
    rows = np.arange(xq.shape[0]) if shared_rows is None else shared_rows
    ref, m = O.fp8_swiglu_ffn(xq[rows], xs[rows], sh["ws1"], sh["ws3"],
                              sh["ws2"])
    fp8_ffn_check(ys[rows], ref, "shared", m,
                  O.dequantize(*sh["ws2"], 128))


def test_small_layer_every_row():
    cfg = _small_cfg()
    z = O.router_logits(f32(inputs.x_tokens(cfg)), inputs.router_weight(cfg))
    idx = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group,
                  cfg.topk)["idx"]
    _assert_layer(cfg, idx)


def test_empty_single_row_and_ragged_chunks():
    """Expert 3 gets no rows, expert 0 one row (MMA N = 16), expert 1 33
    rows (chunks of 32 and 1), expert 2 64 rows (two full chunks)."""
    cfg = _small_cfg()
    T, K = 200, cfg.topk
    idx = np.zeros((T, K), np.int32)
    want = {0: 1, 1: 33, 2: 64}
    rest = [4, 5, 6, 7]
    slots = []
    for e, n in want.items():
        slots += [e] * n
    i = 0
    while len(slots) < T * K:
        slots.append(rest[i % 4])
        i += 1
    slots = np.array(slots)
    # one expert per slot, never twice in a token: slot k of token t takes
    # the (t + k*T)-th entry of an ordering where no token repeats
    idx[:, 0] = slots[:T]
    idx[:, 1] = slots[T:]
    same = idx[:, 0] == idx[:, 1]
    idx[same, 1] = np.where(idx[same, 0] == 4, 5, 4)
    counts = O.expert_counts(idx, cfg.E)
    assert counts[3] == 0 and counts[0] >= 1
    _assert_layer(cfg, idx, T=T)


@pytest.mark.parametrize("E,G,K,I,Is,T", [
    (32, 4, 3, 384, 128, 77),      # 32 experts, shared I != routed I
    (16, 4, 1, 128, 256, 33),      # top-1, one feature block per expert
    (64, 8, 6, 256, 384, 250),
    (1024, 8, 8, 128, 128, 600),   # the largest expert count
])
def test_expert_and_width_shapes(E, G, K, I, Is, T):
    cfg = inputs.custom_config("fp8s", 980 + E + K, T=T, H=384, E=E,
                               n_group=G, topk_group=G // 2, topk=K, I=I,
                               I_shared=Is, router_sigma=0.05)
    z = O.router_logits(f32(inputs.x_tokens(cfg)), inputs.router_weight(cfg))
    idx = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group,
                  cfg.topk)["idx"]
    _assert_layer(cfg, idx)


def test_no_tokens_is_a_no_op():
    cfg = _small_cfg()
    d = ops.dims_of(cfg, T=0)
    routed, _ = _stack(cfg, None)
    W = ops.WeightsFp8(**{n: (dev(q), dev(s)) for n, (q, s) in
                          {**routed, **_shared(cfg)}.items()})
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN_FP8)
    off = torch.zeros(cfg.E + 1, dtype=torch.int32, device="cuda")
    ops.moe_expert_ffn_fp8(d, W, None, None, None, None, off, None, None, ws)
    assert ops.moe_get_device_error(ws) == 0


@pytest.mark.parametrize("name", ["decode_v3", "prefill_v3"])
def test_v3_full_size_sampled_experts(name):
    """The V3 decode (T = 128) and prefill (T = 4096: ~128 rows per expert,
    four 32-row chunks sharing each weight tile) layers: 256 experts of
    7168 x 2048, top-8.  All weights are generated and quantized on the
    device; the oracle quantizes the sampled experts' bf16 weights
    itself."""
    cfg = inputs.CONFIGS[name]
    T, K, E, H, I = cfg.T, cfg.topk, cfg.E, cfg.H, cfg.I
    d = ops.dims_of(cfg)
    w1, w3, w2 = inputs.device_expert_weights(cfg, "cuda")
    s1, s3, s2 = (dev(m) for m in inputs.shared_weights(cfg))
    W = ops.WeightsFp8.quantize(w1, w3, w2, s1, s3, s2)
    del w1, w3, w2
    z = O.router_logits(f32(inputs.x_tokens(cfg)), inputs.router_weight(cfg))
    idx = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group,
                  K)["idx"]
    p = O.permutation(idx, E)
    xq, xs = O.quantize_1x128(f32(inputs.x_tokens(cfg)))
    tok = p["src_row"] // K
    yp = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
    ys = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN_FP8)
    ops.moe_expert_ffn_fp8(d, W, dev(xq[tok]), dev(xs[tok]), dev(xq), dev(xs),
                           dev(p["offsets"]), yp, ys, ws)
    assert ops.moe_get_device_error(ws) == 0
    yp, ys = bf16_dev_to_f32(yp), bf16_dev_to_f32(ys)
    counts = np.diff(p["offsets"])
    busy = np.argsort(-counts, kind="stable")[:2].tolist()
    one = int(np.nonzero(counts == 1)[0][0]) if np.any(counts == 1) else None
    for e in busy + ([one] if one is not None else []):
        a, b = p["offsets"][e], p["offsets"][e + 1]
        rows = tok[a:b]
        hw = _host_weights(cfg, e)
        ref, m = O.fp8_swiglu_ffn(xq[rows], xs[rows], *hw)
        fp8_ffn_check(yp[a:b], ref, f"expert {e}", m,
                      O.dequantize(*hw[2], 128))
    sh = _shared(cfg)
    rows = np.arange(0, T, max(9, T // 40))
    ref, m = O.fp8_swiglu_ffn(xq[rows], xs[rows], sh["ws1"], sh["ws3"],
                              sh["ws2"])
    fp8_ffn_check(ys[rows], ref, "shared", m,
                  O.dequantize(*sh["ws2"], 128))
