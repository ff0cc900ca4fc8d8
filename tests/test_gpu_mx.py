"""FP8 with power-of-two group scales on the GPU against the oracle
("02 · DeepSeek-V3" §2: E4M3 operands in 1 x 128 activation tiles and
128 x 128 weight blocks; here each group's scale is a power of two held as
a UE8M0 byte, the microscaling form the page points to for Blackwell's
tensor cores, which apply it inside the block-scaled MMA).

Quantization is integer work decided from the same fp32 values on both
sides: codes and scale bytes are compared bit for bit, on inputs that reach
the rule's edges (all-zero tiles, subnormal maxima, maxima exactly 448 * 2^k
and one bf16 step above, the largest bf16 magnitudes).  The FFN is compared
with the oracle's FFN on the oracle's own codes and scales, with the FP8
bar of gpu_helpers.fp8_ffn_check: fp32 accumulation order and the fp32
SwiGLU, plus the rare one-step flips of an intermediate code."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import bf16_dev_to_f32, dev, fp8_ffn_check, host

pytestmark = pytest.mark.gpu

f32 = inputs.bf16_bits_to_f32


def _bf16_bits(x):
    """fp32 -> bf16 bits by truncation (the test inputs are exact bf16)."""
    return (np.asarray(x, np.float32).view(np.uint32) >> 16).astype(np.uint16)


def _scale_bytes(s):
    """UE8M0 bytes of the oracle's power-of-two scales."""
    m, e = np.frexp(np.asarray(s, np.float64))
    assert np.all(m == 0.5)
    return (e - 1 + 127).astype(np.uint8)


def _edge_rows(rng, R, C):
    """bf16 rows whose 128-wide tiles hit the exponent rule's edges."""
    x = (rng.standard_normal((R, C)) *
         np.exp2(rng.integers(-30, 30, (R, 1)))).astype(np.float32)
    t = x.reshape(R, C // 128, 128)
    t[0, 0] = 0.0                                   # all-zero tile
    if R > 1:                                       # subnormal maximum
        t[1, 0] = rng.standard_normal(128) * 2.0 ** -140
        t[1, 0, 3] = 2.0 ** -133
    for i, k in enumerate(range(-5, 5)):            # amax = 448 * 2^k ...
        r = 2 + i
        if r >= R:
            break
        t[r, 0] = np.clip(t[r, 0], -1, 1) * 448.0 * 2.0 ** k
        t[r, 0, 7] = 448.0 * 2.0 ** k
        if t.shape[1] > 1:                          # ... and one bf16 step up
            t[r, 1, 9] = np.float32(448.0 * 2.0 ** k * (1 + 2.0 ** -7))
    if R > 1:                                       # largest magnitudes
        t[-1, -1, 0] = 3.3e38
        t[-1, -1, 1] = -3.0e38
    xb = _bf16_bits(t.reshape(R, C))
    return xb, f32(xb)


@pytest.mark.parametrize("R,C", [(37, 512), (1, 128), (300, 1024)])
def test_quantize_rows_bit_exact(R, C):
    rng = np.random.default_rng(R * 7 + C)
    xb, xf = _edge_rows(rng, R, C)
    q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    s = torch.empty((R, C // 128), dtype=torch.uint8, device="cuda")
    ops.moe_quantize_mx_rows(dev(xb.view(np.int16)), q, s)
    wq, ws = O.quantize_1x128_pow2(xf)
    np.testing.assert_array_equal(host(q), wq)
    np.testing.assert_array_equal(host(s), _scale_bytes(ws))


@pytest.mark.parametrize("R,C", [(256, 384), (128, 128)])
def test_quantize_blocks_bit_exact(R, C):
    rng = np.random.default_rng(R + C)
    xb, xf = _edge_rows(rng, R, C)
    q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    s = torch.empty((R // 128, C // 128), dtype=torch.uint8, device="cuda")
    ops.moe_quantize_mx_blocks(dev(xb.view(np.int16)), q, s)
    wq, ws = O.quantize_128x128_pow2(xf)
    np.testing.assert_array_equal(host(q), wq)
    np.testing.assert_array_equal(host(s), _scale_bytes(ws))


def test_permute_mx_rows_are_the_tokens_codes():
    cfg = inputs.custom_config("mxp", 990, T=150, H=384, E=16, n_group=4,
                               topk_group=2, topk=4, I=128, I_shared=128,
                               router_sigma=0.05)
    T, K, H, E = cfg.T, cfg.topk, cfg.H, cfg.E
    d = ops.dims_of(cfg)
    xb = inputs.x_tokens(cfg)
    z = O.router_logits(f32(xb), inputs.router_weight(cfg))
    idx = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group,
                  K)["idx"]
    p = O.permutation(idx, E)
    xq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    xs = torch.empty((T, H // 128), dtype=torch.uint8, device="cuda")
    xpq = torch.empty((T * K, H), dtype=torch.uint8, device="cuda")
    xps = torch.empty((T * K, H // 128), dtype=torch.uint8, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_PERMUTE)
    ops.moe_permute_mx(d, dev(xb), dev(p["dest"]), xq, xs, xpq, xps, ws)
    assert ops.moe_get_device_error(ws) == 0
    wq, wsc = O.quantize_1x128_pow2(f32(xb))
    np.testing.assert_array_equal(host(xq), wq)
    np.testing.assert_array_equal(host(xs), _scale_bytes(wsc))
    tok = p["src_row"] // K
    np.testing.assert_array_equal(host(xpq), wq[tok])
    np.testing.assert_array_equal(host(xps), _scale_bytes(wsc)[tok])


# ----------------------------------------------------------------- FFN
def _host_weights(cfg, e):
    w1, w3, w2 = (f32(m) for m in inputs.expert_weights(cfg, e))
    return [O.quantize_128x128_pow2(w) for w in (w1, w3, w2)]


def _shared(cfg):
    s1, s3, s2 = (f32(m) for m in inputs.shared_weights(cfg))
    return {"ws1": O.quantize_128x128_pow2(s1),
            "ws3": O.quantize_128x128_pow2(s3),
            "ws2": O.quantize_128x128_pow2(s2)}


def _dev_pair(q, s):
    return dev(q), dev(_scale_bytes(s))


def _ffn(cfg, idx, per, sh, T):
    K, E, H = cfg.topk, cfg.E, cfg.H
    d = ops.dims_of(cfg, T=T)
    p = O.permutation(idx, E)
    xq, xs = O.quantize_1x128_pow2(f32(inputs.x_tokens(cfg, T=T)))
    tok = p["src_row"] // K
    routed = {}
    for i, n in enumerate(("w1", "w3", "w2")):
        routed[n] = (np.concatenate([per[e][i][0] for e in range(E)]),
                     np.concatenate([per[e][i][1] for e in range(E)]))
    W = ops.WeightsMx(**{n: _dev_pair(q, s) for n, (q, s) in
                         {**routed, **sh}.items()})
    yp = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
    ys = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN_MX)
    xsb = _scale_bytes(xs)
    ops.moe_expert_ffn_mx(d, W, dev(xq[tok]), dev(xsb[tok]), dev(xq),
                          dev(xsb), dev(p["offsets"]), yp, ys, ws)
    assert ops.moe_get_device_error(ws) == 0
    return bf16_dev_to_f32(yp), bf16_dev_to_f32(ys), p, xq, xs


def _assert_layer(cfg, idx, T=None, shared_rows=None):
    T = cfg.T if T is None else T
    per = [_host_weights(cfg, e) for e in range(cfg.E)]
    sh = _shared(cfg)
    yp, ys, p, xq, xs = _ffn(cfg, idx, per, sh, T)
    off = p["offsets"]
    pow2 = O.quantize_1x128_pow2
    for e in range(cfg.E):
        a, b = off[e], off[e + 1]
        if a == b:
            continue
        rows = p["src_row"][a:b] // cfg.topk
        ref, m = O.fp8_swiglu_ffn(xq[rows], xs[rows], *per[e], requant=pow2)
        fp8_ffn_check(yp[a:b], ref, f"expert {e}", m,
                      O.dequantize(*per[e][2], 128))
    rows = np.arange(T) if shared_rows is None else shared_rows
    ref, m = O.fp8_swiglu_ffn(xq[rows], xs[rows], sh["ws1"], sh["ws3"],
                              sh["ws2"], requant=pow2)
    fp8_ffn_check(ys[rows], ref, "shared", m, O.dequantize(*sh["ws2"], 128))


def _routed(cfg):
    z = O.router_logits(f32(inputs.x_tokens(cfg)), inputs.router_weight(cfg))
    return O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group,
                   cfg.topk)["idx"]


def test_small_layer_every_row():
    """~75 rows per expert (the streaming shape, chunks up to 192 rows:
    narrow and wide accumulator layouts); the shared expert's 300 rows in
    two chunks of 150 (two token scale atoms)."""
    cfg = inputs.custom_config("mx", 991, T=300, H=512, E=8, n_group=4,
                               topk_group=2, topk=2, I=256, I_shared=256,
                               router_sigma=0.05)
    _assert_layer(cfg, _routed(cfg))


def _idx_with_counts(T, K, want, rest):
    """[T, K] expert ids with expert e in exactly want[e] slots, the other
    slots cycling over `rest`, no token choosing an expert twice."""
    slots = []
    for e, n in want.items():
        slots += [e] * n
    i = 0
    while len(slots) < T * K:
        slots.append(rest[i % len(rest)])
        i += 1
    slots = np.array(slots[:T * K])
    idx = slots.reshape(K, T).T.copy()
    for k in range(1, K):
        for t in np.nonzero(np.any(idx[:, :k] == idx[:, k:k + 1], axis=1))[0]:
            for alt in rest:
                if alt not in idx[t]:
                    idx[t, k] = alt
                    break
    assert np.all([len(set(r)) == K for r in idx])
    return idx.astype(np.int32)


def test_ragged_chunk_shapes():
    """Expert 3 no rows, expert 0 one row (N = 16), expert 1 113 rows (the
    first wide chunk, N = 128), expert 2 193 rows (two chunks of 97 -> N =
    112, narrow), expert 4 129 rows (N = 144: a second token atom)."""
    cfg = inputs.custom_config("mxr", 992, T=400, H=384, E=8, n_group=4,
                               topk_group=2, topk=2, I=256, I_shared=128,
                               router_sigma=0.05)
    idx = _idx_with_counts(400, 2, {0: 1, 1: 113, 2: 193, 4: 129},
                           [5, 6, 7])
    c = O.expert_counts(idx, cfg.E)
    assert c[3] == 0 and c[0] == 1 and c[1] == 113 and c[2] == 193
    _assert_layer(cfg, idx, T=400)


def test_compute_shape_wide_chunks():
    """Mean 300 rows per expert: the 224-row shape; a 224-row expert (one
    full chunk, two token atoms) and a 449-row one (three chunks)."""
    cfg = inputs.custom_config("mxc", 993, T=600, H=256, E=4, n_group=2,
                               topk_group=2, topk=2, I=256, I_shared=128,
                               router_sigma=0.05)
    idx = _idx_with_counts(600, 2, {0: 224, 1: 449}, [2, 3])
    _assert_layer(cfg, idx, T=600)


@pytest.mark.parametrize("E,G,K,I,Is,T,H", [
    (32, 4, 3, 384, 128, 77, 384),   # down: the last 256-feature block
                                     # holds one 128-row tile only
    (16, 4, 1, 128, 256, 33, 640),   # top-1, one feature block per expert
    (64, 8, 6, 256, 384, 250, 256),
    (1024, 8, 8, 128, 128, 600, 256),  # the largest expert count
])
def test_expert_and_width_shapes(E, G, K, I, Is, T, H):
    cfg = inputs.custom_config("mxs", 994 + E + K, T=T, H=H, E=E,
                               n_group=G, topk_group=G // 2, topk=K, I=I,
                               I_shared=Is, router_sigma=0.05)
    _assert_layer(cfg, _routed(cfg))


def test_no_tokens_is_a_no_op():
    cfg = inputs.custom_config("mx0", 995, T=64, H=256, E=8, n_group=4,
                               topk_group=2, topk=2, I=128, I_shared=128,
                               router_sigma=0.05)
    d = ops.dims_of(cfg, T=0)
    per = [_host_weights(cfg, e) for e in range(cfg.E)]
    routed = {n: (np.concatenate([per[e][i][0] for e in range(cfg.E)]),
                  np.concatenate([per[e][i][1] for e in range(cfg.E)]))
              for i, n in enumerate(("w1", "w3", "w2"))}
    W = ops.WeightsMx(**{n: _dev_pair(q, s) for n, (q, s) in
                         {**routed, **_shared(cfg)}.items()})
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN_MX)
    off = torch.zeros(cfg.E + 1, dtype=torch.int32, device="cuda")
    ops.moe_expert_ffn_mx(d, W, None, None, None, None, off, None, None, ws)
    assert ops.moe_get_device_error(ws) == 0


@pytest.mark.parametrize("name", ["decode_v3", "prefill_v3"])
def test_v3_full_size_sampled_experts(name):
    """The V3 decode (T = 128) and prefill (T = 4096, ~128 rows per expert:
    one chunk per weight tile) layers: 256 experts of 7168 x 2048, top-8,
    quantized on the device; the oracle quantizes the sampled experts' bf16
    weights itself.  Compared: the two busiest experts' whole segments, a
    one-row expert if any, and a strided sample of shared-expert rows."""
    cfg = inputs.CONFIGS[name]
    T, K, E, H = cfg.T, cfg.topk, cfg.E, cfg.H
    d = ops.dims_of(cfg)
    w1, w3, w2 = inputs.device_expert_weights(cfg, "cuda")
    s1, s3, s2 = (dev(m) for m in inputs.shared_weights(cfg))
    W = ops.WeightsMx.quantize(w1, w3, w2, s1, s3, s2)
    del w1, w3, w2
    torch.cuda.empty_cache()
    idx = _routed(cfg)
    p = O.permutation(idx, E)
    xq, xs = O.quantize_1x128_pow2(f32(inputs.x_tokens(cfg)))
    xsb = _scale_bytes(xs)
    tok = p["src_row"] // K
    yp = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
    ys = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN_MX)
    ops.moe_expert_ffn_mx(d, W, dev(xq[tok]), dev(xsb[tok]), dev(xq),
                          dev(xsb), dev(p["offsets"]), yp, ys, ws)
    assert ops.moe_get_device_error(ws) == 0
    yp, ys = bf16_dev_to_f32(yp), bf16_dev_to_f32(ys)
    counts = np.diff(p["offsets"])
    busy = np.argsort(-counts, kind="stable")[:2].tolist()
    one = int(np.nonzero(counts == 1)[0][0]) if np.any(counts == 1) else None
    pow2 = O.quantize_1x128_pow2
    for e in busy + ([one] if one is not None else []):
        a, b = p["offsets"][e], p["offsets"][e + 1]
        hw = _host_weights(cfg, e)
        ref, m = O.fp8_swiglu_ffn(xq[tok[a:b]], xs[tok[a:b]], *hw,
                                  requant=pow2)
        fp8_ffn_check(yp[a:b], ref, f"expert {e}", m,
                      O.dequantize(*hw[2], 128))
    sh = _shared(cfg)
    rows = np.arange(0, T, max(9, T // 40))
    ref, m = O.fp8_swiglu_ffn(xq[rows], xs[rows], sh["ws1"], sh["ws3"],
                              sh["ws2"], requant=pow2)
    fp8_ffn_check(ys[rows], ref, "shared", m, O.dequantize(*sh["ws2"], 128))


def test_routed_only_call_equals_the_full_call():
    """moe_expert_ffn_mx_routed (expert parallelism's receive side: rows
    only, no shared expert) on the full call's routed rows gives the same
    outputs bit for bit: the same units, the same accumulation order."""
    cfg = inputs.custom_config("mxro", 996, T=200, H=384, E=8, n_group=4,
                               topk_group=2, topk=2, I=256, I_shared=128,
                               router_sigma=0.05)
    T, K, E, H = cfg.T, cfg.topk, cfg.E, cfg.H
    per = [_host_weights(cfg, e) for e in range(E)]
    sh = _shared(cfg)
    yp, ys, p, xq, xs = _ffn(cfg, _routed(cfg), per, sh, T)
    routed = {n: _dev_pair(np.concatenate([per[e][i][0] for e in range(E)]),
                           np.concatenate([per[e][i][1] for e in range(E)]))
              for i, n in enumerate(("w1", "w3", "w2"))}
    W = ops.WeightsMx(**routed)
    R = T * K
    d = ops.dims(R, H, E, 1, 1, 1, cfg.I, cfg.I_shared, cfg.gamma)
    tok = p["src_row"] // K
    out = torch.zeros((R, H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN_MX)
    ops.moe_expert_ffn_mx_routed(d, W, dev(xq[tok]),
                                 dev(_scale_bytes(xs)[tok]),
                                 dev(p["offsets"]), out, ws)
    assert ops.moe_get_device_error(ws) == 0
    np.testing.assert_array_equal(bf16_dev_to_f32(out), yp)
