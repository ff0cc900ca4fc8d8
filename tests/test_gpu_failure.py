"""Failure detection on the GPU without a fault.

Every wait of the tensor-core kernels is bounded.  Here the bound is made
shorter than any TMA copy takes (1 ns), so the first wait that is not
already satisfied runs out: the kernel records MOE_ERR_TIMEOUT in the
workspace status word, raises its abort flag, drains its in-flight copies
and MMAs with their own bounded waits, frees tensor memory and returns.
The host reads the status, restores the default bound, and the same
context then computes correct results."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import bf16_dev_to_f32, dev

pytestmark = pytest.mark.gpu

TIMEOUT = ops.STATUS_CODES["MOE_ERR_TIMEOUT"]


def _ffn_call(cfg):
    d = ops.dims_of(cfg)
    T, K, H, E = cfg.T, cfg.topk, cfg.H, cfg.E
    x = inputs.x_tokens(cfg)
    z = O.router_logits(inputs.bf16_bits_to_f32(x), inputs.router_weight(cfg))
    idx = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group,
                  cfg.topk)["idx"]
    p = O.permutation(idx, E)
    w = inputs.layer_inputs(cfg)
    W = ops.Weights(dev(w["w_router"]), dev(w["w1"]), dev(w["w3"]),
                    dev(w["w2"]), dev(w["ws1"]), dev(w["ws3"]), dev(w["ws2"]))
    args = (dev(x[p["src_row"] // K]), dev(x), dev(p["offsets"]))

    def run():
        yp = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
        ys = torch.zeros((T, H), dtype=torch.int16, device="cuda")
        ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN)
        ops.moe_expert_ffn(d, W, *args, yp, ys, ws)
        return ops.moe_get_device_error(ws), yp, ys
    return run


def test_expert_ffn_wait_runs_out_then_context_recovers():
    cfg = inputs.custom_config("timeout", 960, T=300, H=512, E=8, n_group=4,
                               topk_group=2, topk=2, I=256, I_shared=128,
                               router_sigma=0.05)
    run = _ffn_call(cfg)
    code, _, _ = run()                    # reference, default bound
    assert code == 0
    _, yp_ref, ys_ref = run()
    try:
        ops.moe_set_wait_timeout_ns(1)
        for _ in range(2):                # twice: each launch recovers
            code, _, _ = run()
            assert code == TIMEOUT
    finally:
        ops.moe_set_wait_timeout_ns(0)    # back to the default bound
    code, yp, ys = run()
    assert code == 0
    assert torch.equal(yp, yp_ref) and torch.equal(ys, ys_ref)
    assert np.isfinite(bf16_dev_to_f32(yp)).all()


def test_router_gemm_wait_runs_out_then_context_recovers():
    cfg = inputs.CONFIGS["prefill_v3"]
    T = 512
    d = ops.dims_of(cfg, T=T)
    x = dev(inputs.x_tokens(cfg, T=T))
    w = dev(inputs.router_weight(cfg))
    ws = ops.workspace(d, ops.MOE_WS_ROUTER_LOGITS)
    z_ref = torch.empty((T, cfg.E), dtype=torch.float32, device="cuda")
    ops.moe_router_logits(d, x, w, z_ref, ws)
    assert ops.moe_get_device_error(ws) == 0
    try:
        ops.moe_set_wait_timeout_ns(1)
        z = torch.empty_like(z_ref)
        ops.moe_router_logits(d, x, w, z, ws)
        assert ops.moe_get_device_error(ws) == TIMEOUT
    finally:
        ops.moe_set_wait_timeout_ns(0)
    z = torch.empty_like(z_ref)
    ops.moe_router_logits(d, x, w, z, ws)
    assert ops.moe_get_device_error(ws) == 0
    assert torch.equal(z, z_ref)


def test_fp8_expert_ffn_wait_runs_out_then_context_recovers():
    """The FP8 GEMMs' waits (producer, MMA, promotion warps) are bounded the
    same way: all four promotion warps stop together on the shared go/stop
    word, TMEM is freed, and the next launch is exact again."""
    cfg = inputs.custom_config("timeout8", 961, T=300, H=512, E=8,
                               n_group=4, topk_group=2, topk=2, I=256,
                               I_shared=256, router_sigma=0.05)
    d = ops.dims_of(cfg)
    T, K, H, E = cfg.T, cfg.topk, cfg.H, cfg.E
    f32 = inputs.bf16_bits_to_f32
    x = f32(inputs.x_tokens(cfg))
    idx = O.route(O.router_logits(x, inputs.router_weight(cfg)),
                  inputs.bias(cfg), cfg.n_group, cfg.topk_group, K)["idx"]
    p = O.permutation(idx, E)
    xq, xs = O.quantize_1x128(x)
    tok = p["src_row"] // K
    per = [[O.quantize_128x128(f32(m)) for m in inputs.expert_weights(cfg, e)]
           for e in range(E)]
    pairs = {n: (dev(np.concatenate([per[e][i][0] for e in range(E)])),
                 dev(np.concatenate([per[e][i][1] for e in range(E)])))
             for i, n in enumerate(("w1", "w3", "w2"))}
    for n, m in zip(("ws1", "ws3", "ws2"), inputs.shared_weights(cfg)):
        q, s = O.quantize_128x128(f32(m))
        pairs[n] = (dev(q), dev(s))
    W = ops.WeightsFp8(**pairs)
    args = (dev(xq[tok]), dev(xs[tok]), dev(xq), dev(xs), dev(p["offsets"]))

    def run():
        yp = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
        ys = torch.zeros((T, H), dtype=torch.int16, device="cuda")
        ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN_FP8)
        ops.moe_expert_ffn_fp8(d, W, *args, yp, ys, ws)
        return ops.moe_get_device_error(ws), yp, ys
    code, yp_ref, ys_ref = run()
    assert code == 0
    try:
        ops.moe_set_wait_timeout_ns(1)
        for _ in range(2):
            code, _, _ = run()
            assert code == TIMEOUT
    finally:
        ops.moe_set_wait_timeout_ns(0)
    code, yp, ys = run()
    assert code == 0
    assert torch.equal(yp, yp_ref) and torch.equal(ys, ys_ref)


def test_mx_expert_ffn_wait_runs_out_then_context_recovers():
    """The power-of-two-scale FP8 GEMMs' waits (weight producer, the scale
    and token producer warp, MMA, the eight epilogue warps) are bounded the
    same way: the epilogue warps vote per unit and stop together, the
    in-flight copies and MMAs are drained, TMEM is freed, and the next
    launch is exact again."""
    cfg = inputs.custom_config("timeoutmx", 962, T=300, H=512, E=8,
                               n_group=4, topk_group=2, topk=2, I=256,
                               I_shared=256, router_sigma=0.05)
    d = ops.dims_of(cfg)
    T, K, H, E = cfg.T, cfg.topk, cfg.H, cfg.E
    f32 = inputs.bf16_bits_to_f32
    x = f32(inputs.x_tokens(cfg))
    idx = O.route(O.router_logits(x, inputs.router_weight(cfg)),
                  inputs.bias(cfg), cfg.n_group, cfg.topk_group, K)["idx"]
    p = O.permutation(idx, E)

    def e8(s):   # power-of-two scales -> UE8M0 bytes
        return (np.frexp(s.astype(np.float64))[1] + 126).astype(np.uint8)
    xq, xs = O.quantize_1x128_pow2(x)
    tok = p["src_row"] // K
    per = [[O.quantize_128x128_pow2(f32(m))
            for m in inputs.expert_weights(cfg, e)] for e in range(E)]
    pairs = {n: (dev(np.concatenate([per[e][i][0] for e in range(E)])),
                 dev(np.concatenate([e8(per[e][i][1]) for e in range(E)])))
             for i, n in enumerate(("w1", "w3", "w2"))}
    for n, m in zip(("ws1", "ws3", "ws2"), inputs.shared_weights(cfg)):
        q, s = O.quantize_128x128_pow2(f32(m))
        pairs[n] = (dev(q), dev(e8(s)))
    W = ops.WeightsMx(**pairs)
    args = (dev(xq[tok]), dev(e8(xs)[tok]), dev(xq), dev(e8(xs)),
            dev(p["offsets"]))

    def run():
        yp = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
        ys = torch.zeros((T, H), dtype=torch.int16, device="cuda")
        ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN_MX)
        ops.moe_expert_ffn_mx(d, W, *args, yp, ys, ws)
        return ops.moe_get_device_error(ws), yp, ys
    code, yp_ref, ys_ref = run()
    assert code == 0
    try:
        ops.moe_set_wait_timeout_ns(1)
        for _ in range(2):
            code, _, _ = run()
            assert code == TIMEOUT
    finally:
        ops.moe_set_wait_timeout_ns(0)
    code, yp, ys = run()
    assert code == 0
    assert torch.equal(yp, yp_ref) and torch.equal(ys, ys_ref)


def test_expert_backward_waits_run_out_then_context_recovers():
    """The backward's four tensor-core GEMMs (recompute, both dgrads, the
    weight gradients) under the 1 ns bound: the call reports
    MOE_ERR_TIMEOUT, twice in a row; with the default bound restored the
    same context reproduces every output bit for bit."""
    cfg = inputs.custom_config("timeout_bwd", 963, T=96, H=256, E=8,
                               n_group=4, topk_group=2, topk=2, I=128,
                               I_shared=128, router_sigma=0.05)
    d = ops.dims_of(cfg)
    w = inputs.layer_inputs(cfg)
    z = O.router_logits(inputs.bf16_bits_to_f32(w["x"]), w["w_router"])
    r = O.route(z, w["bias"], cfg.n_group, cfg.topk_group, cfg.topk)
    W = ops.Weights(dev(w["w_router"]), dev(w["w1"]), dev(w["w3"]),
                    dev(w["w2"]), dev(w["ws1"]), dev(w["ws3"]), dev(w["ws2"]))
    dout = inputs.normal_bf16(12345, (cfg.T, cfg.H), 1.0)
    args = (dev(w["x"]), dev(dout), dev(r["idx"]), dev(r["gate"]))

    def run():
        dx = torch.zeros((cfg.T, cfg.H), dtype=torch.int16, device="cuda")
        dg = torch.zeros((cfg.T, cfg.topk), dtype=torch.float32,
                         device="cuda")
        g = ops.WeightGrads.empty(d)
        ws = ops.workspace(d, ops.MOE_WS_EXPERT_BWD)
        ops.moe_expert_backward(d, W, *args, dx, dg, g, ws)
        code = ops.moe_get_device_error(ws)
        return code, [t.cpu().numpy() for t in [dx, dg] + g.tensors()]
    code, ref = run()
    assert code == 0
    try:
        ops.moe_set_wait_timeout_ns(1)
        for _ in range(2):
            code, _ = run()
            assert code == TIMEOUT
    finally:
        ops.moe_set_wait_timeout_ns(0)
    code, again = run()
    assert code == 0
    for a, b in zip(ref, again):
        assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
