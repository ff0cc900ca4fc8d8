"""Router logits z = x W_r^T (+ o) on the GPU against the oracle's fp64 sum.

Every product x_h * w_h is exact (bf16 x the exact bf16 split of the fp32
weight on the tensor-core path; fp32 FMA on the SIMT path), so the only
error is fp32 accumulation: for any summation order
    |z_gpu - z| <= H * 2^-24 * sum_h |x_h w_h| + 2^-24 |z|
(with an additive per-expert offset o, one more fp32 rounding of the sum:
another 2^-24 |z| + 2^-24 |o|).
The test asserts that bound elementwise, and a typical error far below it."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu


def check_logits(cfg, T=None, offset=None):
    T = cfg.T if T is None else T
    d = ops.dims_of(cfg, T=T)
    x = inputs.x_tokens(cfg, T=T)
    w = inputs.router_weight(cfg)
    z = torch.full((T, cfg.E), np.nan, dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_ROUTER_LOGITS)
    ops.moe_router_logits(d, dev(x), dev(w), z, ws,
                          router_offset=None if offset is None else dev(offset))
    assert ops.moe_get_device_error(ws) == 0
    zg = host(z).astype(np.float64)
    xf = inputs.bf16_bits_to_f32(x).astype(np.float64)
    ref = xf @ w.astype(np.float64).T                 # exact-ish fp64
    mag = np.abs(xf) @ np.abs(w.astype(np.float64)).T
    bound = cfg.H * 2.0 ** -24 * mag + 2.0 ** -24 * np.abs(ref)
    if offset is not None:
        o = offset.astype(np.float64)[None, :]
        bound = bound + 2.0 ** -24 * (np.abs(ref) + np.abs(o))
        ref = ref + o
    err = np.abs(zg - ref)
    assert np.all(err <= bound), (err / bound).max()
    assert np.sqrt(np.mean(err ** 2)) < 1e-2 * np.sqrt(np.mean(bound ** 2))
    # and the oracle's own rounding of the same sum
    np.testing.assert_allclose(zg, O.router_logits(xf, w, offset), rtol=0,
                               atol=float(bound.max()))


def test_router_logits_v3_prefill_4096_tokens():
    check_logits(inputs.CONFIGS["prefill_v3"])


@pytest.mark.parametrize("T", [1, 100, 129])
def test_router_logits_v3_ragged(T):
    check_logits(inputs.CONFIGS["prefill_v3"], T=T)


@pytest.mark.parametrize("E,G", [(16, 4), (32, 4), (64, 8), (128, 8),
                                 (512, 16), (8, 4), (24, 3)])
def test_router_logits_expert_counts(E, G):
    # E % 16 == 0 -> tensor cores with 16/32/64-wide tiles; 8, 24 -> SIMT
    cfg = inputs.custom_config("rl", 700 + E, T=300, H=512, E=E, n_group=G,
                               topk_group=2, topk=2, I=64, I_shared=64,
                               router_sigma=0.05)
    check_logits(cfg)


def test_router_logits_tiny_config():
    check_logits(inputs.CONFIGS["tiny"])


@pytest.mark.parametrize("E,G", [(256, 8), (24, 3)])
def test_router_logits_with_offset(E, G):
    # the skewed workload's per-expert preference as the router's additive
    # term, on the tensor-core (E=256) and SIMT (E=24) paths
    cfg = inputs.custom_config("rlo", 720 + E, T=300, H=512, E=E, n_group=G,
                               topk_group=2, topk=2, I=64, I_shared=64,
                               router_sigma=0.05)
    r = np.random.default_rng(E).permutation(E) + 1
    check_logits(cfg, offset=(1.0 * r ** -1.2).astype(np.float32))


def _bf16_rn(v):
    """fp32 -> nearest bf16 (ties to even), as fp32 (finite inputs)."""
    b = np.asarray(v, np.float32).view(np.uint32).astype(np.uint64)
    r = (b + 0x7FFF + ((b >> 16) & 1)) >> 16
    return (r << 16).astype(np.uint32).view(np.float32)


def test_router_weight_split_is_exact_and_reused_by_the_forward():
    """moe_router_weight_split writes hi = bf16(w), mid = bf16(w - hi),
    lo = bf16(w - hi - mid) (each residual exact in fp32), whose sum is w
    exactly; and moe_forward given that split (no per-call split) produces
    the same layer output, bit for bit, as moe_forward that splits."""
    cfg = inputs.custom_config("split", 1010, T=300, H=512, E=32, n_group=4,
                               topk_group=2, topk=4, I=128, I_shared=128,
                               router_sigma=0.05)
    w = inputs.router_weight(cfg)
    split = torch.zeros((3, cfg.E, cfg.H), dtype=torch.int16, device="cuda")
    ops.moe_router_weight_split(dev(w), split)
    parts = inputs.bf16_bits_to_f32(host(split, np.uint16))
    hi = _bf16_rn(w)
    mid = _bf16_rn(w - hi)
    lo = _bf16_rn((w - hi) - mid)
    np.testing.assert_array_equal(parts[0], hi)
    np.testing.assert_array_equal(parts[1], mid)
    np.testing.assert_array_equal(parts[2], lo)
    total = (parts[0].astype(np.float64) + parts[1] + parts[2])
    np.testing.assert_array_equal(total, w.astype(np.float64))
    lw = inputs.layer_inputs(cfg)
    W = ops.Weights(dev(lw["w_router"]), dev(lw["w1"]), dev(lw["w3"]),
                    dev(lw["w2"]), dev(lw["ws1"]), dev(lw["ws3"]),
                    dev(lw["ws2"]))
    Wp = W.with_router_split()
    d = ops.dims_of(cfg)
    outs = []
    for ww in (W, Wp):
        out = torch.zeros((cfg.T, cfg.H), dtype=torch.int16, device="cuda")
        ws = ops.workspace(d, ops.MOE_WS_FORWARD)
        ops.moe_forward(d, ww, dev(lw["x"]), dev(lw["bias"]), out, ws,
                        update_bias=False)
        assert ops.moe_get_device_error(ws) == 0
        outs.append(out)
    assert torch.equal(outs[0], outs[1])
