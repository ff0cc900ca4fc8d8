"""Routing on the GPU against the oracle, bit for bit, given the same
logits: chosen experts, gates (fp32 bits), per-expert counts; and the bias
step.  Covers the V3 routing shape at its full size (16384 tokens), ragged
token counts, many expert/group shapes, exact ties, and the skewed
multi-step bias trajectory."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import assert_route_bit_exact, dev, f32_bits, host, route_gpu

pytestmark = pytest.mark.gpu


def test_tiny_config_from_oracle_logits():
    cfg = inputs.CONFIGS["tiny"]
    z = O.router_logits(inputs.bf16_bits_to_f32(inputs.x_tokens(cfg)),
                        inputs.router_weight(cfg))
    assert_route_bit_exact(ops.dims_of(cfg), z, inputs.bias(cfg))


def test_v3_routing_full_size_16384_tokens():
    cfg = inputs.CONFIGS["route_v3"]
    z = O.router_logits(inputs.bf16_bits_to_f32(inputs.x_tokens(cfg)),
                        inputs.router_weight(cfg))
    assert 0.3 < z.std() < 0.8      # logits of the recipe's scale
    r = assert_route_bit_exact(ops.dims_of(cfg), z, inputs.bias(cfg))
    assert np.all(r["kept"].sum(1) == 4)


# 1984 / 1985 / 9473: either side of the rounding of the routing blocks'
# number up to a multiple of 148 (31 blocks of 64; 148 of 13-14; 296 of 32)
@pytest.mark.parametrize("T", [1, 2, 63, 64, 65, 1000, 1984, 1985, 4097,
                               9473])
def test_ragged_token_counts(T):
    cfg = inputs.CONFIGS["route_v3"]
    z = inputs.random_logits(cfg, T=T, step=T)
    assert_route_bit_exact(ops.dims_of(cfg, T=T), z, inputs.bias(cfg))


@pytest.mark.parametrize("E,G,M,K", [
    (8, 4, 2, 2), (16, 4, 2, 4), (16, 8, 3, 5), (32, 4, 2, 6), (32, 16, 16, 32),
    (64, 8, 3, 8), (64, 16, 4, 8), (128, 4, 2, 8), (256, 1, 1, 8),
    (256, 8, 8, 8), (256, 8, 4, 1), (256, 32, 4, 8), (512, 16, 4, 16),
    (1024, 32, 8, 32), (1024, 8, 4, 8),
])
def test_expert_and_group_shapes(E, G, M, K):
    cfg = inputs.custom_config("shape", 100 + E + G + M + K, T=777, H=64, E=E,
                               n_group=G, topk_group=M, topk=K, I=64,
                               I_shared=64)
    z = inputs.random_logits(cfg, scale=1.0)
    b = np.random.default_rng(E * 7 + K).uniform(-0.05, 0.05, E).astype(
        np.float32)
    assert_route_bit_exact(ops.dims_of(cfg), z, b)


def test_exact_ties_break_to_the_lower_index():
    """Logits on a coarse grid: many equal affinities, equal group scores.
    Ties are broken by expert / group index on both sides."""
    cfg = inputs.CONFIGS["route_v3"]
    z = (np.round(inputs.random_logits(cfg, T=3000) * 2) / 2).astype(
        np.float32)
    assert_route_bit_exact(ops.dims_of(cfg, T=3000), z,
                           np.zeros(cfg.E, np.float32))
    zt = np.zeros((50, cfg.E), np.float32)        # all equal
    r = assert_route_bit_exact(ops.dims_of(cfg, T=50), zt,
                               np.zeros(cfg.E, np.float32))
    assert np.all(r["idx"] == np.arange(8))


def test_extreme_logits_and_bias():
    cfg = inputs.CONFIGS["route_v3"]
    rng = np.random.default_rng(11)
    z = rng.normal(0, 30, size=(512, cfg.E)).astype(np.float32)
    z[0, :] = 1e30
    z[1, :] = -1e30
    z[2, ::3] = np.inf
    b = rng.uniform(-2, 2, cfg.E).astype(np.float32)
    assert_route_bit_exact(ops.dims_of(cfg, T=512), z, b)


def test_sigmoid_bits_through_single_expert_groups():
    """K = E with one kept group returns every expert with gate s_e/sum s:
    the gates expose the sigmoid of every logit on a dense grid."""
    cfg = inputs.custom_config("sig", 300, T=4096, H=64, E=32, n_group=1,
                               topk_group=1, topk=32, I=64, I_shared=64)
    z = np.linspace(-90, 40, 4096 * 32, dtype=np.float32).reshape(4096, 32)
    assert_route_bit_exact(ops.dims_of(cfg), z, np.zeros(32, np.float32))


def test_bias_update_bit_exact():
    cfg = inputs.CONFIGS["route_v3"]
    d = ops.dims_of(cfg)
    rng = np.random.default_rng(12)
    counts = rng.multinomial(cfg.T * cfg.topk, np.full(cfg.E, 1 / cfg.E))
    counts[:5] = cfg.T * cfg.topk // cfg.E      # exactly at the mean
    counts[5] += cfg.T * cfg.topk - counts.sum()
    counts = counts.astype(np.int32)
    b = inputs.bias(cfg)
    bt = dev(b)
    stats = torch.zeros(3, dtype=torch.float32, device="cuda")
    ops.moe_bias_update(d, dev(counts), bt, stats)
    nb, st = O.bias_update(counts, b, cfg.T, cfg.topk, cfg.gamma)
    assert np.array_equal(f32_bits(host(bt)), f32_bits(nb))
    np.testing.assert_allclose(host(stats), st, rtol=1e-7)


def test_skewed_load_50_route_and_bias_steps():
    """The skewed workload's routing + bias loop (Zipf s=1.2 preference on
    the logits, b0 = 0, gamma = 0.001) on fresh tokens each step; the bias
    trajectory and every step's counts match the oracle bit for bit.  Run at
    4096 tokens per step for all 50 steps (the full 32768 is covered by the
    per-step routing test below)."""
    cfg = inputs.CONFIGS["skewed_v3"]
    T = 4096
    d = ops.dims_of(cfg, T=T)
    wr = inputs.router_weight(cfg)
    pref = inputs.zipf_preference(cfg)
    b = inputs.bias(cfg)
    bt = dev(b)
    ws = ops.workspace(d, ops.MOE_WS_ROUTE)
    idx = torch.empty((T, cfg.topk), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, cfg.topk), dtype=torch.float32, device="cuda")
    counts = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
    first_max = last_max = None
    for step in range(50):
        x = inputs.bf16_bits_to_f32(inputs.x_tokens(cfg, step=step, T=T))
        z = (O.router_logits(x, wr) + pref[None, :]).astype(np.float32)
        ops.moe_route(d, dev(z), bt, idx, gate, counts, ws)
        ops.moe_bias_update(d, counts, bt)
        r = O.route(z, b, cfg.n_group, cfg.topk_group, cfg.topk)
        c = O.expert_counts(r["idx"], cfg.E)
        b, _ = O.bias_update(c, b, T, cfg.topk, cfg.gamma)
        assert np.array_equal(host(counts), c), step
        assert np.array_equal(f32_bits(host(bt)), f32_bits(b)), step
        if step == 0:
            first_max = c.max()
        last_max = c.max()
    assert ops.moe_get_device_error(ws) == 0
    # the +-gamma steps pull the hottest expert's load down
    assert last_max < first_max


def test_skewed_full_size_one_step():
    cfg = inputs.CONFIGS["skewed_v3"]
    x = inputs.bf16_bits_to_f32(inputs.x_tokens(cfg, step=0))
    z = (O.router_logits(x, inputs.router_weight(cfg)) +
         inputs.zipf_preference(cfg)[None, :]).astype(np.float32)
    r = assert_route_bit_exact(ops.dims_of(cfg), z, inputs.bias(cfg))
    c = O.expert_counts(r["idx"], cfg.E)
    assert c.max() > 4 * c.mean()   # the preference makes hot experts


def test_zero_tokens():
    cfg = inputs.CONFIGS["route_v3"]
    d = ops.dims_of(cfg, T=0)
    counts = torch.full((cfg.E,), 5, dtype=torch.int32, device="cuda")
    e = torch.empty(0, dtype=torch.float32, device="cuda")
    ei = torch.empty(0, dtype=torch.int32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_ROUTE)
    ops.moe_route(d, e, dev(inputs.bias(cfg)), ei, e, counts, ws)
    assert np.all(host(counts) == 0)
