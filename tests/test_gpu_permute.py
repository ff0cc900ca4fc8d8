"""Dispatch order and gather on the GPU against the oracle: offsets, dest
and src_row bit for bit (the stable counting sort has one right answer),
and every gathered row equal to its token's row."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu


def permute_gpu(d, x_bits, idx, with_rows=True):
    T, K, H, E = d.T, d.topk, d.H, d.E
    offsets = torch.full((E + 1,), -9, dtype=torch.int32, device="cuda")
    dest = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    src_row = torch.full((T * K,), -9, dtype=torch.int32, device="cuda")
    xp = (torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
          if with_rows else None)
    ws = ops.workspace(d, ops.MOE_WS_PERMUTE)
    ops.moe_permute(d, dev(x_bits) if with_rows else None, dev(idx), offsets,
                    dest, src_row, xp, ws)
    assert ops.moe_get_device_error(ws) == 0
    return (host(offsets), host(dest), host(src_row),
            host(xp, np.uint16) if with_rows else None)


def check(d, x_bits, idx):
    ref = O.permutation(idx, d.E)
    off, dest, src, xp = permute_gpu(d, x_bits, idx)
    assert np.array_equal(off, ref["offsets"])
    assert np.array_equal(dest, ref["dest"])
    assert np.array_equal(src, ref["src_row"])
    t_of_row = src // d.topk
    assert np.array_equal(xp, x_bits[t_of_row])


def _random_idx(T, E, K, rng, hot=None):
    if hot is None:
        p = np.full(E, 1 / E)
    else:
        p = np.full(E, 1.0)
        p[:hot] = 200.0
        p /= p.sum()
    return np.stack([rng.choice(E, K, replace=False, p=p)
                     for _ in range(T)]).astype(np.int32)


# 1984: 31 routing blocks of 64 tokens; 1985: 32 blocks, their number
# rounded up to 148 (13-14 tokens each); 9473: 149 rounded up to 296
@pytest.mark.parametrize("T", [1, 31, 64, 65, 200, 1984, 1985, 4096, 9473])
def test_permute_v3_shape(T):
    cfg = inputs.CONFIGS["prefill_v3"]
    rng = np.random.default_rng(T)
    idx = _random_idx(T, cfg.E, cfg.topk, rng)
    check(ops.dims_of(cfg, T=T), inputs.x_tokens(cfg, T=T), idx)


def test_permute_from_routing_16384_tokens_indices_only():
    cfg = inputs.CONFIGS["route_v3"]
    z = inputs.random_logits(cfg)
    r = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group, cfg.topk)
    ref = O.permutation(r["idx"], cfg.E)
    off, dest, src, _ = permute_gpu(ops.dims_of(cfg), None, r["idx"],
                                    with_rows=False)
    assert np.array_equal(off, ref["offsets"])
    assert np.array_equal(dest, ref["dest"])
    assert np.array_equal(src, ref["src_row"])


def test_permute_hot_experts_and_empty_experts():
    """A few experts take most tokens, most get none (skewed load)."""
    cfg = inputs.custom_config("hot", 400, T=3000, H=256, E=64, n_group=8,
                               topk_group=4, topk=6, I=64, I_shared=64)
    rng = np.random.default_rng(5)
    idx = _random_idx(cfg.T, cfg.E, cfg.topk, rng, hot=6)
    idx[idx >= 40] = idx[idx >= 40] % 6 + 6   # experts 40.. never chosen
    idx = np.stack([np.unique(row) if len(np.unique(row)) == cfg.topk else
                    np.arange(cfg.topk) for row in idx]).astype(np.int32)
    check(ops.dims_of(cfg), inputs.x_tokens(cfg), idx)


def test_permute_tiny_config():
    cfg = inputs.CONFIGS["tiny"]
    z = O.router_logits(inputs.bf16_bits_to_f32(inputs.x_tokens(cfg)),
                        inputs.router_weight(cfg))
    r = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group, cfg.topk)
    check(ops.dims_of(cfg), inputs.x_tokens(cfg), r["idx"])


def test_invalid_expert_ids_are_reported_not_followed():
    """Out-of-range ids are skipped (dest = -1) and reported as a device
    bounds error; nothing is read or written out of bounds."""
    cfg = inputs.custom_config("bad", 401, T=100, H=64, E=32, n_group=4,
                               topk_group=2, topk=2, I=64, I_shared=64)
    d = ops.dims_of(cfg)
    idx = np.tile(np.array([[0, 1]], np.int32), (100, 1))
    idx[7, 1] = 999
    idx[9, 0] = -3
    x = inputs.x_tokens(cfg)
    offsets = torch.empty(33, dtype=torch.int32, device="cuda")
    dest = torch.empty((100, 2), dtype=torch.int32, device="cuda")
    src = torch.empty(200, dtype=torch.int32, device="cuda")
    xp = torch.zeros((200, 64), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_PERMUTE)
    ops.moe_permute(d, dev(x), dev(idx), offsets, dest, src, xp, ws)
    assert ops.moe_get_device_error(ws) == ops.STATUS_CODES["MOE_ERR_DEVICE_BOUNDS"]
    dh = host(dest)
    assert dh[7, 1] == -1 and dh[9, 0] == -1
    assert ops.moe_get_device_error(ws) == 0   # reading clears the word


def test_permute_skewed_32768_tokens_bit_exact():
    """The skewed-load batch (T = 32768, Zipf s = 1.2 preference on the
    logits): hot experts hold thousands of rows each.  Offsets, dest and
    src_row equal the oracle's stable counting sort bit for bit, and every
    one of the 262144 gathered rows equals its token's row."""
    cfg = inputs.CONFIGS["skewed_v3"]
    T, K, E = cfg.T, cfg.topk, cfg.E
    x = inputs.x_tokens(cfg)
    z = O.router_logits(inputs.bf16_bits_to_f32(x), inputs.router_weight(cfg),
                        inputs.zipf_preference(cfg))
    r = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group, K)
    del z
    ref = O.permutation(r["idx"], E)
    counts = np.diff(ref["offsets"])
    assert counts.max() > 8 * counts.mean()
    d = ops.dims_of(cfg)
    offsets = torch.full((E + 1,), -9, dtype=torch.int32, device="cuda")
    dest = torch.full((T, K), -9, dtype=torch.int32, device="cuda")
    src_row = torch.full((T * K,), -9, dtype=torch.int32, device="cuda")
    xd = dev(x)
    xp = torch.zeros((T * K, cfg.H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_PERMUTE)
    ops.moe_permute(d, xd, dev(r["idx"]), offsets, dest, src_row, xp, ws)
    assert ops.moe_get_device_error(ws) == 0
    assert np.array_equal(host(offsets), ref["offsets"])
    assert np.array_equal(host(dest), ref["dest"])
    assert np.array_equal(host(src_row), ref["src_row"])
    tok = torch.from_numpy((ref["src_row"] // K).astype(np.int64)).cuda()
    assert torch.equal(xp, xd[tok])
