"""FP8 (E4M3) quantization on the GPU against the oracle, bit for bit
("02 · DeepSeek-V3" §2: 1 x 128 activation tiles, 128 x 128 weight
blocks, scales from the online max |value|).  Codes are integers decided
by floating point; both sides decide them on the same fp32 quotient, so
codes and scales must match exactly."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu

f32 = inputs.bf16_bits_to_f32


def rows_gpu(xb):
    R, C = xb.shape
    q = torch.full((R, C), 0x5A, dtype=torch.uint8, device="cuda")
    s = torch.full((R, C // 128), -7.0, dtype=torch.float32, device="cuda")
    ops.moe_quantize_fp8_rows(dev(xb), q, s)
    return host(q), host(s)


def blocks_gpu(wb_dev, R, C):
    q = torch.full((R, C), 0x5A, dtype=torch.uint8, device="cuda")
    s = torch.full((R // 128, C // 128), -7.0, dtype=torch.float32,
                   device="cuda")
    ops.moe_quantize_fp8_blocks(wb_dev, q, s)
    return q, s


def test_token_rows_prefill_batch():
    """The 4096 prefill tokens (H = 7168: 56 tiles per token)."""
    cfg = inputs.CONFIGS["prefill_v3"]
    xb = inputs.x_tokens(cfg)
    q, s = rows_gpu(xb)
    rq, rs = O.quantize_1x128(f32(xb))
    np.testing.assert_array_equal(s, rs)
    np.testing.assert_array_equal(q, rq)


@pytest.mark.parametrize("R,C", [(1, 128), (37, 384), (300, 1024)])
def test_ragged_rows_and_widths(R, C):
    g = np.random.default_rng(R + C)
    x = (g.standard_normal((R, C)) * np.exp(g.uniform(-12, 12, (R, 1))))
    xb = inputs.f32_to_bf16_bits(x.astype(np.float32))
    q, s = rows_gpu(xb)
    rq, rs = O.quantize_1x128(f32(xb))
    np.testing.assert_array_equal(s, rs)
    np.testing.assert_array_equal(q, rq)


def test_exact_ties_subnormals_signed_zero_and_zero_tiles():
    """Tile 0: 448 (so s = 1 exactly) and every midpoint between adjacent
    E4M3 values, positive and negative -- ties go to the even code.
    Tile 1: tiny values in the subnormal range of their scale, with -0.
    Tile 2: all zeros (scale 1, codes 0).  Tile 3: -0 and one value."""
    t = O.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = (t[:-1] + t[1:]) / 2
    x = np.zeros((2, 512), np.float32)
    x[0, 0] = 448.0
    x[0, 1:127] = mids[:126]
    x[1, 0] = -448.0
    x[1, 1:127] = -mids[:126]
    x[:, 128] = 1000.0
    x[:, 129:200] = np.linspace(-0.9, 0.9, 71)
    x[:, 200] = -0.0
    x[:, 384] = -0.0
    x[:, 385] = 3.0
    xb = inputs.f32_to_bf16_bits(x)
    assert np.array_equal(f32(xb)[:, :128], x[:, :128])   # midpoints exact
    q, s = rows_gpu(xb)
    rq, rs = O.quantize_1x128(f32(xb))
    np.testing.assert_array_equal(s, rs)
    np.testing.assert_array_equal(q, rq)
    assert s[0, 0] == 1.0 and s[0, 2] == 1.0 and np.all(q[:, 256:384] == 0)


def test_expert_weight_blocks_full_tensor_sampled():
    """W1 of all 256 experts as one [E*I, H] tensor (3.7 G values) on the
    GPU; the blocks of three experts checked against the oracle."""
    cfg = inputs.CONFIGS["prefill_v3"]
    E, I, H = cfg.E, cfg.I, cfg.H
    W1 = torch.empty((E, I, H), dtype=torch.int16, device="cuda")
    for e in range(E):
        W1[e] = inputs.expert_matrix(cfg, "w1", e, "cuda")
    q, s = blocks_gpu(W1.view(E * I, H), E * I, H)
    del W1
    for e in (0, 97, 255):
        w1 = inputs.expert_matrix(cfg, "w1", e)
        rq, rs = O.quantize_128x128(f32(w1))
        np.testing.assert_array_equal(host(s[e * I // 128:(e + 1) * I // 128]),
                                      rs)
        np.testing.assert_array_equal(host(q[e * I:(e + 1) * I]), rq)


def test_weight_blocks_with_outliers_and_zero_block():
    g = np.random.default_rng(9)
    w = (g.standard_normal((256, 384)) * 0.02).astype(np.float32)
    w[3, 7] = 50.0
    w[128:256, 128:256] = 0.0
    wb = inputs.f32_to_bf16_bits(w)
    q, s = blocks_gpu(dev(wb), 256, 384)
    rq, rs = O.quantize_128x128(f32(wb))
    np.testing.assert_array_equal(host(s), rs)
    np.testing.assert_array_equal(host(q), rq)
    assert host(s)[1, 1] == 1.0


def test_quantise_on_permute_matches_oracle_rows():
    """x quantized once per token; the expert-sorted rows are the token's
    codes and scales copied to dest[t, k]."""
    cfg = inputs.CONFIGS["prefill_v3"]
    T, H, K, E = 1024, cfg.H, cfg.topk, cfg.E
    d = ops.dims_of(cfg, T=T)
    xb = inputs.x_tokens(cfg, T=T)
    z = inputs.random_logits(cfg, T=T, step=3)
    idx = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group, K)["idx"]
    p = O.permutation(idx, E)
    xq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    xs = torch.empty((T, H // 128), dtype=torch.float32, device="cuda")
    xpq = torch.full((T * K, H), 0x5A, dtype=torch.uint8, device="cuda")
    xps = torch.full((T * K, H // 128), -7.0, dtype=torch.float32,
                     device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_PERMUTE)
    ops.moe_permute_fp8(d, dev(xb), dev(p["dest"]), xq, xs, xpq, xps, ws)
    assert ops.moe_get_device_error(ws) == 0
    rq, rs = O.quantize_1x128(f32(xb))
    np.testing.assert_array_equal(host(xq), rq)
    np.testing.assert_array_equal(host(xs), rs)
    tok = p["src_row"] // K
    np.testing.assert_array_equal(host(xpq), rq[tok])
    np.testing.assert_array_equal(host(xps), rs[tok])


def test_permute_fp8_bad_dest_is_reported_and_skipped():
    cfg = inputs.CONFIGS["tiny"]
    d = ops.dims_of(cfg, H=128)
    T, K, H = cfg.T, cfg.topk, 128
    dest = np.arange(T * K, dtype=np.int32).reshape(T, K)
    dest[5, 1] = T * K + 3                     # out of range
    xb = inputs.f32_to_bf16_bits(
        np.random.default_rng(1).standard_normal((T, H)).astype(np.float32))
    xq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    xs = torch.empty((T, 1), dtype=torch.float32, device="cuda")
    xpq = torch.zeros((T * K, H), dtype=torch.uint8, device="cuda")
    xps = torch.zeros((T * K, 1), dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_PERMUTE)
    ops.moe_permute_fp8(d, dev(xb), dev(dest), xq, xs, xpq, xps, ws)
    assert ops.moe_get_device_error(ws) == ops.STATUS_CODES[
        "MOE_ERR_DEVICE_BOUNDS"]
    rq, _ = O.quantize_1x128(f32(xb))
    got = host(xpq)
    np.testing.assert_array_equal(got[dest[5, 0]], rq[5])
    assert np.all(got[5 * K + 1] == 0)         # the skipped slot's row
