"""Expert FFNs (grouped tcgen05 GEMMs, SwiGLU epilogue) against the oracle's
fp64 SwiGLU, on segments that span several 128-row tiles with ragged
tails, empty experts, one expert holding every row, and the tile-width
variants of the kernels."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import bf16_dev_to_f32, dev, ffn_bound_check

pytestmark = pytest.mark.gpu


def run_ffn(cfg, idx=None):
    d = ops.dims_of(cfg)
    T, K, H, E = cfg.T, cfg.topk, cfg.H, cfg.E
    x = inputs.x_tokens(cfg)
    if idx is None:
        z = O.router_logits(inputs.bf16_bits_to_f32(x), inputs.router_weight(cfg))
        idx = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group,
                      cfg.topk)["idx"]
    p = O.permutation(idx, E)
    xp = x[p["src_row"] // K]
    w = inputs.layer_inputs(cfg)
    W = ops.Weights(torch.zeros(E, H, dtype=torch.float32, device="cuda"),
                    dev(w["w1"]), dev(w["w3"]), dev(w["w2"]), dev(w["ws1"]),
                    dev(w["ws3"]), dev(w["ws2"]))
    yp = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
    ys = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN)
    ops.moe_expert_ffn(d, W, dev(xp), dev(x), dev(p["offsets"]), yp, ys, ws)
    assert ops.moe_get_device_error(ws) == 0
    f = inputs.bf16_bits_to_f32
    xs = f(x).astype(np.float64)
    ref_s = O.swiglu_ffn(xs, f(w["ws1"]), f(w["ws3"]), f(w["ws2"]))
    ref_p = np.zeros((T * K, H))
    for e in range(E):
        r0, r1 = p["offsets"][e], p["offsets"][e + 1]
        if r1 > r0:
            ref_p[r0:r1] = O.swiglu_ffn(xs[p["src_row"][r0:r1] // K],
                                        f(w["w1"][e]), f(w["w3"][e]),
                                        f(w["w2"][e]))
    gp, gs = bf16_dev_to_f32(yp), bf16_dev_to_f32(ys)
    # elementwise bound from the two bf16 roundings (h and y)
    e1 = ffn_bound_check(gs, xs, f(w["ws1"]), f(w["ws3"]), f(w["ws2"]))
    e2 = 0.0
    for e in range(E):
        r0, r1 = p["offsets"][e], p["offsets"][e + 1]
        if r1 > r0:
            e2 = max(e2, ffn_bound_check(gp[r0:r1], xs[p["src_row"][r0:r1] // K],
                                         f(w["w1"][e]), f(w["w3"][e]),
                                         f(w["w2"][e])))
    # and the typical error is far below the RMS of the result
    for g, r in ((gs, ref_s), (gp, ref_p)):
        assert np.sqrt(np.mean((g - r) ** 2)) <= 5e-3 * np.sqrt(np.mean(r * r))
    return p, e1, e2


def test_ffn_tiny_config():
    run_ffn(inputs.CONFIGS["tiny"])


def test_ffn_multi_tile_ragged_segments_wide_tiles():
    # I, I_s multiples of 128 -> 128-feature up tiles; H % 256 == 0
    cfg = inputs.custom_config("ffn_a", 500, T=700, H=512, E=8, n_group=4,
                               topk_group=2, topk=2, I=256, I_shared=128,
                               router_sigma=0.05)
    p, _, _ = run_ffn(cfg)
    c = np.diff(p["offsets"])
    assert c.max() > 128 and np.any(c % 128 != 0)


def test_ffn_narrow_tiles():
    # H % 128 != 0 -> 64-column down tiles; I % 128 != 0 -> 64-feature up
    cfg = inputs.custom_config("ffn_b", 501, T=300, H=192, E=4, n_group=2,
                               topk_group=1, topk=2, I=192, I_shared=64,
                               router_sigma=0.05)
    run_ffn(cfg)


def test_ffn_mid_width_down_tiles():
    cfg = inputs.custom_config("ffn_c", 502, T=257, H=384, E=16, n_group=4,
                               topk_group=2, topk=4, I=128, I_shared=192,
                               router_sigma=0.05)
    run_ffn(cfg)


def test_ffn_one_expert_takes_everything():
    cfg = inputs.custom_config("ffn_d", 503, T=600, H=256, E=32, n_group=4,
                               topk_group=2, topk=1, I=128, I_shared=128)
    idx = np.full((cfg.T, 1), 17, np.int32)
    p, _, _ = run_ffn(cfg, idx)
    assert np.diff(p["offsets"])[17] == 600


def mixed_load_idx(T, counts):
    """topk=2 routing with the given per-expert loads: the expert-sorted
    slot list is cut in two halves, token t takes slot t of each (distinct
    experts while every load is below T)."""
    flat = np.repeat(np.arange(len(counts), dtype=np.int32), counts)
    assert flat.size == 2 * T and max(counts) < T
    return np.stack([flat[:T], flat[T:]], axis=1)


# (T, per-expert loads) for 8 experts, topk 2.  The first set has a mean
# of 225 rows per expert (the HBM-streaming pipeline shape, chunks <= 192
# rows), the second 325 (the tensor-bound shape, chunks <= 256 rows).
MIXED_LOADS = {
    "stream": (900, [1, 17, 128, 129, 250, 256, 257, 762]),
    "compute": (1300, [1, 17, 128, 129, 256, 257, 600, 1212]),
}


@pytest.mark.parametrize("shape", sorted(MIXED_LOADS))
@pytest.mark.parametrize("ctas", [1, 3, 0])
def test_ffn_mixed_chunk_widths_and_tmem_slots(ctas, shape):
    # loads hit every unit shape: N=16, 32, 128 (one TMEM slot), 144..256
    # (both slots; 256 = two 128-row token boxes), segments cut into
    # several chunks, and the shared segment (all T rows) cut into equal
    # chunks.  With the grid capped, one CTA walks a mixed sequence of
    # one-slot and two-slot units.
    T, counts = MIXED_LOADS[shape]
    cfg = inputs.custom_config("ffn_mix_" + shape, 505, T=T, H=256, E=8,
                               n_group=4, topk_group=2, topk=2, I=256,
                               I_shared=192)
    try:
        ops.moe_set_gemm_ctas(ctas)
        p, _, _ = run_ffn(cfg, mixed_load_idx(T, counts))
    finally:
        ops.moe_set_gemm_ctas(0)
    assert list(np.diff(p["offsets"])) == counts


def test_ffn_single_token():
    cfg = inputs.custom_config("ffn_e", 504, T=1, H=256, E=16, n_group=4,
                               topk_group=2, topk=4, I=64, I_shared=64)
    run_ffn(cfg)


def test_ffn_bad_offsets_are_rejected_on_device():
    cfg = inputs.CONFIGS["tiny"]
    d = ops.dims_of(cfg)
    T, K, H, E = cfg.T, cfg.topk, cfg.H, cfg.E
    z = torch.zeros
    W = ops.Weights(z(E, H, dtype=torch.float32, device="cuda"),
                    *(z(s, dtype=torch.int16, device="cuda") for s in
                      ((E, cfg.I, H), (E, cfg.I, H), (E, H, cfg.I),
                       (cfg.I_shared, H), (cfg.I_shared, H), (H, cfg.I_shared))))
    off = np.arange(E + 1, dtype=np.int32) * 16
    off[5] = 10_000          # beyond T*K rows
    yp = z((T * K, H), dtype=torch.int16, device="cuda")
    ys = z((T, H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN)
    xp_in = z((T * K, H), dtype=torch.int16, device="cuda")
    x_in = z((T, H), dtype=torch.int16, device="cuda")
    ops.moe_expert_ffn(d, W, xp_in, x_in, dev(off), yp, ys, ws)
    assert ops.moe_get_device_error(ws) == ops.STATUS_CODES["MOE_ERR_DEVICE_BOUNDS"]


def test_ffn_large_magnitude_preactivations():
    """Weights ~ N(0, 16): the gate pre-activations p = W1 a reach several
    hundred in magnitude, so silu's far negative tail (p < -88, where
    e^-p overflows fp32) and its linear regime are both exercised.  The
    outputs stay finite and within the elementwise bound of the fp64
    SwiGLU."""
    cfg = inputs.custom_config("ffn_big", 506, T=200, H=256, E=8, n_group=4,
                               topk_group=2, topk=2, I=128, I_shared=128,
                               w_sigma=16.0, router_sigma=0.05)
    f = inputs.bf16_bits_to_f32
    x = f(inputs.x_tokens(cfg)).astype(np.float64)
    ws1 = f(inputs.shared_weights(cfg)[0]).astype(np.float64)
    pre = x @ ws1.T
    assert pre.min() < -200 and pre.max() > 200
    run_ffn(cfg)
