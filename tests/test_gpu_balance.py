"""Sequence-wise balance loss on the GPU against the oracle ("02 ·
DeepSeek-V3" §1.4, eq. 17-20), given the same logits.

The per-sequence top-K counts are integers decided on the bit-exact fp32
sigmoid: compared exactly.  P and the loss are fp32 sums of positive terms
whose rounding is bounded by the kernel's fixed order (u = 2^-24):
  s'   = s * (1/den), den summed in (EPL - 1) lane-local adds + 5
         butterfly adds, one reciprocal, one multiply
                                              -> <= (EPL + 7) u relative
  P    = the sequence cut into rs row splits, each into 32 ranges:
         ceil(T_s/(32 rs)) adds in a range, 31 across ranges, rs - 1
         across splits, one division; the split rule (rs <= ceil(S/256))
         keeps this          -> <= (ceil(S/32) + 33) u more
  loss = f (2 roundings) times P (1), 5 butterfly + up to 31 warp adds,
         times alpha (1)                      -> <= 40 u more
so P is checked to (EPL + ceil(S/32) + 40) u and the loss to that + 40 u,
relative to the oracle's fp64 values (S = min(seq_len, T))."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import dev, host

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


def balance_gpu(d, z, seq_len, alpha):
    n_seq = -(-d.T // seq_len)
    counts = torch.full((n_seq, d.E), -7, dtype=torch.int32, device="cuda")
    P = torch.full((n_seq, d.E), -7.0, dtype=torch.float32, device="cuda")
    loss = torch.full((n_seq,), -7.0, dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_SEQ_BALANCE)
    ops.moe_seq_balance_loss(d, dev(z), seq_len, alpha, counts, P, loss, ws)
    assert ops.moe_get_device_error(ws) == 0
    return host(counts), host(P), host(loss)


def assert_balance_matches(d, z, seq_len, alpha=1e-4):
    r = O.seq_balance_loss(z, seq_len, d.topk, alpha)
    counts, P, loss = balance_gpu(d, z, seq_len, alpha)
    np.testing.assert_array_equal(counts, r["counts"])
    epl = max(1, d.E // 32)
    per = -(-min(seq_len, d.T) // 32)
    tol_p = (epl + per + 40) * U
    np.testing.assert_allclose(P.astype(np.float64), r["P"], rtol=tol_p,
                               atol=0)
    np.testing.assert_allclose(loss.astype(np.float64), r["loss"],
                               rtol=tol_p + 40 * U, atol=0)
    return r


def _dims(E, K, T):
    # the groups play no part in this loss: one group keeps every expert
    cfg = inputs.custom_config("balance", 500 + E + K, T=T, H=64, E=E,
                               n_group=1, topk_group=1, topk=K, I=64,
                               I_shared=64)
    return cfg, ops.dims_of(cfg)


def test_v3_one_4k_sequence():
    """V3: 256 experts, top-8, one 4096-token sequence."""
    cfg = inputs.CONFIGS["prefill_v3"]
    d = ops.dims_of(cfg)
    z = inputs.random_logits(cfg, scale=0.5)
    r = assert_balance_matches(d, z, seq_len=4096)
    assert r["loss"].shape == (1,) and 0.9e-4 < r["loss"][0] < 1.5e-4


def test_v3_logits_from_the_router():
    """Logits of the layer's own router on the prefill tokens."""
    cfg = inputs.CONFIGS["prefill_v3"]
    d = ops.dims_of(cfg, T=1024)
    z = O.router_logits(inputs.bf16_bits_to_f32(inputs.x_tokens(cfg, T=1024)),
                        inputs.router_weight(cfg))
    assert_balance_matches(d, z, seq_len=512)


@pytest.mark.parametrize("T,seq_len", [(4096, 1000), (777, 1), (500, 10 ** 6),
                                       (4097, 64), (1, 1), (65, 33)])
def test_ragged_and_degenerate_sequence_cuts(T, seq_len):
    cfg = inputs.CONFIGS["prefill_v3"]
    d = ops.dims_of(cfg, T=T)
    z = inputs.random_logits(cfg, T=T, step=T + seq_len)
    assert_balance_matches(d, z, seq_len)


@pytest.mark.parametrize("E,K", [(16, 4), (8, 2), (32, 32), (64, 6),
                                 (512, 16), (1024, 8), (256, 1)])
def test_expert_shapes(E, K):
    cfg, d = _dims(E, K, T=700)
    z = inputs.random_logits(cfg, scale=1.0)
    r = assert_balance_matches(d, z, seq_len=128, alpha=3e-3)
    if K == E:                               # every expert chosen by all
        assert np.all(r["counts"] == np.array([128] * 5 + [60])[:, None])


def test_exact_ties_break_to_the_lower_index():
    """Logits on a coarse grid: many equal affinities inside a token."""
    cfg = inputs.CONFIGS["prefill_v3"]
    d = ops.dims_of(cfg, T=2048)
    z = (np.round(inputs.random_logits(cfg, T=2048, step=5) * 4) / 4).astype(
        np.float32)
    assert_balance_matches(d, z, seq_len=256)


def test_skewed_batch_eight_sequences():
    """The skewed-load batch shape: 32768 tokens as eight 4096-token
    sequences, logits with a Zipf per-expert preference added."""
    cfg = inputs.CONFIGS["skewed_v3"]
    d = ops.dims_of(cfg)
    z = (inputs.random_logits(cfg, scale=0.5) +
         inputs.zipf_preference(cfg)[None, :]).astype(np.float32)
    r = assert_balance_matches(d, z, seq_len=4096)
    assert r["loss"].shape == (8,) and np.all(r["loss"] > 1.02e-4)


def test_no_tokens_writes_nothing():
    cfg = inputs.CONFIGS["prefill_v3"]
    d = ops.dims_of(cfg, T=0)
    loss = torch.full((4,), -7.0, dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_SEQ_BALANCE)
    ops.moe_seq_balance_loss(d, None, 16, 1e-4, None, None, loss, ws)
    assert ops.moe_get_device_error(ws) == 0
    assert torch.all(loss == -7.0)
