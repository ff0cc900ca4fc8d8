"""The standalone combine call (moe_combine, eq. 12 of "02 · DeepSeek-V3"
§1.3: out = x + shared expert + gate-weighted routed experts) against
``oracle.moe_output``.

Inputs are the oracle's: gates from its routing of seeded logits, the
dispatch rows from its permutation, and seeded bf16 rows standing in for
the expert outputs yp and ys.  The kernel sums in fp32 (x + ys, then one
multiply-add per slot in slot order) and rounds once to bf16, so per
element
    |out - ref| <= u_bf16 (|ref| + a) + a,   a = (K + 2) 2^-24 S,
with S = |x| + |ys| + sum_k |g_k y_k| (the fp32 accumulation allowance) and
u_bf16 = 2^-8 (round to nearest).  A slot whose dest row is invalid adds
nothing and its row is never read (a NaN planted there must not appear)."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import U_BF16, bf16_dev_to_f32, dev

pytestmark = pytest.mark.gpu

f32 = inputs.bf16_bits_to_f32


def _rows(cfg, tid, shape, sigma):
    key = (cfg.config_id * 7919 + tid) & 0xFFFFFFFF
    return inputs.normal_bf16(key, shape, sigma)


def _inputs(cfg, T):
    z = inputs.random_logits(cfg, T=T)
    r = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group, cfg.topk)
    p = O.permutation(r["idx"], cfg.E)
    x = inputs.x_tokens(cfg, T=T)
    ys = _rows(cfg, 1, (T, cfg.H), 0.5)
    yp = _rows(cfg, 2, (T * cfg.topk, cfg.H), 0.5)
    return x, ys, yp, p["dest"], r["gate"]


def _bound_check(got, x, ys, yp, dest, gate):
    """Element bound of the module docstring; dest < 0 or >= rows: slot
    skipped on both sides."""
    T, K = dest.shape
    X, S, Y = (f32(a).astype(np.float64) for a in (x, ys, yp))
    valid = (dest >= 0) & (dest < Y.shape[0])
    y_slots = np.where(valid[:, :, None], Y[np.where(valid, dest, 0)], 0.0)
    g = np.where(valid, gate, 0.0)
    ref = O.moe_output(X, S, y_slots, g)
    acc = np.abs(X) + np.abs(S) + np.einsum(
        "tk,tkh->th", np.abs(g), np.abs(y_slots))
    a = (K + 2) * 2.0 ** -24 * acc
    bound = U_BF16 * (np.abs(ref) + a) + a + 1e-30
    got = np.asarray(got, np.float64)
    assert np.isfinite(got).all()
    ratio = np.abs(got - ref) / bound
    assert ratio.max() <= 1.0, ratio.max()
    # and it is not trivially loose: the rounding alone reaches a good part
    assert ratio.max() > 0.05
    return ratio.max()


def _combine(cfg, T, x, ys, yp, dest, gate):
    d = ops.dims_of(cfg, T=T)
    out = torch.full((T, cfg.H), 0x7FC0, dtype=torch.int16, device="cuda")
    ops.moe_combine(d, dev(x), dev(ys), dev(yp), dev(dest), dev(gate), out)
    torch.cuda.synchronize()
    return bf16_dev_to_f32(out)


CASES = {
    "tiny": (inputs.CONFIGS["tiny"], 64),
    "one_token": (inputs.CONFIGS["prefill_v3"], 1),
    "ragged": (inputs.custom_config("comb_r", 700, T=77, H=320, E=32,
                                    n_group=4, topk_group=2, topk=6, I=64,
                                    I_shared=64), 77),
    "top12": (inputs.custom_config("comb_k", 701, T=50, H=256, E=64,
                                   n_group=8, topk_group=4, topk=12, I=64,
                                   I_shared=64), 50),
    "prefill_v3": (inputs.CONFIGS["prefill_v3"], 4096),
}


@pytest.mark.parametrize("case", sorted(CASES))
def test_combine_matches_oracle_output(case):
    """Every element of every token; top12 takes the kernel's path for
    more than 8 slots, prefill_v3 the full V3 size (4096 x 7168, top-8)."""
    cfg, T = CASES[case]
    x, ys, yp, dest, gate = _inputs(cfg, T)
    got = _combine(cfg, T, x, ys, yp, dest, gate)
    _bound_check(got, x, ys, yp, dest, gate)


def test_combine_skips_invalid_slots_without_reading_them():
    """dest = -1 (what moe_permute writes for an invalid expert id) and a
    row past the end add nothing; yp row 0, which no valid slot uses, is
    NaN and must not leak into any token."""
    cfg = inputs.custom_config("comb_bad", 702, T=40, H=256, E=16, n_group=4,
                               topk_group=2, topk=4, I=64, I_shared=64)
    T, K = cfg.T, cfg.topk
    rng = np.random.default_rng(11)
    x, ys, yp, _, gate = _inputs(cfg, T)
    dest = np.empty(T * K, np.int32)
    dest[:] = rng.permutation(np.arange(1, T * K + 1))[:T * K]
    dest[dest == T * K] = 1    # keep every valid row in range
    dest = dest.reshape(T, K)
    dest[3, 0] = -1
    dest[17, 2] = -1
    dest[25, 3] = T * K        # one past the end
    dest[39, 1] = 2 ** 30
    yp = yp.copy()
    yp[0, :] = 0x7FC0          # bf16 NaN
    got = _combine(cfg, T, x, ys, yp, dest, gate)
    _bound_check(got, x, ys, yp, dest, gate)
