"""BF16 expert FFNs at the full V3 size, whole expert segments against the
oracle's fp64 SwiGLU ("02 · DeepSeek-V3" §1.1: 256 routed experts of 7168 ->
2048 -> 7168 plus the shared expert, top-8 routing of §1.3).

The routed rows, their order and the segment table come from the oracle's
own routing and permutation of the seeded tokens; the weights are the
device-generated V3 weights (the same bits the host generator gives, see
test_gpu_layer.py), so every compared expert is regenerated on the host.
Compared element by element, with the bound of ``ffn_bound_check`` (bf16
rounding of h and y, fp32 accumulation):

* the two busiest experts' whole segments -- at the skewed T = 32768 batch
  these hold thousands of rows and run the tensor-bound pipeline shape
  (256-row chunks) over the full K = 7168 / 2048 loops;
* the smallest non-empty segment (one row when there is one);
* a strided sample of the shared expert's rows (its segment is all T);
* the intermediate h = silu(p) * q of the busiest expert, read from the
  workspace, within its own bf16 rounding plus fp32 accumulation noise."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import U_BF16, bf16_dev_to_f32, dev, ffn_bound_check

pytestmark = pytest.mark.gpu

f32 = inputs.bf16_bits_to_f32


def _h_check(h_gpu, a, w1, w3):
    """|h - m| <= 1.01 u |m| + |dm/dp| e_p + |dm/dq| e_q, with m = silu(p) q
    in fp64 and e = 64 * 2^-24 * sum_h |a_h w_h| the fp32 accumulation
    allowance of p and q (the tensor cores sum 7168 products in fp32)."""
    a = np.asarray(a, np.float64)
    w1 = np.asarray(w1, np.float64)
    w3 = np.asarray(w3, np.float64)
    p = a @ w1.T
    q = a @ w3.T
    sg = 1.0 / (1.0 + np.exp(-p))
    m = p * sg * q
    aa = np.abs(a)
    e_p = 64 * 2.0 ** -24 * (aa @ np.abs(w1).T)
    e_q = 64 * 2.0 ** -24 * (aa @ np.abs(w3).T)
    dsilu = sg * (1.0 + p * (1.0 - sg))
    bound = 1.01 * U_BF16 * np.abs(m) + np.abs(dsilu * q) * e_p + \
        np.abs(p * sg) * e_q + 1e-30
    ratio = np.abs(np.asarray(h_gpu, np.float64) - m) / bound
    assert np.isfinite(h_gpu).all()
    assert ratio.max() <= 1.0, ratio.max()
    return ratio.max()


@pytest.mark.parametrize("name", ["prefill_v3", "skewed_v3"])
def test_v3_full_size_whole_segments(name, v3_weights):
    cfg = inputs.CONFIGS[name]
    T, K, E, H, I = cfg.T, cfg.topk, cfg.E, cfg.H, cfg.I
    d = ops.dims_of(cfg)
    x = inputs.x_tokens(cfg)
    xf = f32(x)
    pref = inputs.zipf_preference(cfg) if cfg.zipf_s > 0 else None
    z = O.router_logits(xf, inputs.router_weight(cfg), pref)
    r = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group, K)
    p = O.permutation(r["idx"], E)
    del z
    tok = p["src_row"] // K
    xd = dev(x)
    xp = xd[torch.from_numpy(tok.astype(np.int64)).cuda()]
    yp = torch.zeros((T * K, H), dtype=torch.int16, device="cuda")
    ys = torch.zeros((T, H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_FFN)
    ops.moe_expert_ffn(d, v3_weights, xp, xd, dev(p["offsets"]), yp, ys, ws)
    assert ops.moe_get_device_error(ws) == 0
    del xp
    off = p["offsets"]
    counts = np.diff(off)
    busy = np.argsort(-counts, kind="stable")[:2].tolist()
    nz = np.nonzero(counts)[0]
    small = int(nz[np.argmin(counts[nz])])
    if name == "skewed_v3":
        # the hot experts run the tensor-bound shape: chunks of up to 256 rows
        assert counts[busy[0]] > 2048 and T * K // E >= 256
    for e in busy + [small]:
        a, b = int(off[e]), int(off[e + 1])
        w1, w3, w2 = (f32(m) for m in inputs.expert_weights(cfg, e))
        got = bf16_dev_to_f32(yp[a:b])
        assert np.isfinite(got).all()
        ffn_bound_check(got, xf[tok[a:b]], w1, w3, w2)
        if e == busy[0]:
            hb = ws[256:256 + T * K * I * 2].view(torch.int16).view(T * K, I)
            _h_check(bf16_dev_to_f32(hb[a:b]), xf[tok[a:b]], w1, w3)
    rows = np.arange(0, T, max(1, T // 48))
    s1, s3, s2 = (f32(m) for m in inputs.shared_weights(cfg))
    got = bf16_dev_to_f32(ys)[rows]
    ffn_bound_check(got, xf[rows], s1, s3, s2)
    # every routed and shared output is finite
    assert bool(torch.isfinite(yp.view(torch.bfloat16)).all())
    assert bool(torch.isfinite(ys.view(torch.bfloat16)).all())
