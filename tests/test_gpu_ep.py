"""Expert parallelism through the library's kernels ("02 · DeepSeek-V3"
§5.1: experts partitioned over devices; §1.3 node-limited routing; §2
dispatch / combine).

Two ranks share this one GPU as two processes (the exchanges go through
host memory over gloo; no kernel of one rank waits on the other's).  Each
rank holds half of the routed experts, routes its half of the batch, sends
its rows to the experts' rank, runs its experts as one grouped GEMM over the
rows it received (moe_ep_plan / moe_ep_permute_rows regroup them), returns
the outputs and combines.  Per row the expert GEMMs accumulate in the same
order whichever rows share a tile, so every rank's output must equal the
single-GPU moe_forward of its shard bit for bit, the bias step on the
all-reduced load must equal the whole batch's, and the outputs must match
the oracle within the layer tolerance on margin tokens.  The regroup kernels alone are
checked against a numpy reference on ragged counts."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from deepseekmoe_routing_expert_moe_b300 import inputs, ops
from oracle import moe_oracle as O

from gpu_helpers import dev, host, rms_tolerance_check

pytestmark = pytest.mark.gpu

CFG = dict(T=192, H=256, E=16, n_group=4, topk_group=2, topk=4, I=128,
           I_shared=64, router_sigma=0.05)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _cfg():
    return inputs.custom_config("ep_gpu", 910, **CFG)


def _weights(w, lo=0, hi=None):
    E = w["w1"].shape[0]
    hi = E if hi is None else hi
    return ops.Weights(dev(w["w_router"]), dev(w["w1"][lo:hi]),
                       dev(w["w3"][lo:hi]), dev(w["w2"][lo:hi]),
                       dev(w["ws1"]), dev(w["ws3"]), dev(w["ws2"]))


def _worker(rank, world, port, q):
    try:
        import sys
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        sys.path.insert(0, root)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        torch.cuda.set_device(0)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        from deepseekmoe_routing_expert_moe_b300 import ep
        cfg = _cfg()
        w = inputs.layer_inputs(cfg)
        El = cfg.E // world
        n = cfg.T // world
        d = ops.dims_of(cfg, T=n)
        be = ep.CudaBackend(d, _weights(w), _weights(w, rank * El,
                                                     (rank + 1) * El),
                            rank, world)
        layer = ep.ExpertParallel(be, cfg.E, cfg.topk, cfg.topk_group,
                                  cfg.n_group)
        x = dev(w["x"][rank * n:(rank + 1) * n])
        bias = dev(w["bias"])
        out = layer.forward(x, bias, update_bias=True)
        torch.cuda.synchronize()
        q.put((rank, host(out, np.uint16), host(bias),
               host(layer.last["idx"]), None))
        dist.destroy_process_group()
    except Exception as e:  # noqa: BLE001 -- reported to the parent
        q.put((rank, None, None, None, repr(e)))


def test_expert_parallel_two_ranks_equal_single_gpu_forward():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, world, port, q))
          for r in range(world)]
    for p in ps:
        p.start()
    res = sorted([q.get(timeout=300) for _ in range(world)],
                 key=lambda v: v[0])
    for p in ps:
        p.join(timeout=60)
    for r in res:
        assert r[4] is None, r[4]
    assert all(p.exitcode == 0 for p in ps)

    cfg = _cfg()
    w = inputs.layer_inputs(cfg)
    n = cfg.T // world
    d = ops.dims_of(cfg, T=n)
    ws = ops.workspace(d, ops.MOE_WS_FORWARD)
    idx_all = []
    for rank, o, b, i, _ in res:
        # the single-GPU layer on the same shard (same router tiles, so the
        # same logits), no bias step
        out = torch.zeros((n, cfg.H), dtype=torch.int16, device="cuda")
        idx = torch.zeros((n, cfg.topk), dtype=torch.int32, device="cuda")
        ops.moe_forward(d, _weights(w), dev(w["x"][rank * n:(rank + 1) * n]),
                        dev(w["bias"]), out, ws, update_bias=False,
                        topk_idx_out=idx)
        assert ops.moe_get_device_error(ws) == 0
        assert np.array_equal(i, host(idx))
        assert np.array_equal(o, host(out, np.uint16))
        idx_all.append(i)
    # the bias step on the all-reduced load equals the whole batch's
    c = O.expert_counts(np.concatenate(idx_all), cfg.E)
    nb, _ = O.bias_update(c, w["bias"], cfg.T, cfg.topk, cfg.gamma)
    for r in res:
        assert np.array_equal(r[2].view(np.uint32), nb.view(np.uint32))
    # and against the oracle on margin tokens
    f = inputs.bf16_bits_to_f32
    ref = O.layer_forward(f(w["x"]), w["w_router"], w["bias"], f(w["w1"]),
                          f(w["w3"]), f(w["w2"]), f(w["ws1"]), f(w["ws3"]),
                          f(w["ws2"]), n_group=cfg.n_group,
                          topk_group=cfg.topk_group, topk=cfg.topk)
    km, gm = O.routing_margins(ref["route"], cfg.topk_group, cfg.topk)
    ok = (km > 1e-4) & (gm > 1e-4)
    got = f(np.concatenate([r[1] for r in res]))
    rms_tolerance_check(got, ref["out"], rows=ok)


def _np_regroup(counts, rows_src):
    """Expert-major order of source-major rows (numpy reference)."""
    P, El = counts.shape
    blocks = {}
    a = 0
    for s in range(P):
        for l in range(El):
            blocks[(s, l)] = rows_src[a:a + counts[s, l]]
            a += counts[s, l]
    out = [blocks[(s, l)] for l in range(El) for s in range(P)]
    off = np.concatenate([[0], np.cumsum([counts[:, l].sum()
                                          for l in range(El)])])
    return np.concatenate(out), off


@pytest.mark.parametrize("P,El", [(2, 8), (4, 3), (8, 32), (1, 5)])
def test_regroup_matches_numpy_and_inverts(P, El):
    rng = np.random.default_rng(P * 100 + El)
    counts = rng.integers(0, 40, size=(P, El)).astype(np.int32)
    counts[0, 0] = 0
    R = int(counts.sum())
    H = 320
    rows = rng.integers(-30000, 30000, size=(R, H)).astype(np.int16)
    perm = torch.full((R,), -1, dtype=torch.int32, device="cuda")
    off = torch.full((El + 1,), -1, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ops.moe_ep_plan(dev(counts), R, perm, off, ws=ws)
    xr = torch.empty((R, H), dtype=torch.int16, device="cuda")
    ops.moe_ep_permute_rows(dev(rows), perm, xr, inverse=False, ws=ws)
    back = torch.empty_like(xr)
    ops.moe_ep_permute_rows(xr, perm, back, inverse=True, ws=ws)
    assert ops.moe_get_device_error(ws) == 0
    want, want_off = _np_regroup(counts, rows)
    assert np.array_equal(host(off), want_off)
    assert np.array_equal(host(xr), want)
    assert np.array_equal(host(back), rows)


def test_plan_reports_inconsistent_row_counts():
    counts = np.array([[3, 4], [5, 6]], np.int32)
    perm = torch.empty(20, dtype=torch.int32, device="cuda")
    off = torch.empty(3, dtype=torch.int32, device="cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    ops.moe_ep_plan(dev(counts), 20, perm, off, ws=ws)   # counts sum to 18
    assert ops.moe_get_device_error(ws) == ops.STATUS_CODES[
        "MOE_ERR_DEVICE_BOUNDS"]
    p = host(perm)
    assert sorted(p[:18].tolist()) == list(range(18))
    assert p[18:].tolist() == [18, 19]
