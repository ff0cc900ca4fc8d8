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


CFG8 = dict(T=192, H=256, E=16, n_group=4, topk_group=2, topk=4, I=128,
            I_shared=128, router_sigma=0.05)


def _mx(w, lo=0, hi=None):
    """Device E4M3 / power-of-two weights of experts [lo, hi) (and, with
    lo = None, the shared expert as one expert)."""
    if lo is None:
        t = [dev(w[n])[None] for n in ("ws1", "ws3", "ws2")]
    else:
        E = w["w1"].shape[0]
        hi = E if hi is None else hi
        t = [dev(w[n][lo:hi]) for n in ("w1", "w3", "w2")]
    full = ops.WeightsMx.quantize(t[0], t[1], t[2], dev(w["ws1"]),
                                  dev(w["ws3"]), dev(w["ws2"]))
    return ops.WeightsMx(**{n: full.pairs[n] for n in ("w1", "w3", "w2")})


def _worker_mx(rank, world, port, q):
    try:
        import sys
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        sys.path.insert(0, root)
        os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
        torch.cuda.set_device(0)
        dist.init_process_group("gloo", rank=rank, world_size=world)
        from deepseekmoe_routing_expert_moe_b300 import ep
        cfg = inputs.custom_config("ep_gpu8", 911, **CFG8)
        w = inputs.layer_inputs(cfg)
        El = cfg.E // world
        n = cfg.T // world
        d = ops.dims_of(cfg, T=n)
        be = ep.CudaBackend(d, _weights(w), _weights(w, rank * El,
                                                     (rank + 1) * El),
                            rank, world,
                            mx=(_mx(w, rank * El, (rank + 1) * El),
                                _mx(w, None)))
        layer = ep.ExpertParallel(be, cfg.E, cfg.topk, cfg.topk_group,
                                  cfg.n_group)
        out = layer.forward(dev(w["x"][rank * n:(rank + 1) * n]),
                            dev(w["bias"]), update_bias=False)
        torch.cuda.synchronize()
        q.put((rank, host(out, np.uint16), host(layer.last["idx"]), None))
        dist.destroy_process_group()
    except Exception as e:  # noqa: BLE001 -- reported to the parent
        q.put((rank, None, None, repr(e)))


def test_expert_parallel_fp8_dispatch_equals_single_gpu_fp8_layer():
    """Dispatch in FP8 ("02 · DeepSeek-V3" §2): each rank quantizes its
    tokens once (power-of-two scales), sends E4M3 codes and scale bytes,
    the owners run their experts on them (moe_expert_ffn_mx_routed) and
    return bf16 rows.  Every rank's output must equal, bit for bit, the
    single-GPU layer on its shard through the public FP8 calls
    (moe_permute_mx, moe_expert_ffn_mx with all experts and the shared one,
    moe_combine)."""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker_mx, args=(r, world, port, q))
          for r in range(world)]
    for p in ps:
        p.start()
    res = sorted([q.get(timeout=300) for _ in range(world)],
                 key=lambda v: v[0])
    for p in ps:
        p.join(timeout=60)
    for r in res:
        assert r[3] is None, r[3]
    cfg = inputs.custom_config("ep_gpu8", 911, **CFG8)
    w = inputs.layer_inputs(cfg)
    n, K, E, H = cfg.T // world, cfg.topk, cfg.E, cfg.H
    d = ops.dims_of(cfg, T=n)
    W = _weights(w)
    Wq = ops.WeightsMx.quantize(dev(w["w1"]), dev(w["w3"]), dev(w["w2"]),
                                dev(w["ws1"]), dev(w["ws3"]), dev(w["ws2"]))
    ws = ops.workspace(d, ops.MOE_WS_FORWARD)
    for rank, o, i, _ in res:
        x = dev(w["x"][rank * n:(rank + 1) * n])
        z = torch.zeros((n, E), dtype=torch.float32, device="cuda")
        idx = torch.zeros((n, K), dtype=torch.int32, device="cuda")
        gate = torch.zeros((n, K), dtype=torch.float32, device="cuda")
        counts = torch.zeros(E, dtype=torch.int32, device="cuda")
        off = torch.zeros(E + 1, dtype=torch.int32, device="cuda")
        dest = torch.zeros((n, K), dtype=torch.int32, device="cuda")
        src = torch.zeros(n * K, dtype=torch.int32, device="cuda")
        u8 = dict(dtype=torch.uint8, device="cuda")
        xq, xs = torch.zeros((n, H), **u8), torch.zeros((n, H // 128), **u8)
        xpq = torch.zeros((n * K, H), **u8)
        xps = torch.zeros((n * K, H // 128), **u8)
        yp = torch.zeros((n * K, H), dtype=torch.int16, device="cuda")
        ys = torch.zeros((n, H), dtype=torch.int16, device="cuda")
        out = torch.zeros((n, H), dtype=torch.int16, device="cuda")
        ops.moe_router_logits(d, x, W.w_router, z, ws)
        ops.moe_route(d, z, dev(w["bias"]), idx, gate, counts, ws)
        ops.moe_permute(d, None, idx, off, dest, src, None, ws)
        ops.moe_permute_mx(d, x, dest, xq, xs, xpq, xps, ws)
        ops.moe_expert_ffn_mx(d, Wq, xpq, xps, xq, xs, off, yp, ys, ws)
        ops.moe_combine(d, x, ys, yp, dest, gate, out)
        assert ops.moe_get_device_error(ws) == 0
        assert np.array_equal(i, host(idx))
        assert np.array_equal(o, host(out, np.uint16))


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


@pytest.mark.parametrize("P,El,H", [(2, 8, 320), (4, 3, 320), (8, 32, 320),
                                    (1, 5, 320), (4, 6, 28), (3, 4, 1)])
def test_regroup_matches_numpy_and_inverts(P, El, H):
    """Rows of 640 bytes (bf16 rows: 16-byte vectors), of 56 bytes (the
    scale bytes of 7168-wide E4M3 rows: 4-byte words) and of 2 bytes."""
    rng = np.random.default_rng(P * 100 + El)
    counts = rng.integers(0, 40, size=(P, El)).astype(np.int32)
    counts[0, 0] = 0
    R = int(counts.sum())
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
    # the map itself, index for index, against the oracle's
    operm, ooff = O.ep_plan(counts)
    assert np.array_equal(host(perm), operm)
    assert np.array_equal(host(off), ooff)
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
