"""Expert parallelism on CPU: the exchange logic of ``ep.ExpertParallel``
over two gloo ranks ("02 · DeepSeek-V3" §1.3 node-limited routing, §2
dispatch / combine, §5.1 experts partitioned over devices).

Each rank holds half of the routed experts and routes its own half of the
batch.  The per-rank arithmetic is the oracle's (a numpy backend defined
here, rows carried as fp64), so this checks the orchestration alone: the
count exchange, the split sizes, the source-major to expert-major regroup
and back, the return trip and the combine.  Every rank's output must equal
the unsharded oracle layer on its tokens (fp64, only summation order may
differ), the rows each rank receives must be exactly the unsharded
permutation's rows of its experts, every token's rows must reach at most
topk_group groups, and the bias step on the all-reduced load must equal
the unsharded batch's bit for bit."""
import os
import socket

import numpy as np
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

CFG = dict(T=64, H=128, E=16, n_group=4, topk_group=2, topk=4, I=64,
           I_shared=64)
CFG8 = dict(T=64, H=256, E=16, n_group=4, topk_group=2, topk=4, I=128,
            I_shared=128)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


class NumpyBackend:
    """The oracle's arithmetic behind the backend interface of ep.py; rows
    travel as fp64 tensors."""

    def __init__(self, cfg, w, rank, world):
        from oracle import moe_oracle as O
        self.O, self.cfg, self.w = O, cfg, w
        self.El = cfg.E // world
        self.e0 = rank * self.El

    def route(self, x, bias):
        c, O = self.cfg, self.O
        z = O.router_logits(x.numpy(), self.w["w_router"])
        r = O.route(z, bias.numpy(), c.n_group, c.topk_group, c.topk)
        counts = O.expert_counts(r["idx"], c.E)
        return (torch.from_numpy(r["idx"]), torch.from_numpy(r["gate"]),
                torch.from_numpy(counts.astype(np.int32)))

    def permute(self, x, idx):
        p = self.O.permutation(idx.numpy(), self.cfg.E)
        xp = x.numpy()[p["src_row"] // self.cfg.topk]
        return (torch.from_numpy(p["offsets"]), torch.from_numpy(p["dest"]),
                torch.from_numpy(np.ascontiguousarray(xp)))

    def plan(self, recv_counts, rows):
        rc = recv_counts.numpy()
        P, El = rc.shape
        src_off = np.concatenate([[0], np.cumsum(rc.ravel())])
        exp_order = [(s, l) for l in range(El) for s in range(P)]
        exp_off = {}
        run = 0
        for s, l in exp_order:
            exp_off[(s, l)] = run
            run += rc[s, l]
        perm = np.empty(rows, np.int32)
        for s in range(P):
            for l in range(El):
                a = src_off[s * El + l]
                n = rc[s, l]
                perm[a:a + n] = exp_off[(s, l)] + np.arange(n)
        off = np.array([exp_off[(0, l)] for l in range(El)] + [rows], np.int32)
        return torch.from_numpy(perm), torch.from_numpy(off)

    def permute_rows(self, rows, perm, inverse):
        r, p = rows.numpy(), perm.numpy()
        out = np.empty_like(r)
        if inverse:
            out[:] = r[p]
        else:
            out[p] = r
        return torch.from_numpy(out)

    def experts(self, xr, offsets_local):
        O, w, off = self.O, self.w, offsets_local.numpy()
        xr = xr.numpy()
        y = np.zeros_like(xr)
        for l in range(self.El):
            e = self.e0 + l
            a, b = off[l], off[l + 1]
            if b > a:
                y[a:b] = O.swiglu_ffn(xr[a:b], w["w1"][e], w["w3"][e],
                                      w["w2"][e])
        return torch.from_numpy(y)

    def shared(self, x):
        w = self.w
        return torch.from_numpy(self.O.swiglu_ffn(x.numpy(), w["ws1"],
                                                  w["ws3"], w["ws2"]))

    def combine(self, x, ys, yp, dest, gate):
        y = yp.numpy()[dest.numpy()]
        return torch.from_numpy(self.O.moe_output(x.numpy(), ys.numpy(), y,
                                                  gate.numpy()))

    def bias_update(self, counts_global, bias, tokens_global):
        c = self.cfg
        nb, _ = self.O.bias_update(counts_global.numpy(), bias.numpy(),
                                   tokens_global, c.topk, c.gamma)
        bias.copy_(torch.from_numpy(nb))


class NumpyBackendFp8(NumpyBackend):
    """FP8 dispatch (§2: activations cast to FP8 before they are sent, the
    outputs returned in BF16 -- here fp64): the tokens' E4M3 codes and
    power-of-two 1 x 128 scales travel as two row tensors, and the experts
    and the shared expert run the oracle's FP8 FFN on them."""

    def __init__(self, cfg, w, rank, world):
        super().__init__(cfg, w, rank, world)
        O, f32 = self.O, np.float32
        self.wq = {e: [O.quantize_128x128_pow2(w[n][e].astype(f32))
                       for n in ("w1", "w3", "w2")]
                   for e in range(self.e0, self.e0 + self.El)}
        self.sq = [O.quantize_128x128_pow2(w[n].astype(f32))
                   for n in ("ws1", "ws3", "ws2")]

    def permute(self, x, idx):
        O = self.O
        p = O.permutation(idx.numpy(), self.cfg.E)
        xq, xs = O.quantize_1x128_pow2(x.numpy().astype(np.float32))
        self._tok = (xq, xs)
        tok = p["src_row"] // self.cfg.topk
        rows = (torch.from_numpy(np.ascontiguousarray(xq[tok])),
                torch.from_numpy(np.ascontiguousarray(xs[tok])))
        return (torch.from_numpy(p["offsets"]), torch.from_numpy(p["dest"]),
                rows)

    def experts(self, xr, offsets_local):
        O = self.O
        codes, scales = (t.numpy() for t in xr)
        off = offsets_local.numpy()
        y = np.zeros((codes.shape[0], self.cfg.H))
        for l in range(self.El):
            a, b = off[l], off[l + 1]
            if b > a:
                y[a:b] = O.fp8_swiglu_ffn(codes[a:b], scales[a:b],
                                          *self.wq[self.e0 + l],
                                          requant=O.quantize_1x128_pow2)[0]
        return torch.from_numpy(y)

    def shared(self, x):
        xq, xs = self._tok
        return torch.from_numpy(self.O.fp8_swiglu_ffn(
            xq, xs, *self.sq, requant=self.O.quantize_1x128_pow2)[0])


def _setup(fp8=False):
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    from deepseekmoe_routing_expert_moe_b300 import inputs
    cfg = (inputs.custom_config("ep_gloo8", 901, **CFG8) if fp8 else
           inputs.custom_config("ep_gloo", 900, **CFG))
    w = inputs.layer_inputs(cfg)
    f = inputs.bf16_bits_to_f32
    vals = {k: (f(v).astype(np.float64) if v.dtype == np.uint16 else v)
            for k, v in w.items()}
    return cfg, w, vals


def _worker(rank, world, port, q, fp8=False):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    cfg, w, vals = _setup(fp8)
    from deepseekmoe_routing_expert_moe_b300 import ep
    be = (NumpyBackendFp8 if fp8 else NumpyBackend)(cfg, vals, rank, world)
    layer = ep.ExpertParallel(be, cfg.E, cfg.topk, cfg.topk_group,
                              cfg.n_group)
    n = cfg.T // world
    x = torch.from_numpy(vals["x"][rank * n:(rank + 1) * n].copy())
    bias = torch.from_numpy(w["bias"].copy())
    out = layer.forward(x, bias, update_bias=True)
    q.put((rank, out.numpy(), bias.numpy(), layer.last["recv_counts"],
           layer.last["send"], layer.last["idx"].numpy()))
    dist.destroy_process_group()


def test_expert_parallel_exchange_equals_the_unsharded_layer():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, world, port, q))
          for r in range(world)]
    for p in ps:
        p.start()
    res = sorted([q.get(timeout=180) for _ in range(world)],
                 key=lambda v: v[0])
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0

    cfg, w, vals = _setup()
    from oracle import moe_oracle as O
    ref = O.layer_forward(vals["x"], vals["w_router"], w["bias"], vals["w1"],
                          vals["w3"], vals["w2"], vals["ws1"], vals["ws3"],
                          vals["ws2"], n_group=cfg.n_group,
                          topk_group=cfg.topk_group, topk=cfg.topk)
    n = cfg.T // world
    El = cfg.E // world
    idx_all = ref["route"]["idx"]
    gsz = cfg.E // cfg.n_group
    for rank, out, bias, rc, send, idx in res:
        rows = slice(rank * n, (rank + 1) * n)
        assert np.array_equal(idx, idx_all[rows])
        np.testing.assert_allclose(out, ref["out"][rows], rtol=1e-12,
                                   atol=1e-12)
        # node-limited: each token's experts lie in at most topk_group groups
        assert np.all([len(set((row // gsz).tolist())) <= cfg.topk_group
                       for row in idx])
        # what this rank received: the sources' counts of its experts
        for s, (_, _, _, _, _, idx_s) in enumerate(res):
            c = O.expert_counts(idx_s, cfg.E)[rank * El:(rank + 1) * El]
            assert np.array_equal(rc[s], c)
        assert sum(send) == n * cfg.topk
    c_all = O.expert_counts(idx_all, cfg.E)
    nb, _ = O.bias_update(c_all, w["bias"], cfg.T, cfg.topk, cfg.gamma)
    for r in res:
        assert np.array_equal(r[2].view(np.uint32), nb.view(np.uint32))


def _fp8_layer(cfg, vals, bias):
    """The unsharded layer with FP8 experts (power-of-two scales) on every
    token: x + FFN_s(xq) + sum_k g_k FFN_{e_k}(xq), the oracle's FP8 FFN."""
    from oracle import moe_oracle as O
    f32 = np.float32
    x = vals["x"]
    z = O.router_logits(x, vals["w_router"])
    r = O.route(z, bias, cfg.n_group, cfg.topk_group, cfg.topk)
    xq, xs = O.quantize_1x128_pow2(x.astype(f32))
    pow2 = O.quantize_1x128_pow2
    sq = [O.quantize_128x128_pow2(vals[n].astype(f32))
          for n in ("ws1", "ws3", "ws2")]
    out = x + O.fp8_swiglu_ffn(xq, xs, *sq, requant=pow2)[0]
    for e in range(cfg.E):
        t, k = np.nonzero(r["idx"] == e)
        if len(t):
            wq = [O.quantize_128x128_pow2(vals[n][e].astype(f32))
                  for n in ("w1", "w3", "w2")]
            y = O.fp8_swiglu_ffn(xq[t], xs[t], *wq, requant=pow2)[0]
            out[t] += r["gate"][t, k][:, None] * y
    return out, r


def test_expert_parallel_fp8_dispatch_equals_the_unsharded_fp8_layer():
    """Dispatch in FP8: the codes and scale rows cross the all-to-all, the
    outputs come back; every rank's output must equal the unsharded layer
    with the same FP8 experts on its tokens (fp64; only summation order may
    differ), and the bias step on the all-reduced load must be the whole
    batch's."""
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, world, port, q, True))
          for r in range(world)]
    for p in ps:
        p.start()
    res = sorted([q.get(timeout=180) for _ in range(world)],
                 key=lambda v: v[0])
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    cfg, w, vals = _setup(True)
    from oracle import moe_oracle as O
    ref, r = _fp8_layer(cfg, vals, w["bias"])
    n = cfg.T // world
    for rank, out, bias, rc, send, idx in res:
        rows = slice(rank * n, (rank + 1) * n)
        assert np.array_equal(idx, r["idx"][rows])
        np.testing.assert_allclose(out, ref[rows], rtol=1e-12, atol=1e-12)
    c_all = O.expert_counts(r["idx"], cfg.E)
    nb, _ = O.bias_update(c_all, w["bias"], cfg.T, cfg.topk, cfg.gamma)
    for rr in res:
        assert np.array_equal(rr[2].view(np.uint32), nb.view(np.uint32))
