#!/usr/bin/env python
"""Throughput of the DeepSeek-V3-shaped MoE layer forward on B300.

A step is one pass of the whole hot path over one batch: router logits,
routing (sigmoid + bias, group-limited top-8, gates), load histogram and
bias step, dispatch order, gather, grouped expert GEMMs (SwiGLU fused),
combine with the shared expert and the residual.  Default workload: the
prefill layer, T = 4096 tokens, hidden 7168, 256 routed experts (I = 2048) +
1 shared, top-8 of 8 groups / 4 kept; bf16 weights and activations, fp32
accumulation; seeded synthetic inputs.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl b300|reference]

Prints ONE JSON line (rank 0).  --impl reference times the CPU oracle (the
only reference that exists for this layer) on a bounded token sample.
Multi-GPU: replicas only -- every rank runs its own layer on its own tokens,
no collective on the data path; value = all ranks' tokens / max rank time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = ("tokens/s per V3-shaped MoE layer on 1 B300 (bf16); "
          "% of TC peak / HBM roofline")
FALLBACK_PEAKS = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0,
                  "bf16_tflops_sustained": 1400.0}


# ------------------------------------------------------------------ utils
def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return d, "measured"
    except (OSError, ValueError):
        return dict(FALLBACK_PEAKS), "fallback"


def blas_threads() -> int:
    try:
        from threadpoolctl import threadpool_info
        n = [i["num_threads"] for i in threadpool_info()
             if i.get("user_api") == "blas"]
        return max(n) if n else (os.cpu_count() or 1)
    except Exception:  # noqa: BLE001
        return os.cpu_count() or 1


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled during the timed region."""
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown",
             "sw_power_cap")

    def __init__(self, gpu_index: int):
        self.idx = gpu_index
        self.proc = None
        self.out = None

    def __enter__(self):
        try:
            self.out = open(os.devnull, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx),
                 f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE,
                stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *a):
        self.lines = []
        if self.proc is not None:
            time.sleep(0.15)
            self.proc.terminate()
            try:
                out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                out, _ = self.proc.communicate()
            self.lines = [l for l in out.splitlines() if l.strip()]

    def summary(self):
        sm, mx, reasons = [], [], set()
        for l in self.lines:
            f = [x.strip() for x in l.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                mx.append(float(f[1]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, f[4:8]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [],
                    "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_index_for_smi(local_rank: int) -> int:
    vis = os.environ.get("CUDA_VISIBLE_DEVICES")
    if vis:
        parts = [p.strip() for p in vis.split(",") if p.strip()]
        if local_rank < len(parts) and parts[local_rank].isdigit():
            return int(parts[local_rank])
    return local_rank


def source_hash(*rel) -> str:
    h = hashlib.sha256()
    for r in rel:
        with open(os.path.join(ROOT, r), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel: str, workload: str):
    """dram read+write bytes per launch of `kernel` from the committed ncu
    summary, if it was taken on the current kernel source; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    try:
        with open(p) as f:
            d = json.load(f)
        e = d[f"{kernel}@{workload}"]
        if e["source_hash"] != source_hash(*e["sources"]):
            return None
        return float(e["dram_bytes_per_launch"])
    except (OSError, KeyError, ValueError):
        return None


def route_blocks(T):
    """Routing blocks of a T-token batch, as the library forms them: ranges
    of at most 64 tokens; from 32 blocks on, their number rounded up to a
    multiple of the 148 SMs."""
    nb = -(-T // 64)
    return -(-nb // 148) * 148 if nb >= 32 else nb


def router_extra_launches(T, H, E, presplit=False):
    """Launches of the router logits beyond one: the weight split on the
    tensor-core path (none when the weights carry a prepared split), and
    the partial-sum kernel when the library splits the reduction over H
    (when the router's tiles fill fewer than half of the 148 SMs)."""
    if E % 16:
        return 0
    split = 0 if presplit else 1
    if T >= 1024 and E % 128 == 0:
        bn = 256 if E % 256 == 0 else 128
    else:
        bn = 64 if E % 64 == 0 else (32 if E % 32 == 0 else 16)
    units = -(-T // 128) * (E // bn)
    nkb = H // 64
    if 2 * units > 148 or nkb // 4 < 2:
        return split
    ks = min(148 // units, nkb // 4)
    kper = -(-nkb // ks)
    return split + (1 if -(-nkb // kper) > 1 else 0)


# ------------------------------------------------------------ CPU oracle
def oracle_sample(cfg, n_tokens: int, step: int = 0):
    """Inputs of a bounded sample for the oracle: the first n_tokens of the
    step's batch plus the weights of every expert they route to (generated
    outside the timed part)."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    from oracle import moe_oracle as O
    f = inputs.bf16_bits_to_f32
    x = f(inputs.x_tokens(cfg, step=step, T=n_tokens))
    wr = inputs.router_weight(cfg)
    b = inputs.bias(cfg)
    pref = inputs.zipf_preference(cfg) if cfg.zipf_s > 0 else None
    z = O.router_logits(x, wr, pref)
    r = O.route(z, b, cfg.n_group, cfg.topk_group, cfg.topk)
    ew = {int(e): tuple(f(a) for a in inputs.expert_weights(cfg, int(e)))
          for e in np.unique(r["idx"])}
    sw = tuple(f(a) for a in inputs.shared_weights(cfg))
    return dict(x=x, wr=wr, b=b, ew=ew, sw=sw, pref=pref)


def oracle_time(cfg, s) -> float:
    """Seconds for the oracle's layer forward of the sample (logits,
    routing, load + bias step, every chosen expert, shared expert, combine)."""
    from oracle import moe_oracle as O
    t0 = time.perf_counter()
    z = O.router_logits(s["x"], s["wr"], s["pref"])
    r = O.route(z, s["b"], cfg.n_group, cfg.topk_group, cfg.topk)
    c = O.expert_counts(r["idx"], cfg.E)
    O.bias_update(c, s["b"], len(s["x"]), cfg.topk, cfg.gamma)
    O.layer_rows(s["x"], r["idx"], r["gate"], lambda e: s["ew"][e], s["sw"])
    return time.perf_counter() - t0


# --------------------------------------------------------------- the arm
def workload_desc(cfg) -> str:
    d = (f"{cfg.name}: V3 MoE layer forward + bias step, T={cfg.T}, "
         f"H={cfg.H}, E={cfg.E}+1 shared, I={cfg.I}, top-{cfg.topk} of "
         f"{cfg.n_group} groups / {cfg.topk_group} kept")
    if cfg.zipf_s > 0:
        d += (f"; skewed load: logits + {cfg.zipf_beta} * r_e^-{cfg.zipf_s} "
              "(Zipf preference over a seeded expert ranking), bias from 0, "
              "fresh tokens each step")
    return d


def config_json(cfg, n_gpus):
    return {"workload": workload_desc(cfg), "T": cfg.T, "H": cfg.H,
            "E": cfg.E, "I": cfg.I, "I_shared": cfg.I_shared,
            "topk": cfg.topk, "n_group": cfg.n_group,
            "topk_group": cfg.topk_group, "global_batch": cfg.T * n_gpus,
            "parallelism": f"replicas x{n_gpus} (no data-path collective)",
            "l2": "inputs larger than L2: 22.6 GB of expert weights streamed "
                  "per step; 4 rotating activation batches"}


def e2e_loop_multi(step, host_in, out_like, steps, stream,
                   barrier=lambda: None):
    """End to end with host buffers: every step uploads its inputs from
    pinned host memory and downloads its outputs into pinned host memory.
    host_in[b] is the list of pinned host inputs of batch b (steps cycle
    over the batches); out_like lists (shape, dtype) of the outputs.  The
    copies run on their own streams with double-buffered device inputs and
    outputs, so that step i+1's uploads and step i's downloads overlap
    step i's compute.  step(ins_dev, outs_dev) enqueues one step on
    `stream`.  Returns the elapsed ms of `steps` steps."""
    import torch
    NB = len(host_in)
    ind = [[torch.empty_like(t, device="cuda") for t in host_in[0]]
           for _ in range(2)]
    outd = [[torch.empty(sh, dtype=dt, device="cuda") for sh, dt in out_like]
            for _ in range(2)]
    outh = [[torch.empty(sh, dtype=dt).pin_memory() for sh, dt in out_like]
            for _ in range(2)]
    up_s, dn_s = torch.cuda.Stream(), torch.cuda.Stream()
    ev = lambda: torch.cuda.Event()  # noqa: E731
    h2d_done = [ev() for _ in range(2)]
    comp_done = [ev() for _ in range(2)]
    d2h_done = [ev() for _ in range(2)]
    for e in comp_done + d2h_done:
        e.record(stream)
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    barrier()
    e0.record(stream)
    up_s.wait_event(e0)
    dn_s.wait_event(e0)
    for i in range(steps):
        b = i % 2
        up_s.wait_event(comp_done[b])          # ind[b] no longer read
        with torch.cuda.stream(up_s):
            for dst, src in zip(ind[b], host_in[i % NB]):
                dst.copy_(src, non_blocking=True)
        h2d_done[b].record(up_s)
        stream.wait_event(h2d_done[b])
        stream.wait_event(d2h_done[b])         # outd[b] already downloaded
        step(ind[b], outd[b])
        comp_done[b].record(stream)
        dn_s.wait_event(comp_done[b])
        with torch.cuda.stream(dn_s):
            for dst, src in zip(outh[b], outd[b]):
                dst.copy_(src, non_blocking=True)
        d2h_done[b].record(dn_s)
    stream.wait_event(d2h_done[(steps - 1) % 2])
    stream.wait_event(d2h_done[steps % 2])
    e1.record(stream)
    barrier()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1)


def e2e_loop(step, xs, T, H, steps, stream, barrier=lambda: None):
    """e2e_loop_multi for a layer with one input x [T, H] bf16 and one
    output [T, H] bf16: step(x_dev, out_dev)."""
    import torch
    host_in = [[xs[i].cpu().pin_memory()] for i in range(len(xs))]
    return e2e_loop_multi(lambda i_, o_: step(i_[0], o_[0]), host_in,
                          [((T, H), torch.int16)], steps, stream, barrier)


def run_gpu(args, rank, world, local_rank):
    import torch
    from deepseekmoe_routing_expert_moe_b300 import inputs, ops
    torch.cuda.set_device(local_rank)
    cfg = inputs.CONFIGS[args.workload]
    d = ops.dims_of(cfg)
    T, H, E, K = cfg.T, cfg.H, cfg.E, cfg.topk

    # ---- inputs resident in HBM
    w1, w3, w2 = inputs.device_expert_weights(cfg, "cuda")
    ws1, ws3, ws2 = inputs.shared_weights(cfg, "cuda")
    wr = torch.from_numpy(inputs.router_weight(cfg)).cuda()
    # the skewed-load workload's per-expert preference enters as the
    # router's additive term (zero preference: no term)
    pref = (torch.from_numpy(inputs.zipf_preference(cfg)).cuda()
            if cfg.zipf_s > 0 else None)
    # the router weight's bf16 split made once, as deployed weights would
    # carry it (moe_router_weight_split)
    W = ops.Weights(wr, w1, w3, w2, ws1, ws3, ws2,
                    router_offset=pref).with_router_split()
    # fresh seeded tokens every step for the skewed run (its config asks
    # for them; up to its 50 steps), 4 rotating batches otherwise
    NB = min(max(args.steps, 4), cfg.steps) if cfg.zipf_s > 0 else 4
    xs = [inputs.x_tokens(cfg, step=i + 1000 * rank, device="cuda")
          for i in range(NB)]
    bias = torch.from_numpy(inputs.bias(cfg)).cuda()
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    counts = torch.zeros(E, dtype=torch.int32, device="cuda")
    # per-step load statistics (max, mean, min of the expert counts),
    # written by the count-scan kernel of each timed step
    # (rows padded to 16 bytes: the library takes 16-byte-aligned pointers)
    load = torch.zeros((args.steps, 4), dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_FORWARD)
    stream = torch.cuda.current_stream()

    def step(i, counts_out=None, stats=None):
        ops.moe_forward(d, W, xs[i % NB], bias, out, ws, update_bias=True,
                        counts_out=counts_out, load_stats_out=stats)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert ops.moe_get_device_error(ws) == 0

    def barrier():
        if world > 1:
            import torch.distributed as dist
            dist.barrier()
        torch.cuda.synchronize()

    # ---- timed region: exactly K steps
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index_for_smi(local_rank)) as clk:
        barrier()
        ev0.record(stream)
        for i in range(args.steps):
            step(i, stats=load[i])
        ev1.record(stream)
        barrier()
    ms = ev0.elapsed_time(ev1)
    clocks = clk.summary()
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([ms], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        ms = float(t.item())
    ms_per_step = ms / args.steps
    value = world * T * args.steps / (ms / 1e3)

    # ---- kernel-level timing (separate pass, same steps, events between
    #      the library's launches on its stream)
    nk = ops.MOE_FORWARD_KERNELS
    sets = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)]
            for _ in range(args.steps)]
    for i in range(args.steps):
        ops.moe_set_profile_events(sets[i])
        step(i, counts_out=counts if i == args.steps - 1 else None)
    ops.moe_set_profile_events(None)
    torch.cuda.synchronize()
    kt = np.array([[s[j].elapsed_time(s[j + 1]) for j in range(nk)]
                   for s in sets])          # ms, [steps, kernels]
    kmean = kt.mean(0)
    kernels = {n: round(float(v), 4) for n, v in
               zip(ops.FORWARD_KERNEL_NAMES, kmean)}
    c = counts.cpu().numpy().astype(np.int64)
    assert c.sum() == T * K
    lo = load.cpu().numpy().astype(np.float64)
    mom = lo[:, 0] / lo[:, 1]
    load_json = {"max_over_mean_first": round(float(mom[0]), 3),
                 "max_over_mean_last": round(float(mom[-1]), 3),
                 "max_over_mean_avg": round(float(mom.mean()), 3),
                 "min_over_mean_avg": round(float((lo[:, 2] / lo[:, 1]).mean()),
                                            3)}
    if cfg.zipf_s > 0:
        load_json["max_over_mean_per_step"] = [round(float(v), 3) for v in mom]

    # ---- roofline of the dominant kernel (expert up-projection GEMM)
    pk, pk_src = peaks()
    touched = int((c > 0).sum())
    I, Is = cfg.I, cfg.I_shared
    up_bytes = (touched * 2 * I * H * 2 + 2 * Is * H * 2 +     # W1, W3 (+shared)
                T * K * H * 2 + T * H * 2 +                    # A: xp, x
                T * K * I * 2 + T * Is * 2)                    # h written
    up_flops = 2.0 * (T * K + T) * H * 2 * I
    dn_bytes = (touched * H * I * 2 + H * Is * 2 + T * K * I * 2 + T * Is * 2
                + T * K * H * 2 + T * H * 2)
    dn_flops = 2.0 * (T * K + T) * I * H
    t_up = kmean[5] / 1e3
    t_dn = kmean[6] / 1e3
    hbm = float(pk["hbm_gbs"])
    tc = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
    up_hbm_s = up_bytes / (hbm * 1e9)
    up_tc_s = up_flops / (tc * 1e12)
    if up_hbm_s >= up_tc_s:
        roof = {"bound": "hbm", "achieved": round(up_bytes / t_up / 1e9, 1),
                "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor",
                "achieved": round(up_flops / t_up / 1e12, 1),
                "peak": tc, "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = ncu_traffic("gemm_up_swiglu", cfg.name)
    roof["kernel"] = "grouped_gemm_kernel<up,N=256> (expert up-projection + SwiGLU)"
    roof["algorithmic_bytes"] = int(up_bytes)
    roof["peak_source"] = f"{pk_src} (MEASURED_PEAKS.json)" \
        if pk_src == "measured" else "fallback (profiling recipe)"
    roof["tensor_frac"] = round(up_flops / t_up / 1e12 / tc, 4)
    roof["down_gemm"] = {"ms": round(kmean[6], 4),
                         "hbm_frac": round(dn_bytes / t_dn / 1e9 / hbm, 4),
                         "tensor_frac": round(dn_flops / t_dn / 1e12 / tc, 4),
                         "algorithmic_bytes": int(dn_bytes),
                         "traffic": ncu_traffic("gemm_down", cfg.name)}

    # ---- end to end through the C ABI with host buffers: every step copies
    #      its x from pinned host memory and its output back; the copies run
    #      on their own streams (double-buffered device x/out) so that step
    #      i+1's upload and step i's download overlap step i's compute
    e2e_ms = e2e_loop(
        lambda x, o: ops.moe_forward(d, W, x, bias, o, ws, update_bias=True,
                                     stream=stream),
        xs, T, H, args.steps, stream, barrier)
    if world > 1:
        import torch.distributed as dist
        t = torch.tensor([e2e_ms], dtype=torch.float64, device="cuda")
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        e2e_ms = float(t.item())
    assert ops.moe_get_device_error(ws) == 0

    res = {
        "metric": METRIC, "value": round(value, 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic, seeded (x ~N(0,1), expert weights ~N(0,0.02) "
                "bf16, router ~N(0,0.006) fp32, bias ~U(-0.01,0.01))",
        "config": config_json(cfg, world),
        "roofline": roof,
        "e2e": {"value": round(world * T * args.steps / (e2e_ms / 1e3), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2,
                "overlap": "uploads/downloads on their own streams, "
                           "double-buffered"},
        # the router logits are one launch (the weights carry their
        # prepared bf16 split), two when its k ranges are split (the partial
        # sums are added by a kernel); the dispatch copy is a launch only at
        # >= 64 rows per expert (below that the up GEMM gathers the rows
        # from x itself)
        "gpu_launches": (nk - (0 if T * K >= 64 * E else 1)
                         + router_extra_launches(T, H, E, presplit=True))
                        * args.steps,
        "clocks": clocks,
        "kernels_ms": kernels,
        "experts_touched": touched,
        "load": load_json,
        "impl": "b300",
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = oracle_sample(cfg, args.cpu_sample_tokens)
        sec = oracle_time(cfg, s)
        res["cpu_baseline"] = {
            "value": round(args.cpu_sample_tokens / sec, 4),
            "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"first {args.cpu_sample_tokens} tokens of the batch "
                      f"through the numpy fp64 oracle ({sec:.1f} s: logits, "
                      "routing, bias step, their experts + shared expert)"}
    return res


def run_route_gpu(args, rank, world, local_rank):
    """The routing-only configuration (T=16384 at the V3 shape): per step,
    from precomputed fp32 logits, moe_route (sigmoid + bias, group-limited
    top-8, gates, histogram), moe_permute without rows (offsets, dest,
    src_row) and moe_bias_update -- the public calls a user makes.  8
    rotating logits batches (134 MB, larger than L2)."""
    import torch
    from deepseekmoe_routing_expert_moe_b300 import inputs, ops
    torch.cuda.set_device(local_rank)
    cfg = inputs.CONFIGS[args.workload]
    d = ops.dims_of(cfg)
    T, E, K = cfg.T, cfg.E, cfg.topk
    NB = 8
    wr = torch.from_numpy(inputs.router_weight(cfg)).cuda()
    zs = []
    for i in range(NB):   # logits on the device from the seeded tokens
        x = inputs.x_tokens(cfg, step=i + 1000 * rank, device="cuda")
        z = torch.empty((T, E), dtype=torch.float32, device="cuda")
        wsl = ops.workspace(d, ops.MOE_WS_ROUTER_LOGITS)
        ops.moe_router_logits(d, x, wr, z, wsl)
        zs.append(z)
    del wsl
    bias = torch.from_numpy(inputs.bias(cfg)).cuda()
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, K), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    dest = torch.empty((T, K), dtype=torch.int32, device="cuda")
    src_row = torch.empty(T * K, dtype=torch.int32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_PERMUTE)
    stream = torch.cuda.current_stream()

    calls = (
        lambda i: ops.moe_route(d, zs[i % NB], bias, idx, gate, counts, ws),
        lambda i: ops.moe_permute(d, None, idx, offsets, dest, src_row, None,
                                  ws),
        lambda i: ops.moe_bias_update(d, counts, bias),
    )

    def step(i):
        for c in calls:
            c(i)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert ops.moe_get_device_error(ws) == 0
    # The step is six small kernels: launched one by one from Python the
    # host would be timed, so NB consecutive steps (one per logits batch)
    # are captured once in a CUDA graph and the graph is replayed.
    side = torch.cuda.Stream()
    side.wait_stream(stream)

    def capture(fn):
        gr = torch.cuda.CUDAGraph()
        with torch.cuda.stream(side):
            with torch.cuda.graph(gr, stream=side):
                for i in range(NB):
                    fn(i)
        return gr

    g = capture(step)
    # each public call alone, NB times per graph (its own per-call time,
    # with nothing recorded between the kernels)
    g_calls = [capture(c) for c in calls]
    stream.wait_stream(side)
    reps = max(1, args.steps // NB)
    for _ in range(max(1, args.warmup // NB)):
        g.replay()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index_for_smi(local_rank)) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    clocks = clk.summary()
    args.steps = reps * NB
    kt = []
    for gc in g_calls:
        gc.replay()
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(reps):
            gc.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
        kt.append(ev0.elapsed_time(ev1) / (reps * NB))
    kt = np.array(kt)
    # algorithmic bytes of the routing call (logits + bias read; idx,
    # gates, counts and the per-block histogram rows written)
    nblk = route_blocks(T)
    route_bytes = T * E * 4 + E * 4 + T * K * 8 + E * 4 + 2 * nblk * E * 4
    perm_bytes = T * K * 4 + 2 * T * K * 4 + (E + 1) * 4 + 3 * nblk * E * 4
    pk, pk_src = peaks()
    hbm = float(pk["hbm_gbs"])
    roof = {"bound": "hbm",
            "achieved": round(route_bytes / (kt[0] / 1e3) / 1e9, 1),
            "peak": hbm, "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / hbm, 4)
    roof["traffic"] = ncu_traffic("route", cfg.name)
    roof["kernel"] = ("moe_route call (route_kernel + count scan): "
                      "logits -> idx, gates, counts")
    roof["algorithmic_bytes"] = int(route_bytes)
    roof["peak_source"] = f"{pk_src} (MEASURED_PEAKS.json)"
    roof["permute_call"] = {"ms": round(float(kt[1]), 4),
                            "algorithmic_bytes": int(perm_bytes)}
    # end to end with host buffers: each step uploads its logits from
    # pinned memory and downloads idx, gates and dest (launched eagerly,
    # host launch time included)
    zh = [torch.empty((T, E), dtype=torch.float32).pin_memory()
          for _ in range(2)]
    for i in range(2):
        zh[i].copy_(zs[i].cpu())
    oh = [torch.empty((T, K), dtype=torch.int32).pin_memory() for _ in range(3)]
    zd = torch.empty((T, E), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        zd.copy_(zh[i % 2], non_blocking=True)
        ops.moe_route(d, zd, bias, idx, gate, counts, ws)
        ops.moe_permute(d, None, idx, offsets, dest, src_row, None, ws)
        ops.moe_bias_update(d, counts, bias)
        oh[0].copy_(idx, non_blocking=True)
        oh[1].copy_(gate.view(torch.int32), non_blocking=True)
        oh[2].copy_(dest, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    assert ops.moe_get_device_error(ws) == 0
    return {
        "metric": "tokens/s routed (routing + dispatch order + bias step) "
                  "at the V3 shape on 1 B300; % of HBM roofline",
        "value": round(T * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic, seeded (logits from x ~N(0,1), W_router "
                "~N(0,0.006); bias ~U(-0.01,0.01))",
        "config": {"workload": f"{cfg.name}: routing-only, T={T}, E={E}, "
                               f"top-{K} of {cfg.n_group} groups / "
                               f"{cfg.topk_group} kept, from fp32 logits",
                   "T": T, "E": E, "topk": K, "n_group": cfg.n_group,
                   "topk_group": cfg.topk_group,
                   "l2": "8 rotating logits batches, 134 MB > L2"},
        "roofline": roof,
        "e2e": {"value": round(T * args.steps / (e2e_ms / 1e3), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": T * E * 4,
                "d2h_bytes_per_step": 3 * T * K * 4},
        "gpu_launches": 6 * args.steps,
        "clocks": clocks,
        "calls_ms": {"moe_route": round(float(kt[0]), 4),
                     "moe_permute": round(float(kt[1]), 4),
                     "moe_bias_update": round(float(kt[2]), 4)},
        "impl": "b300",
    }


def run_balance_gpu(args, rank, world, local_rank):
    """The sequence-wise balance loss (the complementary loss beside the
    bias): per step, moe_seq_balance_loss on T=16384 fp32 logits at the V3
    shape (256 experts, top-8) cut into four 4096-token sequences -> the
    per-sequence counts, P and loss.  8 rotating logits batches (134 MB,
    larger than L2), replayed from a CUDA graph like the routing workload."""
    import torch
    from deepseekmoe_routing_expert_moe_b300 import inputs, ops
    from oracle import moe_oracle as O
    torch.cuda.set_device(local_rank)
    cfg = inputs.CONFIGS["route_v3"]
    d = ops.dims_of(cfg)
    T, E, K, S = cfg.T, cfg.E, cfg.topk, 4096
    n_seq = -(-T // S)
    alpha = 1e-4
    NB = 8
    wr = torch.from_numpy(inputs.router_weight(cfg)).cuda()
    zs = []
    wsl = ops.workspace(d, ops.MOE_WS_ROUTER_LOGITS)
    for i in range(NB):
        x = inputs.x_tokens(cfg, step=i + 1000 * rank, device="cuda")
        z = torch.empty((T, E), dtype=torch.float32, device="cuda")
        ops.moe_router_logits(d, x, wr, z, wsl)
        zs.append(z)
    del wsl
    counts = torch.empty((n_seq, E), dtype=torch.int32, device="cuda")
    P = torch.empty((n_seq, E), dtype=torch.float32, device="cuda")
    loss = torch.empty(n_seq, dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_SEQ_BALANCE)
    stream = torch.cuda.current_stream()

    def step(i):
        ops.moe_seq_balance_loss(d, zs[i % NB], S, alpha, counts, P, loss, ws)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert ops.moe_get_device_error(ws) == 0
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(g, stream=side):
            for i in range(NB):
                step(i)
    stream.wait_stream(side)
    reps = max(1, args.steps // NB)
    for _ in range(max(1, args.warmup // NB)):
        g.replay()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index_for_smi(local_rank)) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    args.steps = reps * NB
    # algorithmic bytes: the logits read once, the per-sequence counts, P
    # and loss written (the s' / flag rows the kernels pass between their
    # passes are this implementation's own traffic, 10 bytes per logit)
    alg = T * E * 4 + n_seq * E * 8 + n_seq * 4
    pk, pk_src = peaks()
    hbm = float(pk["hbm_gbs"])
    roof = {"bound": "hbm",
            "achieved": round(alg * args.steps / (ms / 1e3) / 1e9, 1),
            "peak": hbm, "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / hbm, 4)
    roof["traffic"] = None
    roof["kernel"] = ("moe_seq_balance_loss call (balance_token_kernel + "
                      "balance_seq_kernel + balance_loss_kernel)")
    roof["algorithmic_bytes"] = int(alg)
    roof["peak_source"] = f"{pk_src} (MEASURED_PEAKS.json)"
    # end to end: logits uploaded from pinned memory, the per-sequence
    # losses read back, every step
    zh = [torch.empty((T, E), dtype=torch.float32).pin_memory()
          for _ in range(2)]
    for i in range(2):
        zh[i].copy_(zs[i].cpu())
    lh = torch.empty(n_seq, dtype=torch.float32).pin_memory()
    zd = torch.empty((T, E), dtype=torch.float32, device="cuda")
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(args.steps):
        zd.copy_(zh[i % 2], non_blocking=True)
        ops.moe_seq_balance_loss(d, zd, S, alpha, counts, P, loss, ws)
        lh.copy_(loss, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = e0.elapsed_time(e1)
    assert ops.moe_get_device_error(ws) == 0
    res = {
        "metric": "tokens/s through the sequence-wise balance loss (eq. "
                  "17-20) at the V3 shape on 1 B300; % of HBM roofline",
        "value": round(T * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic, seeded (logits from x ~N(0,1), W_router "
                "~N(0,0.006))",
        "config": {"workload": f"balance_v3: sequence-wise balance loss, "
                               f"T={T} as {n_seq} sequences of {S}, E={E}, "
                               f"top-{K}, alpha={alpha}",
                   "T": T, "E": E, "topk": K, "seq_len": S,
                   "l2": "8 rotating logits batches, 134 MB > L2"},
        "roofline": roof,
        "e2e": {"value": round(T * args.steps / (e2e_ms / 1e3), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": T * E * 4,
                "d2h_bytes_per_step": n_seq * 4},
        "gpu_launches": 3 * args.steps,
        "clocks": clk.summary(),
        "impl": "b300",
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        zc = zs[0][:S].cpu().numpy()
        O.seq_balance_loss(zc, S, K, alpha)
        t0 = time.perf_counter()
        reps_cpu = 0
        while time.perf_counter() - t0 < 10.0:
            O.seq_balance_loss(zc, S, K, alpha)
            reps_cpu += 1
        dt = time.perf_counter() - t0
        res["cpu_baseline"] = {
            "value": round(S * reps_cpu / dt, 1), "unit": "tokens/s",
            "cores": blas_threads(), "kind": "oracle",
            "sample": f"one {S}-token sequence of the first logits batch "
                      f"through the numpy oracle, repeated for ~10 s"}
    return res


FP8_WORKLOADS = ("decode_v3_fp8", "prefill_v3_fp8", "decode_v3_e32_fp8",
                 "prefill_v3_e32_fp8", "decode_v3_mx", "prefill_v3_mx",
                 "decode_v3_e32_mx", "prefill_v3_e32_mx")


def fp8_kind(workload):
    """("fp8" | "mx", base configuration) of an FP8 workload name: _fp8 is
    the fp32-scale path (CUDA-core promotion), _mx the power-of-two-scale
    path (scales applied by the tensor cores)."""
    kind = "mx" if workload.endswith("_mx") else "fp8"
    return kind, workload[:-len("_" + kind)]


def run_fp8_gpu(args, rank, world, local_rank):
    """A V3 layer with FP8 experts -- decode (T=128) or prefill (T=4096):
    per step, through the public calls, router logits -> moe_route ->
    moe_permute (indices) -> quantise-on-permute (moe_permute_fp8 |
    moe_permute_mx) -> FP8 experts (moe_expert_ffn_fp8 | moe_expert_ffn_mx)
    -> moe_combine -> moe_bias_update.  The weights are quantized to E4M3
    (128 x 128 block scales: fp32, or power-of-two UE8M0 bytes) once,
    before timing, as a deployment would store them.  4 rotating token
    batches; the E4M3 weights (11.3 GB at 256 experts, 1.4 GB for the
    32-expert profiling stand-in) exceed L2."""
    import torch
    from deepseekmoe_routing_expert_moe_b300 import inputs, ops
    torch.cuda.set_device(local_rank)
    kind, base = fp8_kind(args.workload)
    mx = kind == "mx"
    cfg = inputs.CONFIGS[base]
    d = ops.dims_of(cfg)
    T, H, E, K, I, Is = cfg.T, cfg.H, cfg.E, cfg.topk, cfg.I, cfg.I_shared
    w1, w3, w2 = inputs.device_expert_weights(cfg, "cuda")
    ws1, ws3, ws2 = inputs.shared_weights(cfg, "cuda")
    Wq = (ops.WeightsMx if mx else ops.WeightsFp8).quantize(
        w1, w3, w2, ws1, ws3, ws2)
    del w1, w3, w2
    torch.cuda.empty_cache()
    wr = torch.from_numpy(inputs.router_weight(cfg)).cuda()
    NB = 4
    xs = [inputs.x_tokens(cfg, step=i + 1000 * rank, device="cuda")
          for i in range(NB)]
    bias = torch.from_numpy(inputs.bias(cfg)).cuda()
    z = torch.empty((T, E), dtype=torch.float32, device="cuda")
    idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
    gate = torch.empty((T, K), dtype=torch.float32, device="cuda")
    counts = torch.empty(E, dtype=torch.int32, device="cuda")
    offsets = torch.empty(E + 1, dtype=torch.int32, device="cuda")
    dest = torch.empty((T, K), dtype=torch.int32, device="cuda")
    src_row = torch.empty(T * K, dtype=torch.int32, device="cuda")
    sdt = torch.uint8 if mx else torch.float32
    xq = torch.empty((T, H), dtype=torch.uint8, device="cuda")
    xsc = torch.empty((T, H // 128), dtype=sdt, device="cuda")
    xpq = torch.empty((T * K, H), dtype=torch.uint8, device="cuda")
    xps = torch.empty((T * K, H // 128), dtype=sdt, device="cuda")
    permute_q = ops.moe_permute_mx if mx else ops.moe_permute_fp8
    ffn_q = ops.moe_expert_ffn_mx if mx else ops.moe_expert_ffn_fp8
    yp = torch.empty((T * K, H), dtype=torch.int16, device="cuda")
    ys = torch.empty((T, H), dtype=torch.int16, device="cuda")
    out = torch.empty((T, H), dtype=torch.int16, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_FORWARD)
    stream = torch.cuda.current_stream()

    def step(x, o, ev=None):
        ops.moe_router_logits(d, x, wr, z, ws)
        ops.moe_route(d, z, bias, idx, gate, counts, ws)
        ops.moe_permute(d, None, idx, offsets, dest, src_row, None, ws)
        permute_q(d, x, dest, xq, xsc, xpq, xps, ws)
        if ev: ev[0].record(stream)
        ffn_q(d, Wq, xpq, xps, xq, xsc, offsets, yp, ys, ws)
        if ev: ev[1].record(stream)
        ops.moe_combine(d, x, ys, yp, dest, gate, o)
        ops.moe_bias_update(d, counts, bias)

    for i in range(args.warmup):
        step(xs[i % NB], out)
    torch.cuda.synchronize()
    assert ops.moe_get_device_error(ws) == 0
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index_for_smi(local_rank)) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(args.steps):
            step(xs[i % NB], out)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    clocks = clk.summary()
    # FFN call alone (events around it, separate pass)
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)]
           for _ in range(args.steps)]
    for i in range(args.steps):
        step(xs[i % NB], out, evs[i])
    torch.cuda.synchronize()
    t_ffn = float(np.mean([e[0].elapsed_time(e[1]) for e in evs])) / 1e3
    c = counts.cpu().numpy().astype(np.int64)
    touched = int((c > 0).sum())
    nkh = H // 128
    sb = 1 if mx else 4                                         # scale bytes
    ffn_bytes = (touched * 3 * I * H + 3 * Is * H +             # E4M3 weights
                 (touched * 3 * (I // 128) * nkh) * sb +        # their scales
                 3 * (Is // 128) * nkh * sb +
                 (T * K + T) * H * (1 + sb / 128) +             # token codes
                 2 * (T * K * I + T * Is) * (1 + sb / 128) +    # m out + in
                 (T * K + T) * H * 2)                           # y (bf16)
    pk, pk_src = peaks()
    hbm = float(pk["hbm_gbs"])
    roof = {"bound": "hbm", "achieved": round(ffn_bytes / t_ffn / 1e9, 1),
            "peak": hbm, "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / hbm, 4)
    roof["traffic"] = ncu_traffic("ffn_" + kind, args.workload)
    roof["kernel"] = (("moe_expert_ffn_mx call (mx_gemm_kernel up + down, "
                       "block-scaled tcgen05 MMAs" if mx else
                       "moe_expert_ffn_fp8 call (fp8_gemm_kernel up + down")
                      + ", E4M3 weights streamed once)")
    roof["algorithmic_bytes"] = int(ffn_bytes)
    roof["ffn_ms"] = round(t_ffn * 1e3, 4)
    roof["peak_source"] = f"{pk_src} (MEASURED_PEAKS.json)"
    # end to end: x uploaded from pinned memory, out read back, every step
    # (copies overlapped with the neighbouring steps' compute)
    torch.cuda.synchronize()
    e2e_ms = e2e_loop(step, xs, T, H, args.steps, stream)
    assert ops.moe_get_device_error(ws) == 0
    return {
        "metric": f"tokens/s per V3-shaped MoE {base.split('_')[0]} layer "
                  "on 1 B300 with FP8 (E4M3) experts"
                  + (" (power-of-two scales)" if mx else "")
                  + "; % of HBM roofline",
        "value": round(T * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "e4m3 experts (1x128 / 128x128 "
                 + ("UE8M0 power-of-two" if mx else "fp32")
                 + " scales), bf16 activations elsewhere, fp32 routing",
        "data": f"synthetic, seeded (the {base} inputs; weights "
                "quantized from the bf16 ones before timing)",
        "config": {"workload": f"{args.workload}: V3 layer T={T}, "
                               f"H={H}, E={E}+1 shared, I={I}, top-{K}, "
                               "FP8 experts"
                               + (", power-of-two scales" if mx else ""),
                   "T": T, "H": H, "E": E, "topk": K, "I": I,
                   "l2": f"{(E * 3 * I * H + 3 * Is * H) / 1e9:.1f} GB of "
                         "E4M3 weights streamed per step > L2"},
        "roofline": roof,
        "e2e": {"value": round(T * args.steps / (e2e_ms / 1e3), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": T * H * 2,
                "d2h_bytes_per_step": T * H * 2},
        # router 1 (+ weight split, + split-K sum), route + count scan 2,
        # dispatch order (block counts, scan, dest) 3, quantise-on-permute
        # 1, FP8 up + down 2, combine 1, bias step 1
        "gpu_launches": (11 + router_extra_launches(T, H, E)) * args.steps,
        "clocks": clocks,
        "experts_touched": touched,
        "impl": "b300",
    }


def run_decode_fp8_reference(args):
    """Oracle arm of the FP8 workloads: per step one token of the batch
    through the oracle's routing and FP8 experts (its 8 routed experts and
    the shared one; fp32 or power-of-two scales as the workload's GPU arm);
    the oracle quantizes those experts' weights once before timing, as the
    GPU arm does."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    from oracle import moe_oracle as O
    kind, base = fp8_kind(args.workload)
    cfg = inputs.CONFIGS[base]
    if kind == "mx":
        q_w, q_a = O.quantize_128x128_pow2, O.quantize_1x128_pow2
    else:
        q_w, q_a = O.quantize_128x128, O.quantize_1x128
    f32 = inputs.bf16_bits_to_f32
    x = f32(inputs.x_tokens(cfg))[:1]
    wr = inputs.router_weight(cfg)
    b = inputs.bias(cfg)
    idx = O.route(O.router_logits(x, wr), b, cfg.n_group, cfg.topk_group,
                  cfg.topk)["idx"][0]
    qw = {int(e): [q_w(f32(m)) for m in inputs.expert_weights(cfg, int(e))]
          for e in idx}
    qs = [q_w(f32(m)) for m in inputs.shared_weights(cfg)]

    def one():
        z = O.router_logits(x, wr)
        r = O.route(z, b, cfg.n_group, cfg.topk_group, cfg.topk)
        aq, as_ = q_a(x)
        y = x.astype(np.float64) + O.fp8_swiglu_ffn(aq, as_, *qs,
                                                    requant=q_a)[0]
        for k, e in enumerate(r["idx"][0]):
            y = y + float(r["gate"][0, k]) * O.fp8_swiglu_ffn(
                aq, as_, *qw[int(e)], requant=q_a)[0]
        return y

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    tot = time.perf_counter() - t0
    v = args.steps / tot
    sample = ("one token per step through the numpy oracle: logits, "
              "routing, 1x128 quantization, its 8 FP8 experts + the shared "
              "one (weights quantized before timing)")
    return {
        "metric": f"tokens/s per V3-shaped MoE {base.split('_')[0]} layer "
                  "with FP8 experts"
                  + (" (power-of-two scales)" if kind == "mx" else "")
                  + "; oracle on the host cores",
        "value": round(v, 4), "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64 on e4m3 values", "data": "synthetic, seeded",
        "config": {"workload": f"{args.workload}: V3 layer, FP8 experts"},
        "impl": "reference",
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s",
                         "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_backward_gpu(args, rank, world, local_rank):
    """The routing side of a training step's backward at the V3 shape: per
    step, moe_route_balance_backward (the gates' gradient and the
    sequence-wise balance loss's gradient to the logits in one pass; equal
    bit for bit to moe_route_backward followed by
    moe_seq_balance_loss_backward), on T=16384 fp32 logits (four 4096-token
    sequences).  8 rotating batches (134 MB of logits > L2), replayed from a
    CUDA graph."""
    import torch
    from deepseekmoe_routing_expert_moe_b300 import inputs, ops
    torch.cuda.set_device(local_rank)
    cfg = inputs.CONFIGS["route_v3"]
    d = ops.dims_of(cfg)
    T, E, K, S = cfg.T, cfg.E, cfg.topk, 4096
    n_seq = -(-T // S)
    NB = 8
    wr = torch.from_numpy(inputs.router_weight(cfg)).cuda()
    bias = torch.from_numpy(inputs.bias(cfg)).cuda()
    wsl = ops.workspace(d, ops.MOE_WS_FORWARD)
    zs, idxs, cnts = [], [], []
    for i in range(NB):   # logits, routing and balance counts per batch
        x = inputs.x_tokens(cfg, step=i + 1000 * rank, device="cuda")
        z = torch.empty((T, E), dtype=torch.float32, device="cuda")
        ops.moe_router_logits(d, x, wr, z, wsl)
        idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, K), dtype=torch.float32, device="cuda")
        counts = torch.empty(E, dtype=torch.int32, device="cuda")
        ops.moe_route(d, z, bias, idx, gate, counts, wsl)
        cs = torch.empty((n_seq, E), dtype=torch.int32, device="cuda")
        P = torch.empty((n_seq, E), dtype=torch.float32, device="cuda")
        loss = torch.empty(n_seq, dtype=torch.float32, device="cuda")
        ops.moe_seq_balance_loss(d, z, S, 1e-4, cs, P, loss, wsl)
        zs.append(z)
        idxs.append(idx)
        cnts.append(cs)
    g = torch.Generator(device="cuda").manual_seed(5 + rank)
    dgate = torch.randn((T, K), device="cuda", generator=g)
    dloss = torch.ones(n_seq, device="cuda")
    dz = torch.empty((T, E), dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_ROUTE)
    stream = torch.cuda.current_stream()

    def step(i):
        ops.moe_route_balance_backward(d, zs[i % NB], idxs[i % NB], dgate, S,
                                       1e-4, cnts[i % NB], dz, ws,
                                       dloss=dloss)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert ops.moe_get_device_error(ws) == 0
    side = torch.cuda.Stream()
    side.wait_stream(stream)
    gr = torch.cuda.CUDAGraph()
    with torch.cuda.stream(side):
        with torch.cuda.graph(gr, stream=side):
            for i in range(NB):
                step(i)
    stream.wait_stream(side)
    reps = max(1, args.steps // NB)
    gr.replay()
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index_for_smi(local_rank)) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(reps):
            gr.replay()
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    args.steps = reps * NB
    # algorithmic bytes of a step: logits, top-K ids, gate gradients and
    # counts read once; dlogits written once
    alg = T * E * 4 + T * K * 8 + n_seq * E * 4 + n_seq * 4 + T * E * 4
    pk, pk_src = peaks()
    hbm = float(pk["hbm_gbs"])
    roof = {"bound": "hbm",
            "achieved": round(alg * args.steps / (ms / 1e3) / 1e9, 1),
            "peak": hbm, "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / hbm, 4)
    roof["traffic"] = None
    roof["kernel"] = ("route_balance_backward_kernel (both gradients, the "
                      "logits read once, dlogits written once)")
    roof["algorithmic_bytes"] = int(alg)
    roof["peak_source"] = f"{pk_src} (MEASURED_PEAKS.json)"
    clocks = clk.summary()
    # end to end: each step uploads its logits, top-K ids, gate gradients
    # and sequence counts from pinned memory and reads dlogits back (the
    # copies of neighbouring steps overlap the compute)
    host_in = [[zs[i].cpu().pin_memory(), idxs[i].cpu().pin_memory(),
                dgate.cpu().pin_memory(), cnts[i].cpu().pin_memory()]
               for i in range(NB)]
    e2e_steps = min(args.steps, 64)
    e2e_ms = e2e_loop_multi(
        lambda ins, outs: ops.moe_route_balance_backward(
            d, ins[0], ins[1], ins[2], S, 1e-4, ins[3], outs[0], ws,
            dloss=dloss),
        host_in, [((T, E), torch.float32)], e2e_steps, stream)
    assert ops.moe_get_device_error(ws) == 0
    h2d = sum(t.numel() * t.element_size() for t in host_in[0])
    return {
        "metric": "tokens/s through the routing backward (gates + "
                  "sequence-wise balance loss to the router logits) at the "
                  "V3 shape on 1 B300; % of HBM roofline",
        "value": round(T * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic, seeded (logits from the routing workload; "
                "dgate ~N(0,1))",
        "config": {"workload": f"route_backward_v3: T={T} as {n_seq} "
                               f"sequences of {S}, E={E}, top-{K}",
                   "T": T, "E": E, "topk": K, "seq_len": S,
                   "l2": "8 rotating logits batches, 134 MB > L2"},
        "roofline": roof,
        "e2e": {"value": round(T * e2e_steps / (e2e_ms / 1e3), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": T * E * 4},
        "gpu_launches": args.steps,
        "clocks": clocks,
        "impl": "b300",
    }


EP_SOURCES = 8   # devices of the expert-parallel deployment


def ep_counts(P, El, T, oracle=False):
    """[P, El] rows each of P sources sends to the first device's El
    experts: the per-expert counts of each source's top-8 routing of T
    tokens of seeded logits -- moe_route on the GPU arm, the oracle's
    routing on the oracle arm (routing is bit-exact, so both see the same
    layout)."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    cfg = inputs.CONFIGS["route_v3"]
    out = np.zeros((P, El), np.int32)
    for s in range(P):
        z = inputs.random_logits(cfg, T=T, step=100 + s)
        if oracle:
            from oracle import moe_oracle as O
            r = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group,
                        cfg.topk)
            out[s] = O.expert_counts(r["idx"], cfg.E)[:El]
        else:
            import torch
            from deepseekmoe_routing_expert_moe_b300 import ops
            d = ops.dims_of(cfg, T=T)
            idx = torch.empty((T, cfg.topk), dtype=torch.int32, device="cuda")
            gate = torch.empty((T, cfg.topk), dtype=torch.float32,
                               device="cuda")
            cnt = torch.empty(cfg.E, dtype=torch.int32, device="cuda")
            ws = ops.workspace(d, ops.MOE_WS_ROUTE)
            ops.moe_route(d, torch.from_numpy(z).cuda(),
                          torch.from_numpy(inputs.bias(cfg)).cuda(), idx,
                          gate, cnt, ws)
            out[s] = cnt.cpu().numpy()[:El]
    return out


def run_ep_gpu(args, rank, world, local_rank):
    """Expert parallelism's receive side at the V3 shape: one device of an
    8-way deployment (32 local experts of 256) at T = 4096 tokens per
    source.  Per step: moe_ep_plan on the [8, 32] counts the sources send,
    moe_ep_permute_rows of the received bf16 rows into expert-major order
    (the grouped GEMM's segments) and of the expert outputs back into
    source-major order for the return trip.  One GPU: the exchange itself
    is not part of the step; the received rows are resident (470 MB, larger
    than L2)."""
    import torch
    from deepseekmoe_routing_expert_moe_b300 import inputs, ops
    torch.cuda.set_device(local_rank)
    cfg = inputs.CONFIGS["prefill_v3"]
    T, E, H = cfg.T, cfg.E, cfg.H
    P = EP_SOURCES
    El = E // P
    counts = ep_counts(P, El, T)
    rows = int(counts.sum())
    cnt_d = torch.from_numpy(counts).cuda()
    g = torch.Generator(device="cuda").manual_seed(17 + rank)
    xr = (torch.randn((rows, H), device="cuda", generator=g)
          .to(torch.bfloat16).view(torch.int16))
    perm = torch.empty(rows, dtype=torch.int32, device="cuda")
    off = torch.empty(El + 1, dtype=torch.int32, device="cuda")
    xe = torch.empty_like(xr)
    yb = torch.empty_like(xr)
    ws = torch.zeros(256, dtype=torch.uint8, device="cuda")
    stream = torch.cuda.current_stream()

    def step(src, dst):
        ops.moe_ep_plan(cnt_d, rows, perm, off, ws=ws)
        ops.moe_ep_permute_rows(src, perm, xe, inverse=False, ws=ws)
        ops.moe_ep_permute_rows(xe, perm, dst, inverse=True, ws=ws)

    for _ in range(args.warmup):
        step(xr, yb)
    torch.cuda.synchronize()
    assert ops.moe_get_device_error(ws) == 0
    assert torch.equal(yb, xr)      # the return trip restores the order
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index_for_smi(local_rank)) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        for _ in range(args.steps):
            step(xr, yb)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    clocks = clk.summary()
    row_b = H * 2
    alg = (P * El * 4 + rows * 4 + (El + 1) * 4 +      # the plan
           2 * (2 * rows * row_b + rows * 4))           # two row moves
    pk, pk_src = peaks()
    hbm = float(pk["hbm_gbs"])
    roof = {"bound": "hbm",
            "achieved": round(alg * args.steps / (ms / 1e3) / 1e9, 1),
            "peak": hbm, "unit": "GB/s"}
    roof["frac"] = round(roof["achieved"] / hbm, 4)
    roof["traffic"] = ncu_traffic("ep_step", args.workload)
    roof["kernel"] = ("ep_rows_kernel (two row moves) + ep_plan_kernel; "
                      "the moves read and write every received row once")
    roof["algorithmic_bytes"] = int(alg)
    roof["peak_source"] = f"{pk_src} (MEASURED_PEAKS.json)"
    # end to end: the received rows uploaded, the returned rows read back
    host_in = [[xr.cpu().pin_memory()]]
    e2e_steps = min(args.steps, 8)
    e2e_ms = e2e_loop_multi(lambda ins, outs: step(ins[0], outs[0]),
                            host_in, [((rows, H), torch.int16)], e2e_steps,
                            stream)
    assert ops.moe_get_device_error(ws) == 0
    return {
        "metric": "received rows/s through the expert-parallel receive "
                  "side (plan, rows to expert order and back) at the V3 "
                  "shape on 1 B300; % of HBM roofline",
        "value": round(rows * args.steps / (ms / 1e3), 1),
        "unit": "rows/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(ms / args.steps, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "bf16", "data": "synthetic, seeded (counts from routing 8 "
                                 "sources' logits; rows ~N(0,1))",
        "config": {"workload": f"ep_v3: one device of {P}-way expert "
                               f"parallelism, {El} of {E} experts, "
                               f"{rows} received rows of H={H}",
                   "sources": P, "local_experts": El, "rows": rows, "H": H,
                   "l2": "470 MB of received rows per move > L2"},
        "roofline": roof,
        "e2e": {"value": round(rows * e2e_steps / (e2e_ms / 1e3), 1),
                "unit": "rows/s", "h2d_bytes_per_step": rows * row_b,
                "d2h_bytes_per_step": rows * row_b},
        "gpu_launches": 3 * args.steps,
        "clocks": clocks,
        "impl": "b300",
    }


def run_ep_reference(args):
    """Oracle arm of ep_v3: per step the oracle's map (ep_plan) and the two
    row moves in numpy, on the same counts with rows cut to their first 1024
    of 7168 columns (a bounded sample of the bytes)."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    from oracle import moe_oracle as O
    cfg = inputs.CONFIGS["prefill_v3"]
    P = EP_SOURCES
    El = cfg.E // P
    counts = ep_counts(P, El, cfg.T, oracle=True)
    rows = int(counts.sum())
    x = np.random.default_rng(17).standard_normal((rows, 1024)).astype(
        np.float32).view(np.int32).astype(np.int16)

    def one():
        perm, _ = O.ep_plan(counts)
        xe = np.empty_like(x)
        xe[perm] = x
        return xe[perm]

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    tot = time.perf_counter() - t0
    v = rows * args.steps / tot
    sample = (f"all {rows} received rows per step, cut to 1024 of 7168 "
              "columns, through the oracle's map and numpy row moves")
    return {
        "metric": "received rows/s through the expert-parallel receive side "
                  "at the V3 shape; oracle on the host cores",
        "value": round(v, 1), "unit": "rows/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "int16 rows", "data": "synthetic, seeded",
        "config": {"workload": f"ep_v3: {P} sources, {El} local experts, "
                               f"{rows} rows (1024 columns)"},
        "impl": "reference",
        "cpu_baseline": {"value": round(v, 1), "unit": "rows/s",
                         "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 1), "unit": "rows/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_expert_backward_gpu(args, rank, world, local_rank):
    """The experts' backward at the V3 prefill size (T = 4096, 256 experts of
    7168 x 2048 + shared, top-8): per step one moe_expert_backward call --
    recompute of p, q, dgrad of the down and up projections, fp32 weight
    gradients of every expert, token and gate gradients -- for the routing
    the forward chose.  Two rotating (x, dout) batches; 22.6 GB of weights
    read and 45 GB of fp32 weight gradients written per step (> L2)."""
    import torch
    from deepseekmoe_routing_expert_moe_b300 import inputs, ops
    torch.cuda.set_device(local_rank)
    cfg = inputs.CONFIGS["prefill_v3_e16" if args.workload.endswith("_e16")
                         else "prefill_v3"]
    d = ops.dims_of(cfg)
    T, H, E, K, I, Is = cfg.T, cfg.H, cfg.E, cfg.topk, cfg.I, cfg.I_shared
    w1, w3, w2 = inputs.device_expert_weights(cfg, "cuda")
    ws1, ws3, ws2 = inputs.shared_weights(cfg, "cuda")
    wr = torch.from_numpy(inputs.router_weight(cfg)).cuda()
    W = ops.Weights(wr, w1, w3, w2, ws1, ws3, ws2)
    NB = 2
    wsf = ops.workspace(d, ops.MOE_WS_FORWARD)
    xs, dos, idxs, gates = [], [], [], []
    bias = torch.from_numpy(inputs.bias(cfg)).cuda()
    g = torch.Generator(device="cuda").manual_seed(11 + rank)
    for i in range(NB):   # the forward's routing of each batch
        x = inputs.x_tokens(cfg, step=i + 1000 * rank, device="cuda")
        out = torch.empty((T, H), dtype=torch.int16, device="cuda")
        idx = torch.empty((T, K), dtype=torch.int32, device="cuda")
        gate = torch.empty((T, K), dtype=torch.float32, device="cuda")
        ops.moe_forward(d, W, x, bias, out, wsf, topk_idx_out=idx,
                        topk_gate_out=gate)
        dout = (torch.randn((T, H), device="cuda", generator=g)
                .to(torch.bfloat16).view(torch.int16))
        xs.append(x)
        dos.append(dout)
        idxs.append(idx)
        gates.append(gate)
    del wsf
    grads = ops.WeightGrads.empty(d)
    dx = torch.empty((T, H), dtype=torch.int16, device="cuda")
    dg = torch.empty((T, K), dtype=torch.float32, device="cuda")
    ws = ops.workspace(d, ops.MOE_WS_EXPERT_BWD)
    stream = torch.cuda.current_stream()

    def step(i, xi=None, di=None, dxo=None, dgo=None):
        b = i % NB
        ops.moe_expert_backward(d, W, xs[b] if xi is None else xi,
                                dos[b] if di is None else di, idxs[b],
                                gates[b], dx if dxo is None else dxo,
                                dg if dgo is None else dgo, grads, ws)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize()
    assert ops.moe_get_device_error(ws) == 0
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(gpu_index_for_smi(local_rank)) as clk:
        torch.cuda.synchronize()
        ev0.record(stream)
        for i in range(args.steps):
            step(i)
        ev1.record(stream)
        torch.cuda.synchronize()
    ms = ev0.elapsed_time(ev1)
    clocks = clk.summary()
    # per-stage times (separate pass, events between the stages)
    ns = 6
    sets = [[torch.cuda.Event(enable_timing=True)
             for _ in range(ops.MOE_FORWARD_KERNELS + 1)]
            for _ in range(args.steps)]
    for i in range(args.steps):
        ops.moe_set_profile_events(sets[i])
        step(i)
    ops.moe_set_profile_events(None)
    torch.cuda.synchronize()
    st = np.array([[s_[j].elapsed_time(s_[j + 1]) for j in range(ns)]
                   for s_ in sets]).mean(0)
    names = ("dispatch", "recompute", "dgrad_down", "dgrad_up", "wgrad",
             "finalize")
    c = np.bincount(idxs[(args.steps - 1) % NB].cpu().numpy().ravel(),
                    minlength=E)
    touched = int((c > 0).sum())
    TK = T * K
    # algorithmic bytes / flops per stage (real rows; the 16-row padding of
    # the segments is this design's own)
    wgt = touched * I * H * 2
    stage_bytes = {
        "recompute": 2 * wgt + 2 * Is * H * 2 + (TK + T) * H * 2 +
                     (TK + T) * I * (4 + 4 + 2),
        "dgrad_down": wgt + Is * H * 2 + (TK + T) * H * 2 +
                      (TK + T) * I * (8 + 4),
        "dgrad_up": 2 * wgt + 2 * Is * H * 2 + (TK + T) * I * 4 +
                    (TK + T) * H * 2,
        "wgrad": (touched + 0.0) * 3 * I * H * 4 + 3 * Is * H * 4 +
                 (TK + T) * (2 * I * 2 + H * 2 + I * 2 + H * 2),
    }
    stage_flops = {"recompute": 2.0 * (TK + T) * H * 2 * I,
                   "dgrad_down": 2.0 * (TK + T) * H * I,
                   "dgrad_up": 2.0 * (TK + T) * H * 2 * I,
                   "wgrad": 2.0 * (TK + T) * 3 * H * I}
    pk, pk_src = peaks()
    hbm = float(pk["hbm_gbs"])
    tc = float(pk.get("bf16_tflops_sustained", pk["bf16_tflops"]))
    stages = {}
    for j, n in enumerate(names):
        e = {"ms": round(float(st[j]), 4)}
        if n in stage_bytes:
            sec = st[j] / 1e3
            e["hbm_frac"] = round(stage_bytes[n] / sec / 1e9 / hbm, 4)
            e["tensor_frac"] = round(stage_flops[n] / sec / 1e12 / tc, 4)
            e["algorithmic_bytes"] = int(stage_bytes[n])
        stages[n] = e
    dom = max(stage_bytes, key=lambda n: st[names.index(n)])
    t_dom = st[names.index(dom)] / 1e3
    if stage_bytes[dom] / (hbm * 1e9) >= stage_flops[dom] / (tc * 1e12):
        roof = {"bound": "hbm",
                "achieved": round(stage_bytes[dom] / t_dom / 1e9, 1),
                "peak": hbm, "unit": "GB/s"}
    else:
        roof = {"bound": "tensor",
                "achieved": round(stage_flops[dom] / t_dom / 1e12, 1),
                "peak": tc, "unit": "TFLOP/s"}
    roof["frac"] = round(roof["achieved"] / roof["peak"], 4)
    roof["traffic"] = ncu_traffic(dom, args.workload)
    roof["kernel"] = {"wgrad": "wgrad_gemm_kernel (fp32 dW1, dW3, dW2)",
                      "recompute": "dgrad_gemm_kernel<recompute>",
                      "dgrad_down": "dgrad_gemm_kernel<dgrad_down>",
                      "dgrad_up": "dgrad_gemm_kernel<dgrad_up>"}[dom]
    roof["algorithmic_bytes"] = int(stage_bytes[dom])
    roof["peak_source"] = f"{pk_src} (MEASURED_PEAKS.json)"
    # end to end: x and dout uploaded from pinned memory, dx and the gate
    # gradients read back every step (the weight gradients stay on the
    # device for the optimizer); the copies of neighbouring steps overlap
    # the compute (e2e_loop_multi)
    host_in = [[xs[i].cpu().pin_memory(), dos[i].cpu().pin_memory()]
               for i in range(NB)]
    cnt = [0]

    def e2e_step(ins, outs):
        step(cnt[0], ins[0], ins[1], outs[0], outs[1])
        cnt[0] += 1
    e2e_ms = e2e_loop_multi(e2e_step, host_in,
                            [((T, H), torch.int16), ((T, K), torch.float32)],
                            args.steps, stream)
    assert ops.moe_get_device_error(ws) == 0
    res = {
        "metric": "tokens/s through the experts' backward (recompute, dgrad, "
                  "fp32 weight gradients, token and gate gradients) of a "
                  "V3-shaped MoE layer on 1 B300; % of HBM roofline",
        "value": round(T * args.steps / (ms / 1e3), 1), "unit": "tokens/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms / args.steps, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic, seeded (x ~N(0,1), dout ~N(0,1) bf16, expert "
                "weights ~N(0,0.02) bf16; routing from the layer forward)",
        "config": {"workload": f"{args.workload}: experts' backward of the "
                               f"V3 prefill layer, T={T}, H={H}, E={E}+1 "
                               f"shared, I={I}, top-{K}",
                   "T": T, "H": H, "E": E, "I": I, "topk": K,
                   "l2": "22.6 GB of weights read and 45 GB of fp32 weight "
                         "gradients written per step"},
        "roofline": roof,
        "stages_ms": stages,
        "e2e": {"value": round(T * args.steps / (e2e_ms / 1e3), 1),
                "unit": "tokens/s", "h2d_bytes_per_step": 2 * T * H * 2,
                "d2h_bytes_per_step": T * H * 2 + T * K * 4},
        # block counts, count scan, dispatch order, padded dispatch (3),
        # four GEMMs, token / gate gradients
        "gpu_launches": 11 * args.steps,
        "clocks": clocks,
        "experts_touched": touched,
        "impl": "b300",
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        s = expert_backward_sample(cfg, args.cpu_sample_tokens)
        sec = expert_backward_oracle_time(s)
        res["cpu_baseline"] = {
            "value": round(args.cpu_sample_tokens / sec, 4),
            "unit": "tokens/s", "cores": blas_threads(), "kind": "oracle",
            "sample": f"first {args.cpu_sample_tokens} tokens of the batch "
                      f"through the oracle's expert backward ({sec:.1f} s: "
                      "their experts and the shared expert)"}
    return res


def expert_backward_sample(cfg, n):
    """A bounded sample for the oracle's expert backward: the first n
    tokens, their routing, a dout, and the weights of their experts."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    from oracle import moe_oracle as O
    f = inputs.bf16_bits_to_f32
    x = f(inputs.x_tokens(cfg, T=n)).astype(np.float64)
    z = O.router_logits(x, inputs.router_weight(cfg))
    r = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group, cfg.topk)
    dout = np.random.default_rng(3).standard_normal(x.shape)
    ew = {int(e): tuple(f(a) for a in inputs.expert_weights(cfg, int(e)))
          for e in np.unique(r["idx"])}
    sw = tuple(f(a) for a in inputs.shared_weights(cfg))
    return dict(x=x, dout=dout, idx=r["idx"], gate=r["gate"], ew=ew, sw=sw)


def expert_backward_oracle_time(s) -> float:
    """Seconds for the oracle's backward of the sample: the shared expert
    over every sample token and each chosen expert over its tokens
    (swiglu_ffn_backward, the piece layer_backward is built from)."""
    from oracle import moe_oracle as O
    t0 = time.perf_counter()
    x, d = s["x"], s["dout"]
    dx = d + O.swiglu_ffn_backward(x, *s["sw"], d)[0]
    for e, w in s["ew"].items():
        t, k = np.nonzero(s["idx"] == e)
        y = O.swiglu_ffn(x[t], *w)
        np.einsum("nh,nh->n", d[t], y)
        g = s["gate"][t, k].astype(np.float64)[:, None]
        dx[t] += O.swiglu_ffn_backward(x[t], *w, g * d[t])[0]
    return time.perf_counter() - t0


def run_expert_backward_reference(args):
    """Oracle arm of expert_backward_v3: a bounded token sample per step
    through the oracle's expert backward."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    cfg = inputs.CONFIGS["prefill_v3"]
    n = args.ref_tokens
    s = expert_backward_sample(cfg, n)
    for _ in range(args.warmup):
        expert_backward_oracle_time(s)
    tot = sum(expert_backward_oracle_time(s) for _ in range(args.steps))
    v = n * args.steps / tot
    return {
        "metric": "tokens/s through the experts' backward of a V3-shaped MoE "
                  "layer; oracle on the host cores",
        "value": round(v, 4), "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic, seeded",
        "config": {"workload": f"expert_backward_v3: {n} tokens per step"},
        "impl": "reference",
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s",
                         "cores": blas_threads(), "kind": "oracle",
                         "sample": f"{n} tokens of the prefill batch per step"},
        "e2e": {"value": round(v, 4), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_route_reference(args):
    """Oracle arm of route_v3: per step the first 2048 tokens of a V3
    logits batch through the oracle's routing (sigmoid, bias, group-limited
    top-8, gates), dispatch order and bias step -- the GPU arm's three
    calls on a bounded sample."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    from oracle import moe_oracle as O
    cfg = inputs.CONFIGS["route_v3"]
    n = 2048
    z = inputs.random_logits(cfg, T=n)
    bias = inputs.bias(cfg)

    def one():
        r = O.route(z, bias, cfg.n_group, cfg.topk_group, cfg.topk)
        O.permutation(r["idx"], cfg.E)
        O.bias_update(O.expert_counts(r["idx"], cfg.E), bias, n, cfg.topk,
                      cfg.gamma)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    tot = time.perf_counter() - t0
    v = n * args.steps / tot
    sample = (f"the first {n} tokens of a logits batch per step through the "
              "numpy oracle (routing, dispatch order, bias step)")
    return {
        "metric": "tokens/s routed (routing + dispatch order + bias step) "
                  "at the V3 shape; oracle on the host cores",
        "value": round(v, 1), "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic, seeded",
        "config": {"workload": f"route_v3: routing-only, {n} of the "
                               f"{cfg.T} tokens per step, E={cfg.E}, "
                               f"top-{cfg.topk}"},
        "impl": "reference",
        "cpu_baseline": {"value": round(v, 1), "unit": "tokens/s",
                         "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def cpu_baseline_from_reference(args):
    """The cpu_baseline object of a GPU line whose runner times no oracle
    itself: the workload's oracle arm (its bounded sample, the oracle as it
    stands) for a few steps (about 10-30 s of host time)."""
    import copy
    a = copy.copy(args)
    a.impl = "reference"
    # ~10 s of routing samples; an FP8 layer token takes ~10-20 s alone
    a.steps = {"route_v3": 400, "route_backward_v3": 100,
               "ep_v3": 200}.get(args.workload, 1)
    a.warmup = 1 if a.steps > 1 else 0
    r = run_reference(a)
    cb = dict(r["cpu_baseline"])
    cb["sample"] = f"{cb['sample']}; {a.steps} steps"
    return cb


def run_backward_reference(args):
    """Oracle arm of route_backward_v3: one 4096-token sequence of V3
    logits per step through the oracle's gate and balance-loss gradients."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    from oracle import moe_oracle as O
    cfg = inputs.CONFIGS["route_v3"]
    S = 4096
    z = inputs.random_logits(cfg, T=S)
    idx = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group,
                  cfg.topk)["idx"]
    dg = np.random.default_rng(5).standard_normal((S, cfg.topk))

    def one():
        O.route_backward(z, idx, dg)
        O.seq_balance_loss_backward(z, S, cfg.topk)

    for _ in range(args.warmup):
        one()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        one()
    tot = time.perf_counter() - t0
    v = S * args.steps / tot
    return {
        "metric": "tokens/s through the routing backward at the V3 shape; "
                  "oracle on the host cores",
        "value": round(v, 1), "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic, seeded",
        "config": {"workload": f"route_backward_v3: one sequence of {S}"},
        "impl": "reference",
        "cpu_baseline": {"value": round(v, 1), "unit": "tokens/s",
                         "cores": blas_threads(), "kind": "oracle",
                         "sample": f"one {S}-token sequence per step"},
        "e2e": {"value": round(v, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_balance_reference(args):
    """Oracle arm of balance_v3: one 4096-token sequence of V3-shaped
    logits per step through the oracle's balance loss."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    from oracle import moe_oracle as O
    cfg = inputs.CONFIGS["route_v3"]
    S = 4096
    z = inputs.random_logits(cfg, T=S)
    for _ in range(args.warmup):
        O.seq_balance_loss(z, S, cfg.topk)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        O.seq_balance_loss(z, S, cfg.topk)
    tot = time.perf_counter() - t0
    v = S * args.steps / tot
    sample = f"one {S}-token sequence per step through the numpy oracle"
    return {
        "metric": "tokens/s through the sequence-wise balance loss (eq. "
                  "17-20) at the V3 shape; oracle on the host cores",
        "value": round(v, 1), "unit": "tokens/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic, seeded",
        "config": {"workload": f"balance_v3: sequence-wise balance loss, "
                               f"one sequence of {S}, E={cfg.E}, "
                               f"top-{cfg.topk}"},
        "impl": "reference",
        "cpu_baseline": {"value": round(v, 1), "unit": "tokens/s",
                         "cores": blas_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(v, 1), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def run_reference(args):
    """The oracle arm: the CPU oracle as it stands, per step one bounded
    sample of the workload (the same tokens every step)."""
    from deepseekmoe_routing_expert_moe_b300 import inputs
    if args.workload == "balance_v3":
        return run_balance_reference(args)
    if args.workload in FP8_WORKLOADS:
        return run_decode_fp8_reference(args)
    if args.workload == "route_backward_v3":
        return run_backward_reference(args)
    if args.workload == "route_v3":
        return run_route_reference(args)
    if args.workload == "ep_v3":
        return run_ep_reference(args)
    if args.workload in ("expert_backward_v3", "expert_backward_v3_e16"):
        return run_expert_backward_reference(args)
    cfg = inputs.CONFIGS[args.workload]
    n = args.ref_tokens
    s = oracle_sample(cfg, n)
    for _ in range(args.warmup):
        oracle_time(cfg, s)
    times = [oracle_time(cfg, s) for _ in range(args.steps)]
    tot = sum(times)
    v = n * args.steps / tot
    cores = blas_threads()
    sample = (f"{n} tokens of the {cfg.name} batch per step through the numpy "
              "fp64 oracle (logits, routing, bias step, experts, combine)")
    return {
        "metric": METRIC, "value": round(v, 4), "unit": "tokens/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot / args.steps * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f64", "data": "synthetic, seeded",
        "config": config_json(cfg, 1),
        "impl": "reference",
        "cpu_baseline": {"value": round(v, 4), "unit": "tokens/s",
                         "cores": cores, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(v, 4), "unit": "tokens/s",
                "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=("b300", "reference"), default="b300")
    ap.add_argument("--workload", default="prefill_v3",
                    choices=("prefill_v3", "decode_v3", "skewed_v3",
                             "route_v3", "prefill_v3_e32", "balance_v3",
                             *FP8_WORKLOADS,
                             "route_backward_v3", "ep_v3",
                             "expert_backward_v3", "expert_backward_v3_e16"))
    ap.add_argument("--cpu-sample-tokens", type=int, default=4)
    ap.add_argument("--ref-tokens", type=int, default=1)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl")
    if args.workload == "route_v3":
        res = run_route_gpu(args, rank, world, local_rank)
    elif args.workload == "balance_v3":
        res = run_balance_gpu(args, rank, world, local_rank)
    elif args.workload in FP8_WORKLOADS:
        res = run_fp8_gpu(args, rank, world, local_rank)
    elif args.workload == "route_backward_v3":
        res = run_backward_gpu(args, rank, world, local_rank)
    elif args.workload == "ep_v3":
        res = run_ep_gpu(args, rank, world, local_rank)
    elif args.workload in ("expert_backward_v3", "expert_backward_v3_e16"):
        res = run_expert_backward_gpu(args, rank, world, local_rank)
    else:
        res = run_gpu(args, rank, world, local_rank)
    if (rank == 0 and world == 1 and not args.no_cpu_baseline and
            "cpu_baseline" not in res):
        res["cpu_baseline"] = cpu_baseline_from_reference(args)
    if rank == 0:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
