"""Data-parallel replicas on CPU (gloo, world size 2).

The layer shards by token: each replica routes its own tokens.  The bias
step balances the load of the whole batch ("02 · DeepSeek-V3" §1.4), so a
data-parallel step needs one exchange -- a sum of the E-entry count vector
-- after which every replica applies the same +-gamma step.  This checks,
with the oracle on two gloo ranks, that the all-reduced shard histograms
equal the unsharded batch's and that both ranks end with the bias of the
unsharded run, bit for bit; that every rank derives the same
redundant-expert plan (§5.1) from the all-reduced load, equal to the plan of
the unsharded batch; and that the bench's max-over-ranks timing reduction
picks the slowest rank."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    sys.path.insert(0, root)
    from deepseekmoe_routing_expert_moe_b300 import inputs
    from oracle import moe_oracle as O
    cfg = inputs.CONFIGS["route_v3"]
    T = 2048
    z = inputs.random_logits(cfg, T=T)
    b = inputs.bias(cfg)
    shard = z[rank * T // world:(rank + 1) * T // world]
    r = O.route(shard, b, cfg.n_group, cfg.topk_group, cfg.topk)
    c = torch.from_numpy(O.expert_counts(r["idx"], cfg.E).astype(np.int64))
    dist.all_reduce(c, op=dist.ReduceOp.SUM)
    nb, _ = O.bias_update(c.numpy(), b, T, cfg.topk, cfg.gamma)
    plan = O.plan_redundant_experts(c.numpy(), 32, 1)["slot_expert"]
    t = torch.tensor([1.0 + rank], dtype=torch.float64)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    q.put((rank, c.numpy(), nb, plan, float(t)))
    dist.destroy_process_group()


def test_sharded_counts_and_bias_step_match_the_whole_batch():
    world = 2
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, world, port, q))
          for r in range(world)]
    for p in ps:
        p.start()
    res = [q.get(timeout=120) for _ in range(world)]
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0

    from deepseekmoe_routing_expert_moe_b300 import inputs
    from oracle import moe_oracle as O
    cfg = inputs.CONFIGS["route_v3"]
    z = inputs.random_logits(cfg, T=2048)
    b = inputs.bias(cfg)
    r = O.route(z, b, cfg.n_group, cfg.topk_group, cfg.topk)
    c_all = O.expert_counts(r["idx"], cfg.E)
    nb_all, _ = O.bias_update(c_all, b, 2048, cfg.topk, cfg.gamma)
    plan_all = O.plan_redundant_experts(c_all.astype(np.int64), 32, 1)[
        "slot_expert"]
    for rank, c, nb, plan, tmax in res:
        assert np.array_equal(c, c_all)
        assert np.array_equal(nb.view(np.uint32), nb_all.view(np.uint32))
        assert np.array_equal(plan, plan_all)
        assert tmax == 2.0
