"""moe_route_static_scratch: routing for callers that cannot allocate.

Some callers cannot give the library device memory beyond inputs and
outputs (a plugin whose host framework owns every allocation and offers no
scratch; a loop that may not call cudaMalloc after start-up).  The
workspace-free entry point keeps routing's scratch in a static device array.
Here it is called through the C ABI twice in a row, on different inputs (so
stale scratch contents from the first call would show), and each result must
equal moe_route's with a caller workspace -- bit for bit, the tolerance of
every routing test.  This file is collected last on purpose."""
import numpy as np
import pytest
import torch

from deepseekmoe_routing_expert_moe_b300 import inputs, ops

pytestmark = pytest.mark.gpu


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _outs(T, K, E):
    return (torch.full((T, K), -1, dtype=torch.int32, device="cuda"),
            torch.full((T, K), -1.0, dtype=torch.float32, device="cuda"),
            torch.full((E,), -1, dtype=torch.int32, device="cuda"))


def test_static_scratch_route_equals_workspace_route_twice():
    cfg = inputs.CONFIGS["route_v3"]          # 16384 tokens, V3 routing
    d = ops.dims_of(cfg)
    T, K, E = cfg.T, cfg.topk, cfg.E
    b = _dev(inputs.bias(cfg))
    ws = ops.workspace(d, ops.MOE_WS_ROUTE)
    for step in (0, 1):                       # two calls in a row
        z = _dev(inputs.random_logits(cfg, step=step, scale=0.5 + step))
        ref = _outs(T, K, E)
        ops.moe_route(d, z, b, *ref, ws)
        got = _outs(T, K, E)
        ops.moe_route_static_scratch(d, z, b, *got)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            assert torch.equal(g.view(torch.int32), r.view(torch.int32)), step
        assert int(got[2].sum()) == T * K


def test_static_scratch_route_small_then_ragged():
    """A shorter batch after a longer one reads only what it wrote."""
    cfg = inputs.CONFIGS["route_v3"]
    b = _dev(inputs.bias(cfg))
    for T in (4097, 65):
        d = ops.dims_of(cfg, T=T)
        z = _dev(inputs.random_logits(cfg, T=T, step=T))
        ref = _outs(T, cfg.topk, cfg.E)
        ops.moe_route(d, z, b, *ref, ops.workspace(d, ops.MOE_WS_ROUTE))
        got = _outs(T, cfg.topk, cfg.E)
        ops.moe_route_static_scratch(d, z, b, *got)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            assert torch.equal(g.view(torch.int32), r.view(torch.int32)), T


def test_static_scratch_route_rejects_batches_beyond_its_limit():
    cfg = inputs.CONFIGS["route_v3"]
    d = ops.dims_of(cfg, T=65536 + 64)        # ceil(T/64) * 256 > 262144
    one = torch.zeros(16, dtype=torch.int32, device="cuda")
    with pytest.raises(ops.MoeError) as ei:
        ops.moe_route_static_scratch(d, one, one, one, one, one)
    assert ei.value.code == ops.STATUS_CODES["MOE_ERR_WORKSPACE"]
