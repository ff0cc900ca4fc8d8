"""The C ABI's host validation under seeded random invalid calls (no GPU).

Every device entry point validates its arguments on the host before it
launches anything (include/moe.h).  Each call below breaks at least one
documented rule -- a misaligned or NULL required pointer, a too-small
workspace, or an invalid dimension -- with T > 0, so it must come back with
MOE_ERR_INVALID_ARG, _UNSUPPORTED, _ALIGNMENT or _WORKSPACE: never MOE_OK
(work accepted) and never MOE_ERR_CUDA (a CUDA call reached, which on a
machine without a GPU is what a launch would return)."""
import ctypes

import numpy as np
import pytest

from deepseekmoe_routing_expert_moe_b300 import build, ops

A = 1 << 20          # a 16-byte aligned address, never dereferenced
V3 = dict(T=4096, H=7168, E=256, n_group=8, topk_group=4, topk=8, I=2048,
          I_shared=2048, gamma=0.001)
VALIDATION = {1, 2, 3, 4}


@pytest.fixture(scope="module")
def L():
    build.build()
    return ops.lib()


def _breakers(g):
    """(dims overrides, pointer fault) pairs; exactly one kind of fault."""
    kind = g.integers(0, 4)
    if kind == 0:     # an invalid dimension
        bad = [dict(E=255), dict(topk=0), dict(n_group=3), dict(H=100),
               dict(topk_group=9), dict(E=2048, n_group=32),
               dict(gamma=float("inf")), dict(topk=200),
               dict(I=0), dict(I_shared=-64), dict(H=-64)]
        return bad[g.integers(0, len(bad))], None
    if kind == 1:
        return {}, "misaligned"
    if kind == 2:
        return {}, "null"
    return {}, "small_ws"


def _calls(L, d, fault, which, ws_bytes):
    """(pointer count, call taking the pointer picker) per entry point; the
    fault hits pointer `which % count` of that entry point."""
    by = ctypes.byref

    def picker(n):
        k = which % n

        def P(i):
            if fault == "misaligned" and i == k:
                return A + 4
            if fault == "null" and i == k:
                return None
            return A
        return P

    def weights(P):
        return ops.MoeWeights(*(P(i) for i in range(7)), A)

    def weights8(P):
        return ops.MoeWeightsFp8(*(P(i) for i in range(12)))

    def weightsmx(P):
        return ops.MoeWeightsMx(*(P(i) for i in range(12)))

    table = {
        "moe_route": (5, lambda P: L.moe_route(
            by(d), P(0), P(1), P(2), P(3), P(4), A, ws_bytes, None)),
        "moe_permute": (4, lambda P: L.moe_permute(
            by(d), A, P(0), P(1), P(2), P(3), A, A, ws_bytes, None)),
        "moe_expert_ffn": (7, lambda P: L.moe_expert_ffn(
            by(d), by(weights(P)), A, A, A, A, A, A, ws_bytes, None)),
        "moe_combine": (6, lambda P: L.moe_combine(
            by(d), P(0), P(1), P(2), P(3), P(4), P(5), None)),
        "moe_forward": (7, lambda P: L.moe_forward(
            by(d), by(weights(P)), A, A, 1, A, None, None, None, None, None,
            A, ws_bytes, None)),
        "moe_router_logits": (3, lambda P: L.moe_router_logits(
            by(d), P(0), P(1), None, P(2), A, ws_bytes, None)),
        "moe_seq_balance_loss": (4, lambda P: L.moe_seq_balance_loss(
            by(d), P(0), 512, 1e-4, P(1), P(2), P(3), A, ws_bytes, None)),
        "moe_permute_fp8": (6, lambda P: L.moe_permute_fp8(
            by(d), P(0), P(1), P(2), P(3), P(4), P(5), A, ws_bytes, None)),
        "moe_expert_ffn_fp8": (12, lambda P: L.moe_expert_ffn_fp8(
            by(d), by(weights8(P)), A, A, A, A, A, A, A, A, ws_bytes, None)),
        "moe_permute_mx": (6, lambda P: L.moe_permute_mx(
            by(d), P(0), P(1), P(2), P(3), P(4), P(5), A, ws_bytes, None)),
        "moe_expert_ffn_mx": (12, lambda P: L.moe_expert_ffn_mx(
            by(d), by(weightsmx(P)), A, A, A, A, A, A, A, A, ws_bytes, None)),
        "moe_route_backward": (4, lambda P: L.moe_route_backward(
            by(d), P(0), P(1), P(2), 0, P(3), A, ws_bytes, None)),
        "moe_route_balance_backward": (5, lambda P: L.moe_route_balance_backward(
            by(d), P(0), P(1), P(2), 64, 1e-4, P(3), None, 0, P(4), A,
            ws_bytes, None)),
    }
    return {n: (lambda f=f, c=c: f(picker(c))) for n, (c, f) in table.items()}


@pytest.mark.parametrize("seed", range(60))
def test_invalid_calls_are_rejected_before_any_launch(L, seed):
    g = np.random.default_rng(seed)
    over, fault = _breakers(g)
    d = ops.dims(**dict(V3, **over))
    which = int(g.integers(0, 12))
    ws_bytes = 64 if fault == "small_ws" else 1 << 40
    ffn = {"moe_expert_ffn", "moe_forward", "moe_expert_ffn_fp8",
           "moe_expert_ffn_mx"}
    for name, call in _calls(L, d, fault, which, ws_bytes).items():
        if fault == "small_ws" and name == "moe_combine":
            continue                      # takes no workspace
        if set(over) & {"I", "I_shared"} and name not in ffn:
            continue                      # the FFN widths concern the FFNs
        code = call()
        assert code in VALIDATION, (name, over, fault, which, code)
