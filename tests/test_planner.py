"""Redundant-expert placement ("02 · DeepSeek-V3" §5.1: high-load experts
replicated from online load statistics, one extra expert per GPU).  No GPU:
the planner is host code.

Oracle pins (a hand-worked example, the accounting recomputed from the
returned slot table, invariants, degenerate cases) and bit-exact parity of
the library's native planner with the oracle over many random loads."""
import numpy as np
import pytest

from deepseekmoe_routing_expert_moe_b300 import build, inputs, ops
from oracle import moe_oracle as O


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.lib()


def test_worked_example():
    """E = 8 on D = 4 devices (2 each), one slot per device.
    Loads 10 50 3 7 40 1 2 30 -> device loads 60 10 41 32.
    Heaviest first: e1 (50, home d0): free d1..d3, least loaded d1 (10):
      d0 60-25 = 35, d1 10+25 = 35.
    e4 (40, home d2): free d0, d3 -> d3 (32 < 35): d2 41-20 = 21, d3 52.
    e7 (30, home d3): free d0, d2 -> d2 (21): d3 52-15 = 37, d2 36.
    e0 (10, home d0): the only free slot is on d0 -> passed over.
    e3 (7, home d1): free d0 -> d0: d1 35-3 = 32, d0 35+3 = 38."""
    p = O.plan_redundant_experts(np.array([10, 50, 3, 7, 40, 1, 2, 30]),
                                 4, 1)
    assert p["slot_expert"].ravel().tolist() == [3, 1, 7, 4]
    assert p["device_load"].tolist() == [38, 32, 36, 37]
    assert p["base_load"].tolist() == [60, 10, 41, 32]
    assert p["replicated"].tolist() == [1, 4, 7, 3]


def _recount(load, slots, D):
    """Device loads from the slot table alone: every original keeps
    ceil(c/2) if copied, else c; every copy serves floor(c/2)."""
    E = len(load)
    per = E // D
    copied = {int(e) for e in slots.ravel() if e >= 0}
    dev = np.zeros(D, np.int64)
    for e in range(E):
        dev[e // per] += (load[e] + 1) // 2 if e in copied else load[e]
    for d in range(D):
        for e in slots[d]:
            if e >= 0:
                dev[d] += load[e] // 2
    return dev


def _random_cases():
    g = np.random.default_rng(0)
    cases = [(256, 32, 1), (256, 64, 1), (256, 8, 4), (64, 16, 2), (8, 4, 1),
             (16, 1, 3), (32, 32, 1), (12, 3, 0), (256, 256, 1)]
    for E, D, r in cases:
        for k in range(6):
            kind = k % 3
            if kind == 0:      # Zipf-like skew
                load = (4000 * (g.permutation(E) + 1.0) ** -1.2).astype(
                    np.int64)
            elif kind == 1:    # many ties and zeros
                load = g.integers(0, 4, E).astype(np.int64)
            else:
                load = g.integers(0, 10 ** 6, E).astype(np.int64)
            yield E, D, r, kind, load


@pytest.mark.parametrize("case", list(_random_cases()))
def test_invariants(case):
    E, D, r, kind, load = case
    p = O.plan_redundant_experts(load, D, r)
    slots = p["slot_expert"]
    per = E // D
    assert slots.shape == (D, r)
    used = slots[slots >= 0]
    assert len(set(used.tolist())) == len(used)            # one copy at most
    for d in range(D):
        assert all(e // per != d for e in slots[d] if e >= 0)   # not at home
    assert p["device_load"].sum() == load.sum()              # conserved
    np.testing.assert_array_equal(p["device_load"], _recount(load, slots, D))
    assert all(load[e] > 0 for e in used)
    # copies go to the heaviest experts that can be placed: an expert
    # heavier than a copied one was passed over only if, at its turn, every
    # free slot was on its own device -- so every other device ends full
    if len(used):
        lightest = min(load[e] for e in used)
        for e in range(E):
            if load[e] > lightest and e not in used:
                others = np.delete(slots, e // per, axis=0)
                assert np.all(others >= 0), (e, load[e], lightest)
    if kind == 0:   # skewed loads: the hottest device only gets lighter
        assert p["device_load"].max() <= p["base_load"].max()


def test_degenerate_cases():
    load = np.arange(16, dtype=np.int64)
    p = O.plan_redundant_experts(load, 4, 0)                 # no slots
    assert p["slot_expert"].shape == (4, 0)
    np.testing.assert_array_equal(p["device_load"], p["base_load"])
    p = O.plan_redundant_experts(load, 1, 2)                 # one device
    assert np.all(p["slot_expert"] == -1)
    p = O.plan_redundant_experts(np.zeros(16, np.int64), 4, 1)
    assert np.all(p["slot_expert"] == -1)


def test_skewed_v3_loads_balance_over_32_devices():
    """The skewed workload's routing (Zipf preference) on 2048 tokens,
    planned as the pages' prefill deployment: 32 devices x 8 experts plus
    one redundant slot each.  The hottest device's load drops."""
    cfg = inputs.CONFIGS["skewed_v3"]
    T = 2048
    x = inputs.bf16_bits_to_f32(inputs.x_tokens(cfg, T=T))
    z = O.router_logits(x, inputs.router_weight(cfg),
                        inputs.zipf_preference(cfg))
    idx = O.route(z, np.zeros(cfg.E, np.float32), cfg.n_group,
                  cfg.topk_group, cfg.topk)["idx"]
    load = O.expert_counts(idx, cfg.E).astype(np.int64)
    p = O.plan_redundant_experts(load, 32, 1)
    mean = load.sum() / 32
    before = p["base_load"].max() / mean
    after = p["device_load"].max() / mean
    assert (p["slot_expert"] >= 0).all()
    assert after < before and after < 2.0, (before, after)


@pytest.mark.parametrize("case", list(_random_cases()))
def test_library_matches_oracle(lib, case):
    E, D, r, _, load = case
    p = O.plan_redundant_experts(load, D, r)
    slots, dl = ops.moe_plan_redundant_experts(load, D, r)
    np.testing.assert_array_equal(slots, p["slot_expert"])
    np.testing.assert_array_equal(dl, p["device_load"])


def test_library_rejects_bad_arguments(lib):
    load = np.ones(8, np.int64)
    slots = np.zeros(8, np.int32)
    dl = np.zeros(8, np.int64)
    f = lib.moe_plan_redundant_experts
    P = lambda a: a.ctypes.data          # noqa: E731
    assert f(P(load), 8, 3, 1, P(slots), P(dl)) == 1         # E % D
    assert f(None, 8, 4, 1, P(slots), P(dl)) == 1
    assert f(P(load), 8, 4, 1, None, P(dl)) == 1
    assert f(P(load), 8, 4, 0, None, P(dl)) == 0             # no slots
    assert f(P(load), 8, 0, 1, P(slots), P(dl)) == 1
    bad = load.copy()
    bad[3] = -1
    assert f(P(bad), 8, 4, 1, P(slots), P(dl)) == 1
