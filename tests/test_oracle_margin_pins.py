"""Pins for ``oracle.routing_margins`` (no GPU).

The margins decide which tokens the layer-output parity tests compare: a
token whose top-K margin u_(K) - u_(K+1) (over the kept groups' experts) or
group margin S_(M) - S_(M+1) is tiny may legitimately route differently when
the GPU's fp32 logits differ from the oracle's by rounding.  So the margins
are tied here to things other than their own formula:

* the hand-worked example of the routing rule ("02 · DeepSeek-V3" §1.3
  group-limited top-K, §1.4 bias for selection), whose margins are worked
  by hand in tests/golden/routing_worked_example.json;
* a second formulation: min over the chosen experts' u minus max over the
  kept-but-unchosen experts' u, and min over the kept groups' S minus max
  over the dropped groups' S;
* their meaning: a margin is the distance to a different decision -- lifting
  the best unchosen kept expert (or the best dropped group) by more than the
  margin changes the selection, lifting it by less does not;
* the degenerate cases: every group kept (M = G) or every kept expert chosen
  (K = M * E / G) gives an infinite margin.

A slip such as sorting ascending, taking the top-K margin over all experts
instead of the kept ones, or reading the wrong axis fails at least one."""
import json
import os

import numpy as np
import pytest

from oracle import moe_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def test_worked_example_margins():
    with open(os.path.join(GOLD, "routing_worked_example.json")) as f:
        g = json.load(f)
    z = np.array([g["logits"]], F32)
    for case in g["cases"]:
        r = O.route(z, np.array(case["bias"], F32), g["n_group"],
                    g["topk_group"], g["topk"])
        km, gm = O.routing_margins(r, g["topk_group"], g["topk"])
        want = case["margins"]
        assert abs(km[0] - want["topk"]) <= 2e-6, (km[0], want)
        assert abs(gm[0] - want["group"]) <= 2e-6, (gm[0], want)


def _second_formulation(r, n_group, topk):
    """min(chosen u) - max(kept, unchosen u); min(kept S) - max(dropped S)."""
    u = r["u"].astype(np.float64)
    S = r["group_score"].astype(np.float64)
    T, E = u.shape
    gs = E // n_group
    km = np.full(T, np.inf)
    gm = np.full(T, np.inf)
    for t in range(T):
        chosen = set(r["idx"][t].tolist())
        kept = np.nonzero(r["kept"][t])[0]
        rest = [e for e in range(E) if e // gs in kept and e not in chosen]
        if rest:
            km[t] = min(u[t, e] for e in chosen) - max(u[t, e] for e in rest)
        dropped = [q for q in range(n_group) if not r["kept"][t, q]]
        if dropped:
            gm[t] = min(S[t, q] for q in kept) - max(S[t, q] for q in dropped)
    return km, gm


SHAPES = [(8, 2, 1, 2), (12, 3, 2, 3), (16, 4, 2, 4), (16, 4, 3, 5),
          (32, 8, 4, 8), (64, 8, 4, 8)]


@pytest.mark.parametrize("E,G,M,K", SHAPES)
def test_margins_equal_a_second_formulation(E, G, M, K):
    rng = np.random.default_rng(E * 100 + K)
    T = 40
    z = rng.normal(0, 1, size=(T, E)).astype(F32)
    b = rng.uniform(-0.05, 0.05, size=E).astype(F32)
    r = O.route(z, b, G, M, K)
    km, gm = O.routing_margins(r, M, K)
    km2, gm2 = _second_formulation(r, G, K)
    np.testing.assert_array_equal(km, km2)
    np.testing.assert_array_equal(gm, gm2)
    assert np.all(km >= 0) and np.all(gm >= 0)


def _route_one(z_row, b, G, M, K):
    return O.route(z_row[None, :], b, G, M, K)


@pytest.mark.parametrize("E,G,M,K", SHAPES)
def test_margin_is_the_distance_to_a_different_selection(E, G, M, K):
    """Lift the best unchosen kept expert by 2x its top-K margin: it gets
    chosen.  Lift it by half the margin: the chosen set stays.  Likewise
    lifting every expert of the best dropped group by the group margin
    (its score rises by twice that) keeps the group; by a quarter of it
    (half the margin) does not."""
    rng = np.random.default_rng(7 * E + M)
    gs = E // G
    z = rng.normal(0, 1, size=(30, E)).astype(F32)
    b = rng.uniform(-0.05, 0.05, size=E).astype(F32)
    r = O.route(z, b, G, M, K)
    km, gm = O.routing_margins(r, M, K)
    checked_k = checked_g = 0
    for t in range(z.shape[0]):
        chosen = set(r["idx"][t].tolist())
        kept = set(np.nonzero(r["kept"][t])[0].tolist())
        u = r["u"][t].astype(np.float64)
        if np.isfinite(km[t]) and km[t] > 1e-3:
            rest = [e for e in range(E) if e // gs in kept and e not in chosen]
            e_next = max(rest, key=lambda e: (u[e], -e))
            for lift, flips in ((2.0, True), (0.5, False)):
                bb = b.copy()
                bb[e_next] = F32(bb[e_next] + F32(lift * km[t]))
                r2 = _route_one(z[t], bb, G, M, K)
                assert (e_next in r2["idx"][0].tolist()) == flips, (t, lift)
                if not flips:
                    assert set(r2["idx"][0].tolist()) == chosen
            checked_k += 1
        if np.isfinite(gm[t]) and gm[t] > 1e-3:
            S = r["group_score"][t].astype(np.float64)
            g_next = max((q for q in range(G) if q not in kept),
                         key=lambda q: (S[q], -q))
            for lift, flips in ((1.0, True), (0.25, False)):
                bb = b.copy()
                bb[g_next * gs:(g_next + 1) * gs] += F32(lift * gm[t])
                r2 = _route_one(z[t], bb, G, M, K)
                assert bool(r2["kept"][0, g_next]) == flips, (t, lift)
                if not flips:
                    assert set(np.nonzero(r2["kept"][0])[0].tolist()) == kept
            checked_g += 1
    assert checked_k > 0
    assert checked_g > 0 or M == G


def test_all_groups_kept_and_all_kept_experts_chosen_give_infinite_margins():
    rng = np.random.default_rng(3)
    z = rng.normal(0, 1, size=(25, 16)).astype(F32)
    b = np.zeros(16, F32)
    # M = G: no group is dropped
    r = O.route(z, b, 4, 4, 3)
    km, gm = O.routing_margins(r, 4, 3)
    assert np.all(np.isinf(gm)) and np.all(np.isfinite(km))
    # K = M * E / G: every kept expert is chosen
    r = O.route(z, b, 4, 2, 8)
    km, gm = O.routing_margins(r, 2, 8)
    assert np.all(np.isinf(km)) and np.all(np.isfinite(gm))


def test_exact_tie_gives_zero_margin():
    """Two kept experts with the same u straddling the K-th slot: margin 0
    (the worked example's first case is one; here on a random row)."""
    z = np.array([[0.3, 0.3, -1.0, 0.9, -2.0, -2.5, -3.0, -3.5]], F32)
    r = O.route(z, np.zeros(8, F32), 2, 1, 2)
    km, gm = O.routing_margins(r, 1, 2)
    assert km[0] == 0.0
    assert gm[0] > 0
