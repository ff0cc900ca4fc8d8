"""Pins for the CPU oracle (no GPU).

Each test ties a part of the oracle to something other than the oracle
itself: a closed form, a hand-worked example, brute-force enumeration on a
tiny input, an invariant the pages state, or a textbook reduction to a
library routine.  They are chosen so that a plausible slip in the oracle (a
dropped term, a wrong sign or index, a transposed operand, gates taken from
the biased score, groups scored by max instead of top-2 sum, an unstable
permutation) fails at least one of them.
"""
import itertools
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest
from scipy.special import expit

from deepseekmoe_routing_expert_moe_b300 import inputs
from oracle import moe_oracle as O

GOLD = os.path.join(os.path.dirname(__file__), "golden")
F32 = np.float32


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ------------------------------------------------------------------ sigmoid
def test_sig32_within_3_ulp_of_exact_sigmoid():
    """S1 against sigma in fp64 (scipy's expit) on a dense grid: the op
    sequence (Cody-Waite reduction, degree-7 Taylor, rounded steps) is
    accurate to <= 3 ulp of the result wherever it is not clamped."""
    z = np.linspace(-80.0, 40.0, 1_200_001).astype(F32)
    s = O.sig32(z).astype(np.float64)
    ex = expit(z.astype(np.float64))
    ulp = np.spacing(O.sig32(z)).astype(np.float64)
    assert np.max(np.abs(s - ex) / ulp) <= 3.0


def test_sig32_special_values():
    assert O.sig32(F32(0.0)) == F32(0.5)
    out = O.sig32(np.array([np.inf, 1e30, -np.inf, np.nan], F32))
    assert out[0] == 1.0 and out[1] == 1.0 and out[3] == 1.0
    assert 0.0 < out[2] < 1e-34          # clamped at z = -80, still normal
    # monotone non-decreasing on a grid
    z = np.linspace(-20, 20, 200001).astype(F32)
    assert np.all(np.diff(O.sig32(z)) >= 0)


def test_sig32_symmetry():
    """sigma(z) + sigma(-z) = 1 to a few ulp."""
    z = np.linspace(-15, 15, 30001).astype(F32)
    tot = O.sig32(z).astype(np.float64) + O.sig32(-z).astype(np.float64)
    assert np.max(np.abs(tot - 1.0)) < 4 * 2.0 ** -24


def test_sig32_constants_from_mathematics():
    # the two-part split carries ln 2 to ~ 2^-43 (LN2_LO is an fp32 number)
    assert abs(float(O.LN2_HI) + float(O.LN2_LO) - math.log(2)) < 2.0 ** -43
    # LN2_HI has at most 16 significant bits so n*LN2_HI is exact
    m, _ = math.frexp(float(O.LN2_HI))
    assert (m * 2 ** 16) == int(m * 2 ** 16)
    assert abs(float(O.LOG2E) - 1 / math.log(2)) < 1e-7
    for k, c in enumerate(O.TAYLOR):
        assert abs(float(c) * math.factorial(k) - 1.0) < 1e-7


# ------------------------------------------------------------------ routing
def test_worked_example_from_the_rules():
    g = _gold("routing_worked_example.json")
    z = np.array([g["logits"]], F32)
    for case in g["cases"]:
        r = O.route(z, np.array(case["bias"], F32), g["n_group"],
                    g["topk_group"], g["topk"])
        assert r["idx"][0].tolist() == case["idx"]
        assert sorted(np.nonzero(r["kept"][0])[0].tolist()) == \
            case["kept_groups"]
        np.testing.assert_allclose(r["gate"][0], case["gate"], atol=2e-6)


def _brute_route(u, s, n_group, topk_group, topk):
    """Selection by exhaustive search, a formulation independent of sorting:
    group score = max over pairs i != j in the group of u_i + u_j; kept set =
    the topk_group-subset of groups with the largest total score (ties to the
    lexicographically smallest); chosen set = the topk-subset of the kept
    experts with the largest sum of u (ties likewise); slots ordered by u desc,
    index asc."""
    E = u.shape[0]
    gs = E // n_group
    S = []
    for gi in range(n_group):
        mem = range(gi * gs, (gi + 1) * gs)
        S.append(max(float(F32(u[i]) + F32(u[j]))
                     for i, j in itertools.permutations(mem, 2)))
    best = max(itertools.combinations(range(n_group), topk_group),
               key=lambda c: (sum(S[i] for i in c), [-i for i in c]))
    cand = [e for e in range(E) if e // gs in best]
    chosen = max(itertools.combinations(cand, topk),
                 key=lambda c: (sum(float(u[e]) for e in c), [-e for e in c]))
    slots = sorted(chosen, key=lambda e: (-float(u[e]), e))
    return sorted(best), slots


def test_selection_matches_brute_force_tiny_config():
    cfg = inputs.CONFIGS["tiny"]
    z = O.router_logits(inputs.bf16_bits_to_f32(inputs.x_tokens(cfg)),
                        inputs.router_weight(cfg))
    b = inputs.bias(cfg)
    r = O.route(z, b, cfg.n_group, cfg.topk_group, cfg.topk)
    for t in range(cfg.T):
        kept, slots = _brute_route(r["u"][t], r["s"][t], cfg.n_group,
                                   cfg.topk_group, cfg.topk)
        assert sorted(np.nonzero(r["kept"][t])[0].tolist()) == kept, t
        assert r["idx"][t].tolist() == slots, t


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_selection_matches_brute_force_random_shapes(seed):
    rng = np.random.default_rng(seed)
    for (E, G, M, K) in [(8, 2, 1, 2), (12, 3, 2, 3), (16, 4, 3, 5),
                         (8, 4, 4, 8)]:
        z = rng.normal(0, 1, size=(20, E)).astype(F32)
        b = rng.uniform(-0.1, 0.1, size=E).astype(F32)
        r = O.route(z, b, G, M, K)
        for t in range(20):
            kept, slots = _brute_route(r["u"][t], r["s"][t], G, M, K)
            assert sorted(np.nonzero(r["kept"][t])[0].tolist()) == kept
            assert r["idx"][t].tolist() == slots


def test_group_score_is_top2_sum_not_max():
    """A group with one huge and many tiny affinities must lose to a group
    with two moderately high ones (sum of top-2, not max)."""
    E, G = 8, 2
    z = np.array([[4.0, -6, -6, -6, 1.5, 1.5, -6, -6]], F32)
    r = O.route(z, np.zeros(E, F32), G, 1, 2)
    assert r["kept"][0].tolist() == [False, True]
    assert sorted(r["idx"][0].tolist()) == [4, 5]


def test_gates_sum_to_one_and_bias_never_changes_gate_values():
    """§1.3: the chosen gates sum to 1; §1.4: the bias only changes which
    experts are chosen, never the weight of a chosen one."""
    cfg = inputs.CONFIGS["route_v3"]
    z = inputs.random_logits(cfg, T=2048)
    b = inputs.bias(cfg)
    r1 = O.route(z, b, cfg.n_group, cfg.topk_group, cfg.topk)
    r0 = O.route(z, np.zeros_like(b), cfg.n_group, cfg.topk_group, cfg.topk)
    tot = r1["gate"].astype(np.float64).sum(1)
    assert np.max(np.abs(tot - 1.0)) <= cfg.topk * 2.0 ** -24
    # gates against the raw affinity ratio, computed independently in fp64
    # from sigma: within fp32 rounding of s and of the division
    s_ex = expit(z.astype(np.float64))
    chosen = np.take_along_axis(s_ex, r1["idx"], 1)
    np.testing.assert_allclose(r1["gate"], chosen / chosen.sum(1, keepdims=True),
                               rtol=3e-6, atol=0)
    same = np.all(np.sort(r1["idx"], 1) == np.sort(r0["idx"], 1), axis=1)
    assert same.sum() > 100 and (~same).sum() > 0   # the bias does bite
    for t in np.nonzero(same)[0]:
        o1 = np.argsort(r1["idx"][t])
        o0 = np.argsort(r0["idx"][t])
        # same chosen set -> identical gate per expert, bit for bit, as long
        # as the slot order (which fixes the fp32 summation order) agrees
        if np.array_equal(r1["idx"][t], r0["idx"][t]):
            assert np.array_equal(r1["gate"][t], r0["gate"][t])
        else:
            np.testing.assert_allclose(r1["gate"][t][o1], r0["gate"][t][o0],
                                       rtol=2.0 ** -22)


def test_every_selected_expert_is_in_a_kept_group():
    cfg = inputs.CONFIGS["route_v3"]
    z = inputs.random_logits(cfg, T=4096, step=3)
    r = O.route(z, inputs.bias(cfg), cfg.n_group, cfg.topk_group, cfg.topk)
    gs = cfg.E // cfg.n_group
    assert np.all(r["kept"].sum(1) == cfg.topk_group)
    assert np.all(np.take_along_axis(r["kept"], r["idx"] // gs, 1))
    # distinct experts per token
    assert np.all(np.diff(np.sort(r["idx"], 1), axis=1) > 0)
    # slot order: u non-increasing
    uk = np.take_along_axis(r["u"], r["idx"], 1)
    assert np.all(np.diff(uk, axis=1) <= 0)


def test_single_group_no_bias_is_plain_argsort_of_logits():
    """Textbook reduction: one group, zero bias -> top-K of the logits
    (sigmoid is monotone), i.e. numpy's argsort of -z."""
    rng = np.random.default_rng(7)
    z = rng.normal(0, 1, size=(500, 64)).astype(F32)
    r = O.route(z, np.zeros(64, F32), 1, 1, 6)
    np.testing.assert_array_equal(r["idx"], np.argsort(-z, axis=1)[:, :6])


def test_k1_gate_is_exactly_one_and_k_equals_e_chooses_all():
    rng = np.random.default_rng(8)
    z = rng.normal(0, 1, size=(50, 16)).astype(F32)
    r = O.route(z, np.zeros(16, F32), 4, 2, 1)
    assert np.all(r["gate"] == 1.0)
    r = O.route(z, rng.normal(0, .1, 16).astype(F32), 1, 1, 16)
    assert np.all(np.sort(r["idx"], 1) == np.arange(16))


def test_bias_steers_selection():
    """A bias larger than any affinity gap forces an expert into every
    token's choice (selection uses s + b)."""
    cfg = inputs.CONFIGS["route_v3"]
    z = inputs.random_logits(cfg, T=256)
    b = np.zeros(cfg.E, F32)
    b[77] = 2.0
    r = O.route(z, b, cfg.n_group, cfg.topk_group, cfg.topk)
    assert np.all(r["idx"][:, 0] == 77)


def test_group_on_unbiased_ablation_differs():
    cfg = inputs.CONFIGS["route_v3"]
    z = inputs.random_logits(cfg, T=2048)
    b = (inputs.bias(cfg) * 20).astype(F32)
    a = O.route(z, b, cfg.n_group, cfg.topk_group, cfg.topk)
    c = O.route(z, b, cfg.n_group, cfg.topk_group, cfg.topk,
                group_on_unbiased=True)
    assert np.any(a["kept"] != c["kept"])


# ------------------------------------------------------------ permutation
def test_permutation_matches_python_sorted():
    rng = np.random.default_rng(3)
    T, E, K = 300, 16, 4
    idx = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(
        np.int32)
    p = O.permutation(idx, E)
    pairs = sorted(((int(idx[t, k]), t, k) for t in range(T) for k in range(K)))
    for r, (e, t, k) in enumerate(pairs):
        assert p["dest"][t, k] == r
        assert p["src_row"][r] == t * K + k
    assert p["offsets"][0] == 0 and p["offsets"][-1] == T * K
    for e in range(E):
        seg = p["src_row"][p["offsets"][e]:p["offsets"][e + 1]]
        assert np.all(idx.ravel()[seg] == e)
        assert np.all(np.diff(seg // K) > 0)


def test_counts_sum_and_histogram():
    rng = np.random.default_rng(4)
    idx = np.stack([rng.choice(32, 8, replace=False) for _ in range(1000)])
    c = O.expert_counts(idx, 32)
    assert c.sum() == 8000
    for e in range(32):
        assert c[e] == sum(1 for row in idx for v in row if v == e)


# --------------------------------------------------------------- bias step
def test_bias_update_worked_example():
    """E = 4, T = 4, K = 2: mean load 2.  Loads [3, 1, 2, 2]: expert 0 is
    overloaded (-gamma), expert 1 underloaded (+gamma), 2 and 3 sit at the
    mean and are left alone."""
    b = np.array([0.5, -0.25, 0.125, 0.0], F32)
    nb, st = O.bias_update(np.array([3, 1, 2, 2]), b, 4, 2, 0.001)
    g = F32(0.001)
    assert nb[0] == F32(F32(0.5) - g) and nb[1] == F32(F32(-0.25) + g)
    assert nb[2] == b[2] and nb[3] == b[3]
    assert st == (3.0, 2.0, 1.0)
    nb2, _ = O.bias_update(np.array([3, 1, 2, 2]), b, 4, 2, 0.001,
                           tie_overloaded=True)
    assert nb2[2] < b[2] and nb2[3] < b[3]


def test_bias_update_moves_each_expert_by_gamma_toward_balance():
    rng = np.random.default_rng(5)
    E, T, K = 256, 4096, 8
    c = rng.multinomial(T * K, np.full(E, 1 / E))
    b = rng.uniform(-0.01, 0.01, E).astype(F32)
    nb, (mx, mean, mn) = O.bias_update(c, b, T, K, 0.001)
    d = nb.astype(np.float64) - b.astype(np.float64)
    over, under = c > mean, c < mean
    assert np.all(d[over] < 0) and np.all(d[under] > 0)
    assert np.all(d[~over & ~under] == 0)
    np.testing.assert_allclose(np.abs(d[over | under]), 0.001, rtol=1e-4)
    assert mx == c.max() and mn == c.min() and mean == T * K / E


def test_gamma_steps_accumulate_over_steps():
    """b after n steps = b0 + gamma * (#under - #over), to fp32 rounding."""
    rng = np.random.default_rng(6)
    E, T, K = 16, 64, 4
    b0 = np.zeros(E, F32)
    b = b0.copy()
    net = np.zeros(E)
    for _ in range(50):
        c = rng.multinomial(T * K, rng.dirichlet(np.ones(E)))
        b, _ = O.bias_update(c, b, T, K, 0.001)
        net += (c * E < T * K).astype(int) - (c * E > T * K).astype(int)
    np.testing.assert_allclose(b, 0.001 * net, atol=1e-6)


# ------------------------------------------------------------ expert math
def test_router_logits_exact_on_dyadic_inputs():
    """With small dyadic inputs every product and partial sum is exact, so
    the logits must equal exact rational arithmetic (pins operand order:
    z[t, e] pairs token t with expert e's router row)."""
    rng = np.random.default_rng(9)
    x = (rng.integers(-8, 9, size=(5, 24)) / 8).astype(F32)
    w = (rng.integers(-8, 9, size=(7, 24)) / 16).astype(F32)
    z = O.router_logits(x, w)
    assert z.shape == (5, 7)
    for t in range(5):
        for e in range(7):
            ex = sum(Fraction(float(x[t, h])) * Fraction(float(w[e, h]))
                     for h in range(24))
            assert z[t, e] == F32(float(ex))
    # an additive per-expert offset enters once, before the rounding
    o = (rng.integers(-8, 9, size=7) / 4).astype(F32)
    zo = O.router_logits(x, w, o)
    for t in range(5):
        for e in range(7):
            ex = sum(Fraction(float(x[t, h])) * Fraction(float(w[e, h]))
                     for h in range(24)) + Fraction(float(o[e]))
            assert zo[t, e] == F32(float(ex))


def test_swiglu_closed_form_scalar():
    """H = I = 1: y = w2 * silu(w1 a) * (w3 a)."""
    a, w1, w3, w2 = 0.7, 1.3, -0.4, 2.5
    y = O.swiglu_ffn(np.array([[a]]), np.array([[w1]]), np.array([[w3]]),
                     np.array([[w2]]))
    p = w1 * a
    assert abs(y[0, 0] - w2 * (p / (1 + math.exp(-p))) * (w3 * a)) < 1e-15


def test_swiglu_against_einsum_and_expit():
    rng = np.random.default_rng(10)
    a = rng.normal(size=(9, 32))
    w1, w3 = rng.normal(size=(2, 12, 32)) * .2
    w2 = rng.normal(size=(32, 12)) * .2
    p = np.einsum("th,ih->ti", a, w1)
    ref = np.einsum("ti,hi->th", p * expit(p) * np.einsum("th,ih->ti", a, w3),
                    w2)
    np.testing.assert_allclose(O.swiglu_ffn(a, w1, w3, w2), ref, rtol=1e-12,
                               atol=1e-12)


def _tiny_values(cfg):
    d = inputs.layer_inputs(cfg)
    f = inputs.bf16_bits_to_f32
    return (f(d["x"]), d["w_router"], d["bias"], f(d["w1"]), f(d["w3"]),
            f(d["w2"]), f(d["ws1"]), f(d["ws3"]), f(d["ws2"]))


def test_layer_with_zero_routed_experts_is_residual_plus_dense_swiglu():
    cfg = inputs.CONFIGS["tiny"]
    x, wr, b, w1, w3, w2, ws1, ws3, ws2 = _tiny_values(cfg)
    res = O.layer_forward(x, wr, b, 0 * w1, 0 * w3, 0 * w2, ws1, ws3, ws2,
                          n_group=cfg.n_group, topk_group=cfg.topk_group,
                          topk=cfg.topk)
    xs = x.astype(np.float64)
    p = xs @ ws1.astype(np.float64).T
    dense = (p * expit(p) * (xs @ ws3.astype(np.float64).T)) @ \
        ws2.astype(np.float64).T
    np.testing.assert_allclose(res["out"], xs + dense, rtol=1e-12, atol=1e-12)


def test_layer_with_identical_experts_adds_one_full_ffn():
    """All routed experts equal -> routed term = FFN(x) * sum(g) = FFN(x)
    because the gates sum to 1 (eq. 12 with eq. 13)."""
    cfg = inputs.CONFIGS["tiny"]
    x, wr, b, w1, w3, w2, ws1, ws3, ws2 = _tiny_values(cfg)
    W1 = np.broadcast_to(w1[3], w1.shape)
    W3 = np.broadcast_to(w3[3], w3.shape)
    W2 = np.broadcast_to(w2[3], w2.shape)
    res = O.layer_forward(x, wr, b, W1, W3, W2, 0 * ws1, 0 * ws3, 0 * ws2,
                          n_group=cfg.n_group, topk_group=cfg.topk_group,
                          topk=cfg.topk)
    xs = x.astype(np.float64)
    p = xs @ w1[3].astype(np.float64).T
    f = (p * expit(p) * (xs @ w3[3].astype(np.float64).T)) @ \
        w2[3].astype(np.float64).T
    np.testing.assert_allclose(res["out"], xs + f, rtol=1e-6, atol=1e-6)


def test_layer_routed_term_uses_each_chosen_expert_once_with_its_gate():
    """Brute force of eq. 12 for a few tokens, expert by expert."""
    cfg = inputs.CONFIGS["tiny"]
    x, wr, b, w1, w3, w2, ws1, ws3, ws2 = _tiny_values(cfg)
    res = O.layer_forward(x, wr, b, w1, w3, w2, ws1, ws3, ws2,
                          n_group=cfg.n_group, topk_group=cfg.topk_group,
                          topk=cfg.topk)
    r = res["route"]
    xs = x.astype(np.float64)
    for t in (0, 17, 63):
        acc = xs[t].copy()
        for e in range(cfg.E):
            hit = np.nonzero(r["idx"][t] == e)[0]
            for k in hit:
                acc += float(r["gate"][t, k]) * O.swiglu_ffn(
                    xs[t:t + 1], w1[e], w3[e], w2[e])[0]
        acc += O.swiglu_ffn(xs[t:t + 1], ws1, ws3, ws2)[0]
        np.testing.assert_allclose(res["out"][t], acc, rtol=1e-12, atol=1e-12)


def test_layer_rows_agrees_with_layer_forward():
    cfg = inputs.CONFIGS["tiny"]
    x, wr, b, w1, w3, w2, ws1, ws3, ws2 = _tiny_values(cfg)
    res = O.layer_forward(x, wr, b, w1, w3, w2, ws1, ws3, ws2,
                          n_group=cfg.n_group, topk_group=cfg.topk_group,
                          topk=cfg.topk)
    rows = np.array([1, 5, 40])
    out = O.layer_rows(x[rows], res["route"]["idx"][rows],
                       res["route"]["gate"][rows],
                       lambda e: (w1[e], w3[e], w2[e]), (ws1, ws3, ws2))
    np.testing.assert_allclose(out, res["out"][rows], rtol=1e-13, atol=1e-13)


# ------------------------------------------------------ what the pages print
def test_v3_shape_constants_match_the_pages():
    g = _gold("v3_shape.json")
    cfg = inputs.CONFIGS["prefill_v3"]
    assert (cfg.H, cfg.I, cfg.E, cfg.topk, cfg.n_group, cfg.topk_group) == (
        g["hidden_size"], g["moe_intermediate_size"], g["n_routed_experts"],
        g["num_experts_per_tok"], g["n_nodes_or_groups"],
        g["max_groups_per_token"])
    per_expert = 3 * cfg.H * cfg.I
    assert round(per_expert / 1e6, 1) == g["params_per_expert_millions_approx"]
    active = per_expert * (cfg.topk + g["n_shared_experts"])
    assert round(active / 1e6) == g["active_expert_params_per_layer_millions_approx"]
    assert cfg.gamma == g["bias_gamma"]


# ------------------------------------------------------ input generator
def test_generator_host_and_numpy_evaluations_agree():
    """The counter-based cells are the same integers whether evaluated by
    numpy or by torch (the device path uses the torch one)."""
    from deepseekmoe_routing_expert_moe_b300.inputs import (cells_numpy,
                                                            cells_torch)
    for key, start in ((0, 0), (123456789, 5), (0xFFFFFFFF, (1 << 31) - 5000)):
        a = cells_numpy(4096, key, start)
        b = cells_torch(4096, key, "cpu", start).numpy()
        assert np.array_equal(a, b)


def test_generator_statistics():
    from deepseekmoe_routing_expert_moe_b300.inputs import cells_numpy
    c = cells_numpy(1 << 20, 987654321)
    h = np.bincount(c, minlength=65536)
    chi2 = (((h - h.mean()) ** 2) / h.mean()).sum() / 65535
    assert 0.95 < chi2 < 1.05
    cfg = inputs.CONFIGS["tiny"]
    w = inputs.bf16_bits_to_f32(inputs.expert_weights(cfg, 0)[0]).ravel()
    assert abs(w.mean()) < 1e-3 and abs(w.std() - 0.02) < 1e-3
    x = inputs.bf16_bits_to_f32(inputs.x_tokens(cfg)).ravel()
    assert abs(x.std() - 1.0) < 0.02
    assert abs(np.corrcoef(x[:-1], x[1:])[0, 1]) < 0.02
