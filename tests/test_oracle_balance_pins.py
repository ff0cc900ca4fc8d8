"""Pins for the oracle's sequence-wise balance loss (no GPU).

"02 · DeepSeek-V3" (PaperTrace) §1.4, eq. 17-20: per sequence,
L = alpha * sum_i f_i P_i with f_i = E/(K T_s) * (tokens whose raw top-K
holds expert i) and P_i the sequence mean of the normalised affinity
s_i / sum_j s_j.  Each test ties the oracle to a closed form, brute-force
enumeration or an invariant of those definitions, so that a slip (f taken
from the biased or group-limited selection, P not normalised per token, a
missing E/K factor, sequences cut in the wrong place) fails one of them.
"""
import inspect
import itertools
import math

import numpy as np
import pytest

from oracle import moe_oracle as O

F32 = np.float32


def _sigma(v):
    return 1.0 / (1.0 + math.exp(-v))


def test_default_alpha_is_the_pages_value():
    assert inspect.signature(O.seq_balance_loss).parameters[
        "alpha"].default == 1e-4


def test_uniform_affinities_give_alpha_and_lowest_index_ties():
    """All logits equal: every s is the same, so P_i = 1/E and the top-K
    is the K lowest indices (the tie rule); sum_i f_i = E, so L = alpha."""
    E, K, T = 32, 4, 50
    r = O.seq_balance_loss(np.full((T, E), 0.37, F32), seq_len=T, topk=K)
    np.testing.assert_allclose(r["P"][0], 1.0 / E, rtol=1e-14)
    assert r["counts"][0, :K].tolist() == [T] * K
    assert r["counts"][0, K:].sum() == 0
    assert r["loss"][0] == pytest.approx(1e-4, rel=1e-14)


def test_collapsed_routing_closed_form():
    """K experts at logit +a, the rest at -a, on every token: f = E/K on
    the K, 0 elsewhere, P = sigma(a)/den there, so
    L = alpha * E * sigma(a) / (K sigma(a) + (E-K) sigma(-a))."""
    E, K, T, a = 256, 8, 40, 3.0
    z = np.full((T, E), -a, F32)
    hot = [5, 17, 40, 99, 100, 180, 201, 255]
    z[:, hot] = a
    r = O.seq_balance_loss(z, seq_len=T, topk=K)
    den = K * _sigma(a) + (E - K) * _sigma(-a)
    want = 1e-4 * E * _sigma(a) / den
    assert r["loss"][0] == pytest.approx(want, rel=1e-6)
    assert sorted(np.nonzero(r["counts"][0])[0].tolist()) == hot
    np.testing.assert_allclose(r["f"][0, hot], E / K, rtol=0)


def test_evenly_spread_selection_gives_alpha_for_any_P():
    """Token t puts its K largest affinities on block t mod (E/K) of K
    experts and random smaller values elsewhere; with T_s a multiple of E/K
    every f_i is 1, so L = alpha * sum_i P_i = alpha whatever P is."""
    E, K = 64, 4
    nb = E // K
    T = 3 * nb
    rng = np.random.default_rng(3)
    z = rng.uniform(-3.0, -1.0, (T, E)).astype(F32)
    for t in range(T):
        b = t % nb
        z[t, b * K:(b + 1) * K] = rng.uniform(1.0, 3.0, K)
    r = O.seq_balance_loss(z, seq_len=T, topk=K)
    np.testing.assert_array_equal(r["f"][0], np.ones(E))
    assert r["loss"][0] == pytest.approx(1e-4, rel=1e-13)
    assert np.ptp(r["P"][0]) > 1e-3          # P itself is far from uniform


def test_brute_force_on_tiny_input_with_ragged_sequences():
    """E=6, K=2, T=7 cut into sequences of 3, 3, 1.  The raw top-K set is
    the K-subset of largest affinity sum (enumerated); P and L by plain
    loops over the definition."""
    E, K, T, S = 6, 2, 7, 3
    alpha = 2.5e-3
    z = np.random.default_rng(11).normal(0.0, 1.5, (T, E)).astype(F32)
    s = O.sig32(z).astype(np.float64)
    r = O.seq_balance_loss(z, seq_len=S, topk=K, alpha=alpha)
    assert r["loss"].shape == (3,)
    for q, (a, b) in enumerate([(0, 3), (3, 6), (6, 7)]):
        cnt = [0] * E
        Psum = [0.0] * E
        for t in range(a, b):
            best = max(itertools.combinations(range(E), K),
                       key=lambda c: sum(s[t, i] for i in c))
            for i in best:
                cnt[i] += 1
            tot = math.fsum(s[t])
            for i in range(E):
                Psum[i] += s[t, i] / tot
        Ts = b - a
        L = alpha * math.fsum((E / (K * Ts)) * cnt[i] * (Psum[i] / Ts)
                              for i in range(E))
        assert r["counts"][q].tolist() == cnt
        np.testing.assert_allclose(r["P"][q], np.array(Psum) / Ts, rtol=1e-13)
        assert r["loss"][q] == pytest.approx(L, rel=1e-12)


def test_per_sequence_sums_are_fixed():
    """sum_i f_i = E and sum_i P_i = 1 in every sequence (the pages'
    normalisation: f has mean 1, P sums to 1)."""
    E, K = 256, 8
    z = np.random.default_rng(5).normal(0.0, 0.6, (1000, E)).astype(F32)
    r = O.seq_balance_loss(z, seq_len=300, topk=K)
    assert r["loss"].shape == (4,)
    np.testing.assert_allclose(r["f"].sum(1), E, rtol=1e-13)
    np.testing.assert_allclose(r["P"].sum(1), 1.0, rtol=1e-13)
    assert r["counts"].sum(1).tolist() == [300 * K] * 3 + [100 * K]
    assert np.all(r["loss"] > 0)


def test_sequences_are_independent():
    """The loss of each sequence depends on its own tokens only: cutting the
    batch and computing each piece alone gives the same values."""
    E, K, S = 64, 6, 37
    z = np.random.default_rng(8).normal(0.0, 1.0, (130, E)).astype(F32)
    whole = O.seq_balance_loss(z, seq_len=S, topk=K)
    for q in range(4):
        part = O.seq_balance_loss(z[q * S:(q + 1) * S], seq_len=S, topk=K)
        np.testing.assert_array_equal(part["counts"][0], whole["counts"][q])
        assert part["loss"][0] == whole["loss"][q]


def test_counts_use_raw_affinity_not_the_routed_selection():
    """f counts the raw top-K of s over all experts: no bias and no group
    limit (the routed choice uses both).  A bias that pushes expert 0 into
    every token's routed top-K leaves f's counts unchanged."""
    E, G, M, K = 16, 4, 2, 2
    z = np.random.default_rng(2).normal(0.0, 1.0, (200, E)).astype(F32)
    bias = np.zeros(E, F32)
    bias[0] = 10.0
    routed = O.expert_counts(O.route(z, bias, G, M, K)["idx"], E)
    assert routed[0] == 200
    r = O.seq_balance_loss(z, seq_len=200, topk=K)
    s = O.sig32(z)
    raw = np.zeros(E, np.int64)
    for t in range(200):
        for i in np.argsort(-s[t], kind="stable")[:K]:
            raw[i] += 1
    np.testing.assert_array_equal(r["counts"][0], raw)
    assert r["counts"][0, 0] < 200
    unlimited = O.expert_counts(O.route(z, np.zeros(E, F32), 1, 1, K)["idx"],
                                E)
    np.testing.assert_array_equal(r["counts"][0], unlimited)
