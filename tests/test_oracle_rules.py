"""Pins of the oracle's knobs, softmax, residual, inverse CDF and accept rule.

Each check compares the oracle with something other than itself: a closed
form, a counting definition of the kept set, a library routine (numpy argmax,
scipy chi-square), or a property that any correct implementation must have.
"""
import math

import numpy as np
import pytest

import oracle as O


def _softmax_ratio_ok(P, l, T, kept):
    """Kept probabilities are in the ratio exp((l_v - l_w) / T) and sum to 1."""
    idx = np.flatnonzero(kept)
    assert abs(P.sum() - 1.0) < 1e-12
    assert np.all(P[~kept] == 0.0)
    assert np.all(P[idx] > 0.0)
    ref = idx[np.argmax(l[idx])]
    np.testing.assert_allclose(P[idx] / P[ref], np.exp((l[idx] - l[ref]) / T), rtol=1e-12)


# ------------------------------------------------------------- softmax / T --
@pytest.mark.parametrize("T", [0.3, 0.7, 1.0, 2.5])
def test_two_token_softmax_is_logistic(orc, T):
    rng = np.random.default_rng(1)
    for _ in range(50):
        l = rng.normal(0, 4, size=2)
        P, info = orc.row_dist(l, T)
        want = 1.0 / (1.0 + math.exp(-(l[0] - l[1]) / T))
        assert abs(P[0] - want) < 1e-14
        assert abs(P[0] + P[1] - 1.0) < 1e-15
        assert info.n_kept == 2


def test_softmax_ratios_and_lse(orc):
    rng = np.random.default_rng(2)
    l = rng.normal(0, 3, size=257)
    P, info = orc.row_dist(l, 0.7)
    _softmax_ratio_ok(P, l, 0.7, np.ones(l.size, bool))
    lse = np.log(np.sum(np.exp(l / 0.7 - np.max(l / 0.7)))) + np.max(l / 0.7)
    assert abs(info.M + math.log(info.S) - lse) < 1e-10


# ------------------------------------------------------------------ top-k --
def _rank_before(l):
    """before[v, w] = w is ranked strictly before v (higher l, or tie and lower id)."""
    V = l.size
    ids = np.arange(V)
    return (l[None, :] > l[:, None]) | ((l[None, :] == l[:, None]) & (ids[None, :] < ids[:, None]))


@pytest.mark.parametrize("V", [2, 3, 7, 16, 17])
def test_topk_counting_definition(orc, V):
    rng = np.random.default_rng(V)
    for trial in range(40):
        # small integer logits force many ties
        l = rng.integers(-3, 4, size=V).astype(np.float64)
        if trial % 3 == 0:
            l[rng.integers(0, V)] = -np.inf
        T = float(rng.choice([0.5, 1.0, 1.7]))
        for k in range(1, V):
            P, info = orc.row_dist(l, T, top_k=k)
            kept_want = _rank_before(l).sum(axis=1) < k
            kept_want &= np.isfinite(l)          # a -inf logit carries no mass
            assert np.array_equal(P > 0, kept_want), (l, k, P)
            _softmax_ratio_ok(P, l, T, kept_want)
        # k = 0 and k >= V are "off"
        P0, _ = orc.row_dist(l, T, top_k=0)
        PV, _ = orc.row_dist(l, T, top_k=V)
        np.testing.assert_array_equal(P0, PV)
        assert np.array_equal(P0 > 0, np.isfinite(l))


def test_topk_all_equal_keeps_lowest_ids(orc):
    l = np.zeros(10)
    P, info = orc.row_dist(l, 1.0, top_k=4)
    np.testing.assert_array_equal(P, [0.25] * 4 + [0.0] * 6)


# ------------------------------------------------------------------ top-p --
@pytest.mark.parametrize("V", [3, 8, 16])
def test_topp_counting_definition(orc, V):
    rng = np.random.default_rng(100 + V)
    for trial in range(60):
        l = rng.integers(-4, 5, size=V).astype(np.float64) * 0.5
        T = float(rng.choice([0.6, 1.0, 1.3]))
        k = int(rng.choice([0, 0, V // 2 + 1]))
        top_p = float(rng.uniform(0.05, 0.99))
        Pk, _ = orc.row_dist(l, T, top_k=k)      # the distribution top-p walks over
        P, info = orc.row_dist(l, T, top_k=k, top_p=top_p)
        before = _rank_before(l)
        mass_before = (before * Pk[None, :]).sum(axis=1)
        kept_want = (Pk > 0) & (mass_before < top_p)
        if np.all(np.abs(mass_before[Pk > 0] - top_p) > 1e-12):
            assert np.array_equal(P > 0, kept_want), (l, T, k, top_p)
        _softmax_ratio_ok(P, l, T, P > 0)
        # margin: distance of the boundary decisions to top_p; a token with no
        # mass before it (rank 0) is kept by any top_p > 0 and has no margin
        m = np.abs(mass_before[(Pk > 0) & (mass_before > 0)] - top_p)
        if m.size:
            assert info.topp_margin <= m.min() + 1e-12 or info.topp_margin == math.inf
        else:
            assert info.topp_margin == math.inf


def test_topp_strict_prefix_rule_on_exact_masses(orc):
    # four equal logits: masses 1/4 exactly; mass before ranks = 0, .25, .5, .75
    l = np.zeros(4)
    P, info = orc.row_dist(l, 1.0, top_p=0.5)
    np.testing.assert_array_equal(P, [0.5, 0.5, 0.0, 0.0])   # rank 2 has 0.5 before it
    assert info.topp_margin == 0.0
    P, _ = orc.row_dist(l, 1.0, top_p=0.5000001)
    np.testing.assert_allclose(P, [1 / 3, 1 / 3, 1 / 3, 0.0], rtol=1e-15)
    P, _ = orc.row_dist(l, 1.0, top_p=1.0)                   # off
    np.testing.assert_array_equal(P, [0.25] * 4)


def test_topp_tiny_is_argmax(orc):
    rng = np.random.default_rng(5)
    for _ in range(50):
        l = rng.integers(-5, 6, size=33).astype(np.float64)
        P, info = orc.row_dist(l, 1.0, top_p=1e-12)
        assert info.n_kept == 1
        assert P[np.argmax(l)] == 1.0      # numpy's argmax: first of equal maxima


# ---------------------------------------------------------- nonfinite rows --
def test_nonfinite_rows(orc):
    for bad in ([0.0, np.nan, 1.0], [0.0, np.inf, 1.0], [-np.inf, -np.inf]):
        P, info = orc.row_dist(np.array(bad), 1.0)
        assert P is None and info.nonfinite
    P, info = orc.row_dist(np.array([-np.inf, 0.0, -np.inf]), 1.0)
    np.testing.assert_array_equal(P, [0.0, 1.0, 0.0])


# ---------------------------------------------------------------- residual --
def test_residual_identity(orc):
    """min(p_t, p_d) + (1 - sum min) * R / Z == p_t for every token (the two
    routes of the losslessness argument add back to the target)."""
    rng = np.random.default_rng(7)
    for _ in range(200):
        V = int(rng.integers(2, 40))
        Pt, _ = orc.row_dist(rng.normal(0, 2, V), 1.0, top_k=int(rng.integers(0, V)))
        Pd, _ = orc.row_dist(rng.normal(0, 2, V), 0.8, top_p=float(rng.uniform(0.3, 1.0)))
        R, Z = orc.residual(Pt, Pd)
        alpha = np.minimum(Pt, Pd).sum()
        assert abs(Z - (1.0 - alpha)) < 1e-12
        assert np.all(R >= 0)
        if Z > 1e-9:
            np.testing.assert_allclose(np.minimum(Pt, Pd) + (1.0 - alpha) * R / Z, Pt,
                                       atol=1e-12)


# ------------------------------------------------------------- inverse CDF --
def test_inverse_cdf_counts_on_u_grid(orc):
    """On the grid u = m 2^-s every token receives exactly R(v)/Z of the grid
    when the masses are dyadic; zero-mass tokens never."""
    R = np.array([0.0, 0.125, 0.0, 0.25, 0.5, 0.0, 0.125, 0.0])
    n = 1 << 10
    counts = np.zeros(R.size, np.int64)
    for m in range(n):
        t = orc.inverse_cdf(R, m / n)[0]
        counts[t] += 1
    np.testing.assert_array_equal(counts, (R * n).astype(np.int64))
    # non-normalised R: the same, scaled
    counts2 = np.zeros(R.size, np.int64)
    for m in range(n):
        counts2[orc.inverse_cdf(R * 3.0, m / n)[0]] += 1
    np.testing.assert_array_equal(counts2, counts)
    assert orc.inverse_cdf(np.zeros(4), 0.3)[0] == -1


def test_inverse_cdf_margin_and_neighbourhood(orc):
    R = np.array([0.25, 0.25, 0.25, 0.25])
    tok, Z, m, lo, hi = orc.inverse_cdf(R, 0.5 + 1e-9, delta=1e-6)
    assert tok == 2 and abs(m - 1e-9) < 1e-12 and lo == 1 and hi == 2
    tok, Z, m, lo, hi = orc.inverse_cdf(R, 0.375, delta=1e-6)
    assert tok == 1 and abs(m - 0.125) < 1e-12 and lo == hi == 1


# ---------------------------------------------------------------- LM head --
def test_lmhead_matches_numpy_matmul(orc):
    from workloads import bf16_bits_to_f32, f32_to_bf16_bits
    rng = np.random.default_rng(11)
    H = f32_to_bf16_bits(rng.normal(0, 1, (6, 40)).astype(np.float32))
    W = f32_to_bf16_bits(rng.normal(0, 0.02, (40, 23)).astype(np.float32))
    got = orc.lmhead(H, W, 1, 5)
    want = (bf16_bits_to_f32(H).astype(np.float64) @ bf16_bits_to_f32(W).astype(np.float64))[1:5]
    np.testing.assert_allclose(got, want, rtol=1e-13, atol=1e-15)
