"""Pins of the oracle's whole verify step.

* losslessness: the emitted token at every reached position follows the target
  distribution (chi-square, pre-registered p > 1e-3), with and without knobs;
* acceptance rate at a slot equals sum_v min(p_t, p_d);
* E[tokens per pass] equals the closed form, including the printed Table-1
  value 3.69 (tests/golden/tokens_per_pass.txt);
* top-k = 1 reduces to textbook greedy speculative decoding (numpy argmax);
* hand cases: p = q always accepts, q <= p accepts, disjoint supports never
  accept, q = 0 < p accepts;
* status codes and the 1 <= emitted <= K_b + 1 invariant.
"""
import math
import os

import numpy as np
import pytest
from scipy import stats

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tokens_per_pass.txt")
P_MIN = 1e-3


def _chi2_ok(tokens, P, label):
    tokens = np.asarray(tokens)
    n = tokens.size
    counts = np.bincount(tokens, minlength=P.size).astype(np.float64)
    assert np.all(counts[P == 0] == 0), f"{label}: zero-mass token emitted"
    exp = P * n
    big = exp >= 5
    obs = np.append(counts[big], counts[~big].sum())
    ex = np.append(exp[big], exp[~big].sum())
    if ex[-1] < 5:  # lump too small to test on its own: fold it into the largest bin
        i = int(np.argmax(ex[:-1]))
        obs[i] += obs[-1]
        ex[i] += ex[-1]
        obs, ex = obs[:-1], ex[:-1]
    p = stats.chisquare(obs, ex * obs.sum() / ex.sum()).pvalue
    assert p > P_MIN, f"{label}: chi-square p = {p:.2e}"


def _repeat_rows(rows: np.ndarray, B: int) -> np.ndarray:
    return np.ascontiguousarray(np.broadcast_to(rows, (B,) + rows.shape))


@pytest.mark.parametrize("knobs", [
    dict(temperature=1.0),
    dict(temperature=0.7, top_k=5),
    dict(temperature=1.3, top_p=0.8),
    dict(temperature=0.9, top_k=9, top_p=0.7),
])
def test_lossless_chi_square(orc, knobs):
    rng = np.random.default_rng(21)
    V, K, B = 16, 2, 200_000
    tl = rng.normal(0, 1.5, size=(K + 1, V)).astype(np.float32)
    dl = (tl[:K] + rng.normal(0, 1.0, size=(K, V))).astype(np.float32)
    target, draft = _repeat_rows(tl, B), _repeat_rows(dl, B)
    toks, _ = orc.draft_sample(draft, seed=99, **knobs)
    out = orc.verify(target, draft, toks, seed=99, **knobs)
    assert np.all(out["row_status"] == O.ROW_OK)
    Pt = [orc.row_dist(tl[j].astype(np.float64), **knobs)[0] for j in range(K + 1)]
    Pd0 = orc.row_dist(dl[0].astype(np.float64), **knobs)[0]
    # the drafted tokens follow the draft distribution
    _chi2_ok(toks[:, 0], Pd0, "draft sampler")
    # position 0 always follows the target, whatever happened
    _chi2_ok(out["tokens"][:, 0], Pt[0], "position 0")
    # given that position j-1 was accepted, position j follows target row j
    for j in (1, 2):
        reached = out["num_accepted"] >= j
        assert reached.sum() > 20_000
        _chi2_ok(out["tokens"][reached, j], Pt[j], f"position {j}")


def test_acceptance_rate_is_overlap(orc):
    rng = np.random.default_rng(22)
    V, K, B = 12, 1, 200_000
    tl = rng.normal(0, 1.2, size=(K + 1, V)).astype(np.float32)
    dl = (0.6 * tl[:K] + rng.normal(0, 1.0, size=(K, V))).astype(np.float32)
    target, draft = _repeat_rows(tl, B), _repeat_rows(dl, B)
    toks, _ = orc.draft_sample(draft, seed=5)
    out = orc.verify(target, draft, toks, seed=5)
    Pt = orc.row_dist(tl[0].astype(np.float64), 1.0)[0]
    Pd = orc.row_dist(dl[0].astype(np.float64), 1.0)[0]
    alpha = np.minimum(Pt, Pd).sum()
    assert abs(out["alpha"][0, 0] - alpha) < 1e-12
    rate = np.mean(out["num_accepted"] >= 1)
    sigma = math.sqrt(alpha * (1 - alpha) / B)
    assert abs(rate - alpha) < 4 * sigma, (rate, alpha)
    # the residual mass after a rejection is 1 - alpha
    rej = out["num_accepted"] == 0
    np.testing.assert_allclose(out["residual_mass"][rej], 1 - alpha, rtol=1e-12)


def _controlled_alpha_rows(alpha, K, B):
    """V = 2: draft one-hot on token 0, target (alpha, 1 - alpha): every slot
    accepts with probability alpha, independently."""
    tl = np.array([[math.log(alpha), math.log(1 - alpha)]] * (K + 1), np.float32)
    dl = np.array([[0.0, -np.inf]] * K, np.float32)
    return _repeat_rows(tl, B), _repeat_rows(dl, B), np.zeros((B, K), np.int32)


def test_expected_tokens_per_pass_golden(orc):
    rows = [l.split() for l in open(GOLDEN) if l.strip() and not l.startswith("#")]
    for a, k, printed, dec in rows:
        alpha, K, printed, dec = float(a), int(k), float(printed), int(dec)
        closed = (1 - alpha ** (K + 1)) / (1 - alpha)
        assert abs(closed - printed) <= 0.5 * 10 ** -dec + 1e-12
        B = 200_000
        target, draft, toks = _controlled_alpha_rows(alpha, K, B)
        out = orc.verify(target, draft, toks, seed=1234)
        emitted = out["num_accepted"] + 1
        assert emitted.min() >= 1 and emitted.max() <= K + 1
        mean, sem = emitted.mean(), emitted.std() / math.sqrt(B)
        assert abs(mean - closed) < 4 * sem, (mean, closed, sem)


@pytest.mark.parametrize("alpha,K", [(0.7, 4), (0.5, 3), (0.9, 8)])
def test_expected_tokens_per_pass_closed_form(orc, alpha, K):
    B = 100_000
    target, draft, toks = _controlled_alpha_rows(alpha, K, B)
    out = orc.verify(target, draft, toks, seed=77)
    emitted = out["num_accepted"] + 1
    closed = (1 - alpha ** (K + 1)) / (1 - alpha)
    assert abs(emitted.mean() - closed) < 4 * emitted.std() / math.sqrt(B)
    # on rejection the residual (0, 1 - alpha) normalised is one-hot on token 1
    rej = out["num_accepted"] < K
    toks_out = out["tokens"][np.flatnonzero(rej), out["num_accepted"][rej]]
    assert np.all(toks_out == 1)


def test_general_rows_expected_tokens(orc):
    """Rows with different alpha_j: E[emitted] = sum_m prod_{j<m} alpha_j."""
    rng = np.random.default_rng(23)
    V, K, B = 10, 3, 150_000
    tl = rng.normal(0, 1.0, size=(K + 1, V)).astype(np.float32)
    dl = (tl[:K] + rng.normal(0, 0.8, size=(K, V))).astype(np.float32)
    target, draft = _repeat_rows(tl, B), _repeat_rows(dl, B)
    toks, _ = orc.draft_sample(draft, seed=8)
    out = orc.verify(target, draft, toks, seed=8)
    a = [np.minimum(orc.row_dist(tl[j].astype(np.float64), 1.0)[0],
                    orc.row_dist(dl[j].astype(np.float64), 1.0)[0]).sum() for j in range(K)]
    pred = sum(np.prod(a[:m]) for m in range(K + 1))
    em = out["num_accepted"] + 1
    assert abs(em.mean() - pred) < 4 * em.std() / math.sqrt(B)


def test_topk1_is_greedy_speculative_decoding(orc):
    rng = np.random.default_rng(24)
    B, K, V = 400, 5, 9
    target = rng.integers(-3, 4, size=(B, K + 1, V)).astype(np.float32)
    draft = rng.integers(-3, 4, size=(B, K, V)).astype(np.float32)
    am = np.argmax(target, axis=2)           # numpy: first of equal maxima
    # drafts agree with the target argmax for a random prefix, then anything
    toks = rng.integers(0, V, size=(B, K)).astype(np.int32)
    for b in range(B):
        n = rng.integers(0, K + 1)
        toks[b, :n] = am[b, :n]
    out = orc.verify(target, draft, toks, top_k=1, temperature=0.9, seed=3)
    for b in range(B):
        n = 0
        while n < K and toks[b, n] == am[b, n]:
            n += 1
        want = list(toks[b, :n]) + [am[b, n]] + [-1] * (K - n)
        assert out["num_accepted"][b] == n
        assert list(out["tokens"][b]) == want, (b, out["tokens"][b], want)
        assert out["row_status"][b] in (O.ROW_OK, O.ROW_ZERO_RESIDUAL)


def test_hand_cases_v3(orc):
    B, K = 2000, 3
    # p == q: ratio 1, every draft accepted, the last token is the bonus
    tl = np.array([[0.1, 0.5, -0.3]] * (K + 1), np.float32)
    target = _repeat_rows(tl, B)
    draft = np.ascontiguousarray(target[:, :K])
    toks, _ = orc.draft_sample(draft, seed=4)
    out = orc.verify(target, draft, toks, seed=4)
    assert np.all(out["num_accepted"] == K)
    np.testing.assert_array_equal(out["tokens"][:, :K], toks)
    assert np.all(out["tokens"][:, K] >= 0)
    # q <= p at the drafted token: always accepted
    tp = np.log(np.array([0.5, 0.3, 0.2], np.float32))
    dp = np.log(np.array([0.2, 0.3, 0.5], np.float32))
    target = _repeat_rows(np.stack([tp] * (K + 1)), B)
    draft = _repeat_rows(np.stack([dp] * K), B)
    toks = np.zeros((B, K), np.int32)
    out = orc.verify(target, draft, toks, seed=5)
    assert np.all(out["num_accepted"] == K)
    # q > p: rejected with probability 1 - p/q = 1 - 0.2/0.5
    toks2 = np.full((B, K), 2, np.int32)
    out = orc.verify(target, draft, toks2, seed=6)
    rate = np.mean(out["num_accepted"] >= 1)
    assert abs(rate - 0.4) < 4 * math.sqrt(0.24 / B)
    # residual after a rejection: max(0, p_t - p_d) = (0.3, 0, 0) -> token 0
    rej = out["num_accepted"] == 0
    assert np.all(out["tokens"][rej, 0] == 0)
    # disjoint supports: never accepted, one token from p_t
    target = _repeat_rows(np.array([[0.0, 0.0, -np.inf]] * (K + 1), np.float32), B)
    draft = _repeat_rows(np.array([[-np.inf, -np.inf, 0.0]] * K, np.float32), B)
    toks = np.full((B, K), 2, np.int32)
    out = orc.verify(target, draft, toks, seed=7)
    assert np.all(out["num_accepted"] == 0)
    assert set(np.unique(out["tokens"][:, 0])) == {0, 1}
    assert np.all(out["tokens"][:, 1:] == -1)
    # q = 0 < p (a token outside the draft's support): accepted (p / 0 = +inf)
    target = _repeat_rows(np.array([[0.0, 0.0, 0.0]] * (K + 1), np.float32), B)
    draft = _repeat_rows(np.array([[0.0, 0.0, -np.inf]] * K, np.float32), B)
    out = orc.verify(target, draft, np.full((B, K), 2, np.int32), seed=8)
    assert np.all(out["num_accepted"] == K)
    # p = q = 0 (0/0): rejected
    target = _repeat_rows(np.array([[0.0, 0.0, -np.inf]] * (K + 1), np.float32), B)
    out = orc.verify(target, draft, np.full((B, K), 2, np.int32), seed=8)
    assert np.all(out["num_accepted"] == 0)


def test_k_zero_is_plain_sampling(orc):
    rng = np.random.default_rng(25)
    V, B = 14, 200_000
    tl = rng.normal(0, 1.5, size=(3, V)).astype(np.float32)
    target = _repeat_rows(tl, B)
    draft = _repeat_rows(tl[:2], B)
    kpr = np.zeros(B, np.int32)
    out = orc.verify(target, draft, None, kpr, seed=11, temperature=0.8, top_k=10)
    assert np.all(out["num_accepted"] == 0)
    _chi2_ok(out["tokens"][:, 0], orc.row_dist(tl[0].astype(np.float64), 0.8, top_k=10)[0],
             "K=0")
    assert np.all(out["tokens"][:, 1:] == -1)


def test_status_codes(orc):
    rng = np.random.default_rng(26)
    B, K, V = 8, 3, 6
    target = rng.normal(size=(B, K + 1, V)).astype(np.float32)
    draft = rng.normal(size=(B, K, V)).astype(np.float32)
    toks = rng.integers(0, V, size=(B, K)).astype(np.int32)
    kpr = np.array([3, -1, 4, 2, 3, 3, 1, 3], np.int32)
    toks[3, 2] = 999             # beyond K_b = 2: ignored
    toks[4, 1] = V               # out of range
    toks[5, 0] = -1              # out of range
    target[6, 3, 0] = np.nan     # row 3 is beyond K_b + 1 = 2 rows: never read
    target[7, 3, 2] = np.inf     # the bonus row of sequence 7: read
    out = orc.verify(target, draft, toks, kpr, seed=1)
    st = list(out["row_status"])
    assert st[0] in (O.ROW_OK,)
    assert st[1] == O.ROW_BAD_K and st[2] == O.ROW_BAD_K
    assert st[3] == O.ROW_OK
    assert st[4] == O.ROW_BAD_TOKEN and st[5] == O.ROW_BAD_TOKEN
    assert st[6] == O.ROW_OK
    assert st[7] == O.ROW_NONFINITE
    for b in (1, 2, 4, 5, 7):
        assert out["num_accepted"][b] == -1 and np.all(out["tokens"][b] == -1)
    # a draft row with no finite logit
    draft2 = draft.copy()
    draft2[0, 1, :] = -np.inf
    out = orc.verify(target, draft2, toks, kpr, seed=1)
    assert out["row_status"][0] == O.ROW_NONFINITE


def test_emitted_bounds_ragged(orc):
    from workloads import make_workload
    w = make_workload("ragged", B=40, K_max=6, V=300, ragged_k=(0, 6), seed=9,
                      temperature=0.9, top_k=40)
    toks, _ = orc.draft_sample(w.draft, w.k_per_row, temperature=0.9, top_k=40, seed=9)
    out = orc.verify(w.target, w.draft, toks, w.k_per_row, temperature=0.9, top_k=40, seed=9)
    for b in range(w.B):
        kb, n = w.k_per_row[b], out["num_accepted"][b]
        assert out["row_status"][b] == O.ROW_OK
        assert 0 <= n <= kb
        np.testing.assert_array_equal(out["tokens"][b, :n], toks[b, :n])
        assert 0 <= out["tokens"][b, n] < w.V
        assert np.all(out["tokens"][b, n + 1:] == -1)
        assert np.all(toks[b, kb:] == -1)


def test_draft_probs_input(orc):
    """Draft given as probabilities is used as given (no knobs)."""
    rng = np.random.default_rng(27)
    V, K, B = 8, 2, 100_000
    tl = rng.normal(0, 1.0, size=(K + 1, V)).astype(np.float32)
    q = rng.dirichlet(np.ones(V), size=K).astype(np.float32)
    target, draft = _repeat_rows(tl, B), _repeat_rows(q, B)
    toks, _ = orc.draft_sample(draft, draft_kind=O.DRAFT_PROBS, seed=12, top_k=3)
    _chi2_ok(toks[:, 0], q[0].astype(np.float64) / q[0].astype(np.float64).sum(), "probs draft")
    out = orc.verify(target, draft, toks, draft_kind=O.DRAFT_PROBS, seed=12, top_k=3,
                     temperature=0.9)
    Pt = orc.row_dist(tl[0].astype(np.float64), 0.9, top_k=3)[0]
    _chi2_ok(out["tokens"][:, 0], Pt, "position 0 (probs draft)")
    np.testing.assert_allclose(out["p_d_at_draft"][:, 0], q[0][toks[:, 0]].astype(np.float64))


def _layout_uniforms(orc, seed, rnd, b, j, tag):
    """Words of the verify stream: counter ((j << 2) | tag, b, round_lo, round_hi)."""
    ctr = np.array([[(j << 2) | tag, b, rnd & 0xFFFFFFFF, rnd >> 32]], np.uint32)
    w = orc.philox_batch(seed, ctr)[0]
    return [(int(x) >> 8) * 2.0 ** -24 for x in w]


def test_uniform_stream_layout(orc):
    """The counter layout of the uniforms: the accept test of slot j uses word
    0 of counter (j<<2 | 0, b, round), the resample at j* and the bonus at K_b
    use word 1 of their slot's counter, the drafted token uses word 0 of the
    tag-1 counter.  Checked against the separately pinned Philox and inverse
    CDF."""
    rng = np.random.default_rng(28)
    B, K, V = 64, 4, 11
    seed, rnd = 0xABCDEF0123, (5 << 32) + 77
    target = rng.normal(0, 1.5, size=(B, K + 1, V)).astype(np.float32)
    draft = (target[:, :K] + rng.normal(0, 1.5, size=(B, K, V))).astype(np.float32)
    kpr = rng.integers(0, K + 1, size=B).astype(np.int32)
    toks, _ = orc.draft_sample(draft, kpr, seed=seed, round=rnd)
    out = orc.verify(target, draft, toks, kpr, seed=seed, round=rnd)
    for b in range(B):
        for j in range(kpr[b]):
            Pd = orc.row_dist(draft[b, j].astype(np.float64), 1.0)[0]
            u = _layout_uniforms(orc, seed, rnd, b, j, 1)[0]
            assert toks[b, j] == orc.inverse_cdf(Pd, u)[0]
        n = out["num_accepted"][b]
        for j in range(n + (1 if n < kpr[b] else 0)):
            Pt = orc.row_dist(target[b, j].astype(np.float64), 1.0)[0]
            Pd = orc.row_dist(draft[b, j].astype(np.float64), 1.0)[0]
            x = toks[b, j]
            u_acc = _layout_uniforms(orc, seed, rnd, b, j, 0)[0]
            assert (u_acc < Pt[x] / Pd[x]) == (j < n)
        u_smp = _layout_uniforms(orc, seed, rnd, b, n, 0)[1]
        Pt = orc.row_dist(target[b, n].astype(np.float64), 1.0)[0]
        if n < kpr[b]:
            Pd = orc.row_dist(draft[b, n].astype(np.float64), 1.0)[0]
            R = np.maximum(Pt - Pd, 0.0)
        else:
            R = Pt
        assert out["tokens"][b, n] == orc.inverse_cdf(R, u_smp)[0]
