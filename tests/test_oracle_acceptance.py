"""Pins for the oracle's acceptance and sampling rule (CPU only).

Each test checks the oracle against something other than itself: a closed
form the pages print, a value the pages print, the lossless property the
pages state (chi-square against the target distribution), or a special case
with a known answer.
"""
import math
import os

import numpy as np
import pytest
from scipy import stats

from oracle import analytic
from oracle import verify_step as o
import workloads as wl

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def _rng(seed):
    return np.random.default_rng(seed)


def _u24(g, n):
    return (g.integers(0, 1 << 24, size=n) / float(1 << 24)).astype(np.float32)


# ---------------------------------------------------------------------------
# printed values
# ---------------------------------------------------------------------------

def test_closed_forms_match_printed_values():
    for model, a0, step, gamma, printed, dec in _rows("expected_tokens.txt"):
        gamma, dec = int(gamma), int(dec)
        if model == "iid":
            e = analytic.expected_tokens(float(a0), gamma)
        else:
            e = analytic.expected_tokens_conditional(analytic.decaying_alphas(gamma, float(a0), float(step)))
        assert round(e, dec) == pytest.approx(float(printed)), (model, e)
    for a0, step, g0, g1, printed, dec in _rows("decaying_gain.txt"):
        e0 = analytic.expected_tokens_conditional(analytic.decaying_alphas(int(g0), float(a0), float(step)))
        e1 = analytic.expected_tokens_conditional(analytic.decaying_alphas(int(g1), float(a0), float(step)))
        assert round(e1 - e0, int(dec)) == pytest.approx(float(printed))


def test_primer_example_token_counts():
    """3 of 4 right -> 4 tokens, none right -> 1, through the oracle's rule."""
    V = 8
    for gamma, acc, produced in _rows("primer_example.txt"):
        gamma, acc, produced = int(gamma), int(acc), int(produced)
        p = np.full((gamma + 1, V), 1.0 / V, dtype=np.float32)
        q = np.zeros((gamma, V), dtype=np.float32)
        drafts = np.zeros(gamma, dtype=np.int64)
        for i in range(gamma):
            if i < acc:
                q[i] = p[i]                  # q = p at the token: always accepted
            else:
                q[i, 0] = 1.0                # q puts all mass where p has 1/V
        # u = 0.5 rejects the first draft not in agreement (u*q = 0.5 >= 1/8)
        u = np.full(gamma + 1, 0.5, dtype=np.float32)
        a, t = o.accept_and_sample(p, q, drafts, u)
        acc_tokens, emitted, eoff, _ = o.accept_batch(p, q, np.concatenate([[3], drafts]), u, [gamma])
        assert a == acc
        assert len(emitted) == produced == a + 1
        assert 0 <= t < V


def test_draft_budget_rule_matches_printed_table():
    for budget, live, per_agent in _rows("draft_budget.txt"):
        assert wl.swarm_gamma(int(live), budget=int(budget), cap=1 << 20) == int(per_agent)


# ---------------------------------------------------------------------------
# Monte Carlo against the closed forms
# ---------------------------------------------------------------------------

def _mc_expected_tokens(alphas, n, seed):
    """Draft token 0 with q(0) = 0.5 and p(0) = alpha_k / 2: accepted w.p. alpha_k."""
    V = 4
    gamma = len(alphas)
    g = _rng(seed)
    p = np.full((gamma + 1, V), 0.0, dtype=np.float32)
    q = np.full((gamma, V), 0.0, dtype=np.float32)
    for k, a in enumerate(alphas):
        q[k] = [0.5, 0.5, 0.0, 0.0]
        p[k] = [a / 2, 0.0, (1 - a / 2) / 2, (1 - a / 2) / 2]
    p[gamma] = 0.25
    drafts = np.zeros(gamma, dtype=np.int64)
    counts = np.empty(n)
    for t in range(n):
        a, tok = o.accept_and_sample(p, q, drafts, _u24(g, gamma + 1))
        counts[t] = a + 1
    return counts.mean(), counts.std(ddof=1) / math.sqrt(n)


def test_monte_carlo_iid_expected_tokens():
    alpha, gamma = 0.8, 7
    mean, se = _mc_expected_tokens([alpha] * gamma, 40000, 11)
    e = analytic.expected_tokens(alpha, gamma)
    assert abs(mean - e) < 4 * se, (mean, e, se)
    # a count that forgot the final token would sit at e - 1
    assert abs(mean - (e - 1)) > 20 * se


def test_monte_carlo_decaying_expected_tokens():
    alphas = analytic.decaying_alphas(7)
    mean, se = _mc_expected_tokens(alphas, 40000, 12)
    e = analytic.expected_tokens_conditional(alphas)
    assert abs(mean - e) < 4 * se, (mean, e, se)
    # the iid model at the mean acceptance gives a different number
    assert abs(mean - analytic.expected_tokens(0.8, 7)) > 8 * se


# ---------------------------------------------------------------------------
# lossless: emitted tokens follow the target distribution
# ---------------------------------------------------------------------------

def _markov(g, V, conc):
    m = g.dirichlet(np.full(V, conc), size=V)
    return m.astype(np.float32)


def _draw(g, w):
    c = np.cumsum(w.astype(np.float64))
    return int(min(np.searchsorted(c, g.random() * c[-1], side="right"), len(w) - 1))


def _one_step(M, Q, ctx, gamma, g):
    """One speculative step with a Markov target M and a Markov drafter Q."""
    drafts = []
    prev = ctx
    for _ in range(gamma):
        x = _draw(g, Q[prev])
        drafts.append(x)
        prev = x
    inputs = [ctx] + drafts
    p_rows = np.stack([M[t] for t in inputs])
    q_rows = np.stack([Q[t] for t in inputs[:gamma]]) if gamma else np.zeros((0, M.shape[1]), np.float32)
    a, t = o.accept_and_sample(p_rows, q_rows, np.array(drafts, dtype=np.int64), _u24(g, gamma + 1))
    return drafts[:a] + [t]


@pytest.mark.parametrize("gamma", [1, 3])
def test_chi_square_first_token_is_target(gamma):
    V, n = 12, 60000
    g = _rng(100 + gamma)
    M = _markov(g, V, 0.7)
    Q = _markov(g, V, 0.7)
    ctx = 5
    counts = np.zeros(V)
    for _ in range(n):
        counts[_one_step(M, Q, ctx, gamma, g)[0]] += 1
    expected = M[ctx].astype(np.float64) / M[ctx].sum() * n
    keep = expected > 5
    stat = ((counts[keep] - expected[keep]) ** 2 / expected[keep]).sum()
    pval = stats.chi2.sf(stat, keep.sum() - 1)
    assert pval > 1e-4, (stat, pval)


def test_chi_square_two_tokens_follow_chain():
    """The first two generated tokens (across steps if needed) ~ M[ctx][y1] M[y1][y2]."""
    V, n, gamma = 6, 60000, 3
    g = _rng(7)
    M = _markov(g, V, 0.8)
    Q = _markov(g, V, 0.8)
    ctx = 2
    counts = np.zeros((V, V))
    for _ in range(n):
        out = _one_step(M, Q, ctx, gamma, g)
        if len(out) < 2:
            out = out + _one_step(M, Q, out[0], gamma, g)
        counts[out[0], out[1]] += 1
    Mf = M.astype(np.float64)
    Mf /= Mf.sum(axis=1, keepdims=True)
    expected = (Mf[ctx][:, None] * Mf) * n
    keep = expected > 5
    stat = ((counts[keep] - expected[keep]) ** 2 / expected[keep]).sum()
    pval = stats.chi2.sf(stat, keep.sum() - 1)
    assert pval > 1e-4, (stat, pval)


def test_chi_square_detects_a_planted_mistake():
    """Power check: resampling from p instead of the residual breaks the marginal."""
    V, n, gamma = 12, 60000, 1
    g = _rng(9)
    M = _markov(g, V, 0.7)
    Q = _markov(g, V, 0.7)
    ctx = 5
    counts = np.zeros(V)
    for _ in range(n):
        x = _draw(g, Q[ctx])
        u = _u24(g, 2)
        if o.accepts(M[ctx][x], Q[ctx][x], u[0]):
            y = x
        else:
            y = o.inverse_cdf_int(M[ctx], u[1])     # planted: not the residual
        counts[y] += 1
    expected = M[ctx].astype(np.float64) / M[ctx].sum() * n
    keep = expected > 5
    stat = ((counts[keep] - expected[keep]) ** 2 / expected[keep]).sum()
    assert stats.chi2.sf(stat, keep.sum() - 1) < 1e-6


# ---------------------------------------------------------------------------
# special cases
# ---------------------------------------------------------------------------

def test_gamma_zero_is_plain_sampling():
    g = _rng(3)
    V = 50
    for _ in range(200):
        p = g.dirichlet(np.ones(V)).astype(np.float32)
        u = _u24(g, 1)
        a, t = o.accept_and_sample(p[None, :], np.zeros((0, V), np.float32), [], u)
        assert a == 0
        assert t == o.inverse_cdf_int(p, u[0])


def test_q_equal_p_accepts_everything():
    g = _rng(4)
    V, gamma = 40, 6
    for _ in range(200):
        p = g.dirichlet(np.ones(V), size=gamma + 1).astype(np.float32)
        drafts = g.integers(0, V, size=gamma)
        u = _u24(g, gamma + 1)
        a, t = o.accept_and_sample(p, p[:gamma], drafts, u)
        assert a == gamma
        # all accepted: the bonus token comes from p at the last row
        assert t == o.inverse_cdf_int(p[gamma], u[gamma])


def test_target_zero_probability_is_rejected():
    V = 10
    p = np.full((2, V), 0.1, dtype=np.float32)
    p[0, 3] = 0.0
    p[0, 4] = 0.2
    q = np.full((1, V), 0.1, dtype=np.float32)
    for u0 in (0.0, 0.5, 0.999):
        a, t = o.accept_and_sample(p, q, [3], np.array([u0, 0.3], dtype=np.float32))
        assert a == 0
        # residual max(0, p - q) puts all mass on token 4
        assert t == 4


def test_p_equals_q_at_zero_is_rejected():
    p = np.array([[0.0, 1.0], [0.5, 0.5]], dtype=np.float32)
    q = np.array([[0.0, 1.0]], dtype=np.float32)
    a, t = o.accept_and_sample(p, q, [0], np.array([0.0, 0.0], dtype=np.float32))
    assert a == 0
    # residual sums to zero -> falls back to p
    assert t == 1


def test_acceptance_threshold_is_p_over_q():
    """Accept iff u < p/q: sweep u across the threshold on the 24-bit grid."""
    p, q = np.float32(0.375), np.float32(0.75)      # p/q = 0.5 exactly
    assert o.accepts(p, q, np.float32(0.5 - 2 ** -24))
    assert not o.accepts(p, q, np.float32(0.5))
    assert o.accepts(np.float32(0.8), np.float32(0.75), np.float32(0.9999999))


def test_inverse_cdf_hand_cases():
    w = np.array([0.25, 0.5, 0.25], dtype=np.float32)
    # S = 2^32; T = floor(S * floor(u 2^24) / 2^24) = floor(u 2^24) * 2^8
    assert o.inverse_cdf_int(w, np.float32(0.0)) == 0
    assert o.inverse_cdf_int(w, np.float32(0.25 - 2 ** -24)) == 0
    assert o.inverse_cdf_int(w, np.float32(0.25)) == 1
    assert o.inverse_cdf_int(w, np.float32(0.3)) == 1
    assert o.inverse_cdf_int(w, np.float32(0.75 - 2 ** -24)) == 1
    assert o.inverse_cdf_int(w, np.float32(0.75)) == 2
    assert o.inverse_cdf_int(w, np.float32(1 - 2 ** -24)) == 2
    # zero-weight entries are never chosen
    w2 = np.array([0.0, 0.5, 0.0, 0.5, 0.0], dtype=np.float32)
    for u in np.linspace(0, 1 - 2 ** -24, 101, dtype=np.float32):
        assert o.inverse_cdf_int(w2, u) in (1, 3)
    assert o.inverse_cdf_int(np.zeros(4, np.float32), np.float32(0.5)) == -1


def test_inverse_cdf_matches_brute_force_on_tiny_weights():
    """Brute force: enumerate every 24-bit u on a coarse grid, count hits per index."""
    g = _rng(5)
    for _ in range(20):
        k = g.integers(1, 8, size=5)
        w = (k / 16.0).astype(np.float32)              # exact dyadic weights
        tot = k.sum()
        hits = np.zeros(5, dtype=np.int64)
        grid = 4096
        for i in range(grid):
            hits[o.inverse_cdf_int(w, np.float32(i / grid))] += 1
        # with dyadic weights and a grid finer than 1/tot, each index gets
        # exactly its share of the grid (up to the rounding of boundaries)
        assert np.all(np.abs(hits - grid * k / tot) <= 1), (hits, grid * k / tot)


def test_accept_histogram_counts():
    tested, accepted = o.accept_histogram([0, 2, 3, 1], [3, 3, 3, 0], 3)
    # slot0: tested pos0 only; slot1: tested 0,1,2 accepted 0,1; slot2: all accepted; slot3: none
    assert list(tested) == [3, 2, 2]
    assert list(accepted) == [2, 2, 1]
