"""The roofline / speedup model (host-side) against the figures the pages print
from it, and its fit to measured step times (CPU)."""
import os

import numpy as np
import pytest

from speculative_decoding_verify_ragged_gb300 import roofline as rf

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "roofline_model.txt")


def _golden():
    g = {}
    for line in open(GOLDEN):
        line = line.split("#", 1)[0].split()
        if line:
            g[line[0]] = line[1:]
    return g


@pytest.fixture(scope="module")
def pages_model():
    g = _golden()
    return rf.StepModel(float(g["t_w_ms"][0]), float(g["k_ms"][0]), float(g["c_ms"][0])), g


def test_b_star_matches_printed(pages_model):
    m, g = pages_model
    for gamma, key in ((7, "b_star_gamma7"), (3, "b_star_gamma3")):
        want, tol = float(g[key][0]), float(g[key][1])
        assert abs(m.b_star(gamma) - want) <= tol


def test_best_gamma_per_batch_matches_printed(pages_model):
    m, g = pages_model
    for item in g["best_gamma"]:
        B, want = (int(x) for x in item.split(":"))
        assert rf.best_gamma(m, B, rf.decaying) == want, B


def test_break_even_matches_printed(pages_model):
    m, g = pages_model
    assert rf.break_even(m, 7, rf.decaying(7)) == int(g["break_even_decaying_gamma7"][0])
    assert rf.break_even(m, 8, rf.decaying(8)) == int(g["break_even_decaying_gamma8"][0])
    assert rf.break_even(m, 7, rf.expected_tokens_iid(0.6, 7)) == int(g["break_even_iid06_gamma7"][0])


def test_batch_one_speedup_matches_printed(pages_model):
    m, g = pages_model
    s = m.speedup(1, 7, rf.decaying(7))
    assert abs(s - float(g["speedup_batch1"][0])) <= float(g["speedup_batch1"][1])


def test_expected_tokens_closed_forms():
    assert abs(rf.expected_tokens_iid(0.8, 7) - 4.1611392) < 1e-6
    assert abs(rf.decaying(7) - 4.4875309) < 1e-6
    assert rf.expected_tokens_iid(1.0, 5) == 6.0
    assert rf.expected_tokens_conditional([]) == 1.0
    # the iid closed form is the conditional form with equal rates
    for a in (0.1, 0.5, 0.9):
        assert abs(rf.expected_tokens_iid(a, 6) - rf.expected_tokens_conditional([a] * 6)) < 1e-12


def test_rows_budget_is_the_compute_bound_threshold(pages_model):
    m, _ = pages_model
    # at B* the memory and compute times of a verify pass meet
    for gamma in (3, 7):
        B = m.b_star(gamma)
        assert abs((m.t_w + B * m.k) - m.c * B * (gamma + 1)) < 1e-9
        assert abs(m.rows_budget(B) - B * (gamma + 1)) < 1e-9


@pytest.mark.parametrize("noise", [0.0, 0.02])
def test_fit_recovers_parameters(noise):
    true = rf.StepModel(0.33, 0.0021, 0.00095)  # ms: a GB300-like step
    g = np.random.default_rng(5)
    pts = []
    for B in (1, 4, 16, 32, 64, 128):
        for gamma in (0, 1, 2, 3, 4, 7, 8):
            t = true.t_step(B, gamma + 1) * (1 + noise * g.standard_normal())
            pts.append((B, gamma + 1, t))
    m = rf.fit(pts)
    tol = 1e-6 if noise == 0 else 0.1
    assert abs(m.t_w - true.t_w) <= tol * true.t_w
    assert abs(m.c - true.c) <= tol * true.c
    assert abs(m.k - true.k) <= (tol if noise == 0 else 0.5) * true.k
    if noise == 0:
        assert abs(m.b_star(7) - true.b_star(7)) < 1e-6 * true.b_star(7)


def test_fit_needs_points():
    with pytest.raises(ValueError):
        rf.fit([(1, 1, 1.0)])


def test_fit_regimes_on_a_clean_max_model():
    """With steps that follow the max() model and regimes that separate cleanly,
    the regime fit returns the generating parameters."""
    true = rf.StepModel(0.32, 0.004, 0.0028)
    pts = [(B, g + 1, true.t_step(B, g + 1)) for B in (1, 4, 16, 32, 64, 128) for g in (0, 1, 3, 7)]
    m = rf.fit_regimes(pts, compute_rows=true.rows_budget(128) + 1)
    assert abs(m.t_w - true.t_step(1, 1)) < 1e-12 and abs(m.t_w - true.t_w) <= true.k + 1e-12
    assert abs(m.k - true.k) < 1e-9
    assert abs(m.c - true.c) < 1e-12
