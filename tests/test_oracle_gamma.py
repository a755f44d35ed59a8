"""Pins of the dynamic-gamma oracle (CPU only).

Expected tokens per pass against the values the pages print
(tests/golden/expected_tokens.json) and against a simulation of independent
per-draft coins; the chosen depth against the empirical tokens-per-ms of
simulated passes at every candidate depth; the limits (alpha = 0 takes the
shallowest depth, alpha -> 1 with a costly target the deepest); the page's
statement that below alpha = 0.65 a depth beyond 4 does not pay (its 2 ms /
20 ms costs); and the window / warm-up behaviour of the controller.
"""
import json
import os

import numpy as np
import pytest

from oracle import gamma as G

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "expected_tokens.json")


def test_expected_tokens_printed_values():
    with open(GOLDEN) as f:
        g = json.load(f)
    for e in g["printed"]:
        assert round(G.expected_tokens(e["alpha"], e["gamma"]), 2) == e["value"]
    for e in g["printed_but_inconsistent_with_the_formula"]:
        assert round(G.expected_tokens(e["alpha"], e["gamma"]), 2) == e["formula"]


def _simulate(alpha, gamma, N, rng):
    """Tokens per pass: accepted drafts until the first failed coin (at most
    gamma), plus one correction / bonus token."""
    coins = rng.random((N, gamma)) < alpha
    acc = np.cumprod(coins, axis=1).sum(axis=1) if gamma else np.zeros(N)
    return acc + 1.0


def test_expected_tokens_against_simulated_coins():
    rng = np.random.default_rng(1)
    for alpha in (0.3, 0.65, 0.8, 0.95):
        for gamma in (0, 1, 4, 8):
            t = _simulate(alpha, gamma, 200000, rng)
            se = t.std() / np.sqrt(t.size) + 1e-12
            assert abs(t.mean() - G.expected_tokens(alpha, gamma)) < 4 * se + 1e-9


def test_optimal_gamma_matches_simulated_throughput():
    rng = np.random.default_rng(2)
    for alpha, td, tt in ((0.5, 2.0, 20.0), (0.65, 2.0, 20.0), (0.8, 2.0, 20.0), (0.9, 1.0, 20.0),
                          (0.8, 5.0, 10.0)):
        rates, ses = [], []
        for g in range(2, 9):
            t = _simulate(alpha, g, 400000, rng)
            rates.append(t.mean() / (g * td + tt))
            ses.append(t.std() / np.sqrt(t.size) / (g * td + tt))
        rates = np.array(rates)
        best = int(np.argmax(rates)) + 2
        order = np.argsort(-rates)
        gap = rates[order[0]] - rates[order[1]]
        choice = G.optimal_gamma(alpha, 2, 8, td, tt)
        if gap > 4 * (ses[order[0]] + ses[order[1]]):
            assert choice == best, (alpha, td, tt, choice, best)
        else:   # a near tie: the choice is one of the two best
            assert choice in (order[0] + 2, order[1] + 2)


def test_limits_and_the_pages_statement():
    assert G.optimal_gamma(0.0, 2, 8, 2.0, 20.0) == 2
    assert G.optimal_gamma(1.0, 2, 8, 2.0, 20.0) == 8
    assert G.optimal_gamma(0.999, 2, 8, 2.0, 20.0) == 8
    for alpha in (0.4, 0.5, 0.6, 0.64):
        assert G.optimal_gamma(alpha, 2, 8, 2.0, 20.0) <= 4
    # a higher acceptance never asks for a shallower depth
    gs = [G.optimal_gamma(a, 2, 8, 2.0, 20.0) for a in np.linspace(0, 1, 101)]
    assert all(x <= y for x, y in zip(gs, gs[1:]))


def test_controller_window_and_warmup():
    c = G.Controller(gamma_init=4, window=20, min_records=5)
    assert c.alpha() == 0.80
    for _ in range(4):
        assert c.record(4, 0) == 4            # fewer than 5 passes: no decision
    assert c.record(4, 0) == 2                # alpha 0: the shallowest depth
    for _ in range(20):
        c.record(4, 4)                        # the window now holds only full accepts
    assert c.alpha() == 1.0 and c.gamma == 8
    c.record(8, 0)                            # one rejection-only pass among 20
    assert abs(c.alpha() - (19 * 4) / (19 * 4 + 8)) < 1e-12
    with pytest.raises(ValueError):
        c.record(4, 5)
