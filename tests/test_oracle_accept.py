"""Pins of the acceptance oracle against what the pages and probability fix.

CPU only.  Each test checks the oracle against something other than itself:
the pages' worked example and printed expected-token counts, the exact law
of emitted tokens obtained by integrating over the uniforms, a chi-square
goodness-of-fit, the acceptance rate alpha = sum min(p, q), the greedy rule,
and library routines (scipy softmax) / brute-force characterisations of the
nucleus and the inverse CDF.
"""
import itertools
import json
import os

import numpy as np
import pytest
from scipy import special, stats

from oracle import accept as A

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def _gold(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


# ---------------------------------------------------------------- worked example
def test_worked_example_ratio_and_decisions():
    g = _gold("worked_example.json")
    z = np.log(np.array([g["p"], g["p"]]))          # softmax(log p) = p
    q = np.array([g["q"]])
    r = A.accept(z, q, [g["draft"]], [g["r_accept"], 0.5], 1.0)
    assert r.ratios[0] == pytest.approx(g["ratio"], abs=1e-12)
    assert r.n_accepted == 1 and r.tokens[0] == g["draft"] and r.bonus
    for u_draw in (0.0, 0.3, 0.999):
        r = A.accept(z, q, [g["draft"]], [g["r_reject"], u_draw], 1.0)
        assert r.n_accepted == 0
        # residual = max(0, p - q) = [0, 0.35, 0, 0]: only 'green' has mass
        assert r.tokens[0] == g["favoured_on_reject"]
        assert r.tokens[1] == -1


# ---------------------------------------------------------------- softmax / nucleus
def test_softmax_matches_scipy():
    g = np.random.default_rng(0)
    for T in (0.3, 1.0, 2.5):
        z = g.normal(0, 3, size=257).astype(np.float32)
        np.testing.assert_allclose(A.softmax_t(z, T),
                                   special.softmax(z.astype(np.float64) / T),
                                   rtol=1e-13, atol=0)


def _nucleus_bruteforce(P, top_p):
    """tau = the largest probability value v with mass(P >= v) >= top_p."""
    cands = sorted(set(P.tolist()), reverse=True)
    for v in cands:
        if P[P >= v].sum() >= top_p:
            keep = P >= v
            return np.where(keep, P, 0) / P[keep].sum()
    raise AssertionError


def test_nucleus_hand_cases():
    P = np.array([0.5, 0.2, 0.2, 0.1])
    out, info = A.nucleus(P, 0.6)         # crossing at a tie: both 0.2 kept
    np.testing.assert_allclose(out, [0.5 / 0.9, 0.2 / 0.9, 0.2 / 0.9, 0])
    assert info.kept == 3
    out, info = A.nucleus(P, 0.5)         # mass reaches exactly top_p at k*=0
    np.testing.assert_allclose(out, [1, 0, 0, 0])
    assert info.boundary
    out, _ = A.nucleus(P, 1.0)            # no-op
    np.testing.assert_array_equal(out, P)
    out, _ = A.nucleus(np.array([0.4, 0.4, 0.2]), 1e-9)   # -> argmax set
    np.testing.assert_allclose(out, [0.5, 0.5, 0])
    with pytest.raises(ValueError):
        A.nucleus(P, 0.0)


def test_nucleus_matches_bruteforce_characterisation():
    g = np.random.default_rng(1)
    for trial in range(300):
        V = int(g.integers(2, 9))
        # coarse values so that ties occur often
        w = g.integers(1, 6, size=V).astype(np.float64)
        P = w / w.sum()
        top_p = float(g.uniform(0.05, 0.999))
        out, _ = A.nucleus(P, top_p)
        np.testing.assert_allclose(out, _nucleus_bruteforce(P, top_p), rtol=1e-12, atol=1e-15)


# ---------------------------------------------------------------- inverse CDF
def test_inverse_cdf_bins_and_zero_mass():
    w = np.array([0.0, 1.0, 0.0, 2.0, 0.0, 0.5])
    S = w.sum()
    edges = np.concatenate([[0.0], np.cumsum(w)]) / S
    for u in np.linspace(0, 1, 1001, endpoint=False):
        t = A.inverse_cdf(w, u).token
        assert w[t] > 0
        assert edges[t] <= u < edges[t + 1]
    assert A.inverse_cdf(w, 0.0).token == 1


# ---------------------------------------------------------------- exact law, V=3, gamma=2
def _cells(breaks):
    """Midpoints and lengths of the cells of [0,1) cut at the given points."""
    b = np.unique(np.clip(np.concatenate([[0.0, 1.0], breaks]), 0, 1))
    b = b[np.diff(b, prepend=-1) > 1e-15]
    return [((lo + hi) / 2, hi - lo) for lo, hi in zip(b[:-1], b[1:]) if hi - lo > 0]


def test_exact_law_by_integration_over_uniforms():
    """Integrate the oracle's output over the draft tokens and all three
    uniforms; at every position the emitted token must follow p exactly
    (pigeon guide, 'Why the output is exactly p')."""
    P = np.array([[0.5, 0.3, 0.2], [0.1, 0.6, 0.3], [0.25, 0.25, 0.5]])
    Q = np.array([[0.2, 0.2, 0.6], [0.4, 0.4, 0.2]])
    z = np.log(P)
    # where the u_gamma draw can change: CDF points of every row it may use
    breaks = []
    for i in range(2):
        r = np.maximum(P[i] - Q[i], 0)
        breaks += list(np.cumsum(r) / r.sum())
    breaks += list(np.cumsum(P[2]))
    draw_cells = _cells(np.array(breaks))
    law = {}
    for x1, x2 in itertools.product(range(3), repeat=2):
        wx = Q[0, x1] * Q[1, x2]
        a0 = min(1, P[0, x1] / Q[0, x1])
        a1 = min(1, P[1, x2] / Q[1, x2])
        for u0, w0 in _cells(np.array([a0])):
            for u1, w1 in _cells(np.array([a1])):
                for u2, w2 in draw_cells:
                    r = A.accept(z, Q, [x1, x2], [u0, u1, u2], 1.0)
                    key = tuple(t for t in r.tokens if t >= 0)
                    law[key] = law.get(key, 0.0) + wx * w0 * w1 * w2
    assert sum(law.values()) == pytest.approx(1.0, abs=1e-12)
    # position 0 ~ P0
    for a in range(3):
        assert sum(m for k, m in law.items() if k[0] == a) == pytest.approx(P[0, a], abs=1e-12)
    # given the pass reached position k with prefix h, token k ~ P_k
    for k in (1, 2):
        for h in itertools.product(range(3), repeat=k):
            reach = sum(m for s, m in law.items() if len(s) > k and s[:k] == h)
            for b in range(3):
                got = sum(m for s, m in law.items() if len(s) > k and s[:k] == h and s[k] == b)
                assert got == pytest.approx(reach * P[k, b], abs=1e-12)


# ---------------------------------------------------------------- sampling pins
def _simulate(P, Q, gamma, trials, seed, T=1.0):
    """Run the oracle on i.i.d. drafts x ~ q (drawn by the oracle's own
    inverse CDF) and uniforms; return list of AcceptResult."""
    g = np.random.default_rng(seed)
    z = np.log(P)
    out = []
    for _ in range(trials):
        ud = g.random(gamma)
        xs = [A.inverse_cdf(Q[i], ud[i]).token for i in range(gamma)]
        out.append(A.accept(z, Q, xs, g.random(gamma + 1), T))
    return out


def test_chi_square_v8_every_position_follows_p():
    """V=8, gamma=4, fixed (p, q) rows that differ per position; the token
    emitted at position k (given the pass reached k) must follow P_k
    (10^6 passes, the trial count the parity bar names)."""
    V, gamma = 8, 4
    g = np.random.default_rng(7)
    P = g.dirichlet(np.ones(V), size=gamma + 1)
    Q = np.clip(P[:gamma] + g.normal(0, 0.08, size=(gamma, V)), 0.01, None)
    Q /= Q.sum(1, keepdims=True)
    res = _simulate(P, Q, gamma, 1_000_000, seed=11)
    toks = np.array([r.tokens for r in res])
    for k in range(gamma + 1):
        col = toks[:, k]
        col = col[col >= 0]
        obs = np.bincount(col, minlength=V)
        chi = stats.chisquare(obs, P[k] * col.size)
        assert chi.pvalue > 1e-3, (k, chi)


def test_acceptance_rate_equals_alpha():
    """First-draft acceptance frequency = alpha = sum min(p, q) (pigeon
    guide, 'Speed')."""
    V = 8
    g = np.random.default_rng(3)
    p = g.dirichlet(np.ones(V))
    q = g.dirichlet(np.ones(V))
    alpha = np.minimum(p, q).sum()
    res = _simulate(np.array([p, p]), np.array([q]), 1, 100_000, seed=5)
    acc = np.mean([r.n_accepted for r in res])
    sd = np.sqrt(alpha * (1 - alpha) / len(res))
    assert abs(acc - alpha) < 4 * sd


@pytest.mark.parametrize("alpha,gamma,printed", [
    (0.7, 5, 2.94), (0.8, 4, 3.36), (0.8, 8, 4.33)])
def test_mean_tokens_per_pass_matches_printed(alpha, gamma, printed):
    """Two-token vocabulary with sum min(p,q) = alpha; the mean number of
    emitted tokens per pass must hit the pages' printed values."""
    gold = _gold("expected_tokens.json")
    assert any(e["alpha"] == alpha and e["gamma"] == gamma and e["value"] == printed
               for e in gold["printed"])
    p = np.array([0.9, 0.1])
    q = np.array([0.9 - (1 - alpha) + 0.0, 0.1 + (1 - alpha)])   # min-sum = alpha
    assert np.minimum(p, q).sum() == pytest.approx(alpha)
    P = np.tile(p, (gamma + 1, 1))
    Q = np.tile(q, (gamma, 1))
    res = _simulate(P, Q, gamma, 40_000, seed=int(alpha * 100) + gamma)
    n = np.array([r.n_accepted + 1 for r in res], dtype=np.float64)
    se = n.std() / np.sqrt(n.size)
    assert abs(n.mean() - printed) < 4 * se + 0.005 + 1e-9


@pytest.mark.parametrize("alpha", [0.5, 0.8])
def test_mean_tokens_per_pass_at_gamma_2(alpha):
    """gamma = 2 has no printed example: the mean emitted tokens per pass of
    the oracle's rule must equal the expanded geometric sum 1 + alpha +
    alpha^2 (the chance of reaching each position), and the controller's
    closed form must give the same number."""
    from oracle import gamma as OG
    p = np.array([0.9, 0.1])
    q = np.array([0.9 - (1 - alpha), 0.1 + (1 - alpha)])
    assert np.minimum(p, q).sum() == pytest.approx(alpha)
    expect = 1.0 + alpha + alpha * alpha
    assert OG.expected_tokens(alpha, 2) == pytest.approx(expect, abs=1e-12)
    res = _simulate(np.tile(p, (3, 1)), np.tile(q, (2, 1)), 2, 40_000, seed=int(alpha * 10) + 2)
    n = np.array([r.n_accepted + 1 for r in res], dtype=np.float64)
    se = n.std() / np.sqrt(n.size)
    assert abs(n.mean() - expect) < 4 * se + 1e-9


def test_printed_slips_are_not_the_formula():
    """The pages print a few values that disagree with their own formula;
    the oracle follows the formula (recorded in the fixture)."""
    for e in _gold("expected_tokens.json")["printed_but_inconsistent_with_the_formula"]:
        a, k = e["alpha"], e["gamma"]
        f = (1 - a ** (k + 1)) / (1 - a)
        assert abs(f - e["formula"]) < 0.006 and abs(f - e["value"]) > 0.05


# ---------------------------------------------------------------- greedy
def test_greedy_rule():
    V, gamma = 16, 4
    g = np.random.default_rng(9)
    for _ in range(200):
        z = g.normal(size=(gamma + 1, V)).astype(np.float32)
        am = z.argmax(1)
        xs = [int(am[i]) if g.random() < 0.7 else int(g.integers(V)) for i in range(gamma)]
        r = A.accept(z, None, xs, None, 0.0)
        n = 0
        while n < gamma and xs[n] == am[n]:
            n += 1
        assert r.n_accepted == n
        assert r.tokens[:n] == xs[:n]
        assert r.tokens[n] == am[n]
        assert all(t == -1 for t in r.tokens[n + 1:])


def test_greedy_ties_take_lowest_id():
    z = np.array([[1.0, 3.0, 3.0], [2.0, 2.0, 0.0]])
    r = A.accept(z, None, [2], None, 0.0)
    assert r.tokens == [1, -1] and r.n_accepted == 0
    r = A.accept(z, None, [1], None, 0.0)
    assert r.tokens == [1, 0] and r.bonus


def test_zero_q_for_draft_raises():
    z = np.zeros((2, 3))
    with pytest.raises(ValueError):
        A.accept(z, np.array([[0.5, 0.5, 0.0]]), [2], [0.1, 0.1], 1.0)


def test_topp_applies_to_target_rows():
    """With top-p a drafted token outside the target nucleus is always
    rejected and the correction comes from inside it."""
    P = np.array([0.6, 0.3, 0.1])
    z = np.log(np.array([P, P]))
    q = np.array([[0.2, 0.2, 0.6]])
    for u in np.linspace(0, 0.99, 23):
        r = A.accept(z, q, [2], [u, u], 1.0, top_p=0.8)
        assert r.n_accepted == 0 and r.tokens[0] in (0, 1)


def test_draft_sample_pins():
    """The draft sampler on its own: at top_p = 1, q is torch's fp64 softmax
    of z / T; its draws with uniform u follow q (chi-square, 2e5 draws); at
    T = 0 it is the one-hot argmax with the lowest id on ties."""
    import torch
    g = np.random.default_rng(23)
    V, T = 12, 0.7
    z = g.normal(0, 2, size=(1, V))
    q, _, _ = A.draft_sample(z, [0.5], T, 1.0)
    ref = torch.softmax(torch.from_numpy(z[0]) / T, dim=0).numpy()
    np.testing.assert_allclose(q[0], ref, rtol=1e-12, atol=1e-15)
    n = 200_000
    u = g.random(n)
    zz = np.repeat(z, 64, axis=0)
    toks = np.concatenate([A.draft_sample(zz, u[i:i + 64], T, 1.0)[1] for i in range(0, n, 64)])
    obs = np.bincount(toks, minlength=V)
    chi = stats.chisquare(obs, ref * n)
    assert chi.pvalue > 1e-3, chi
    zt = np.array([[0.0, 3.0, 1.0, 3.0]])
    q0, t0, _ = A.draft_sample(zt, [0.9], 0.0)
    assert t0[0] == 1 and q0[0].tolist() == [0.0, 1.0, 0.0, 0.0]


def test_draft_sample_uses_same_rule():
    g = np.random.default_rng(4)
    z = g.normal(0, 2, size=(3, 50)).astype(np.float32)
    u = g.random(3).astype(np.float32)
    q, t, _ = A.draft_sample(z, u, 0.8, 0.9)
    for r in range(3):
        P, _ = A.target_dist(z[r], 0.8, 0.9)
        np.testing.assert_allclose(q[r], P)
        assert t[r] == A.inverse_cdf(P, u[r]).token
