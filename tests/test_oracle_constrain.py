"""Pins of the constrained-acceptance oracle (CPU only).

The masked target distribution must equal the target restricted to the
allowed set and renormalised (computed here from the closed form with
scipy's softmax over the allowed entries only); with the same mask on both
sides the rule must emit exactly that distribution (chi-square) with the
acceptance rate sum_x min(p_m, q_m), and never a disallowed token; a mask on
the draft side alone must break it (the pages' warning); an all-allowed mask
is the identity and an empty row is refused.
"""
import numpy as np
import pytest
from scipy import special, stats

from oracle import accept as OA
from oracle import constrain as OC


def _mask(rng, shape, p_allow=0.5):
    a = rng.random(shape) < p_allow
    a[..., 0] |= ~a.any(axis=-1)          # at least one allowed token per row
    return a


def test_masked_distribution_is_the_restricted_softmax():
    rng = np.random.default_rng(1)
    for V, T in ((8, 1.0), (50, 0.7), (1000, 1.3)):
        z = rng.normal(0, 2, size=V)
        a = _mask(rng, V, 0.3)
        P, _ = OA.target_dist(OC.apply_mask(z, a), T, 1.0)
        ref = np.zeros(V)
        ref[a] = special.softmax(z[a] / T)
        np.testing.assert_allclose(P, ref, rtol=1e-12, atol=1e-300)
        assert (P[~a] == 0).all()


def test_masked_nucleus_keeps_only_allowed_tokens():
    rng = np.random.default_rng(2)
    V = 200
    z = rng.normal(0, 2, size=V)
    a = _mask(rng, V, 0.2)
    P, info = OA.target_dist(OC.apply_mask(z, a), 1.0, 0.9)
    assert (P[~a] == 0).all() and abs(P.sum() - 1) < 1e-12
    # the nucleus of the masked row is the nucleus of the restricted softmax
    Pr = np.zeros(V)
    Pr[a] = special.softmax(z[a])
    Pn, _ = OA.nucleus(Pr, 0.9)
    np.testing.assert_allclose(P, Pn, rtol=1e-12)


def test_same_mask_on_both_sides_emits_the_masked_target():
    """V=8, gamma=1: the first emitted token follows p restricted to the mask
    (chi-square over 200000 trials), the acceptance rate is
    sum_x min(p_m(x), q_m(x)), and no disallowed token is ever emitted."""
    rng = np.random.default_rng(3)
    V, N = 8, 200000
    zp = rng.normal(0, 1.5, size=(2, V))
    zq = zp + rng.normal(0, 1.0, size=(2, V))
    a = np.array([[1, 0, 1, 1, 0, 1, 0, 1]] * 2, dtype=bool)
    zpm, zqm = OC.apply_mask(zp, a), OC.apply_mask(zq, a)
    pm, _ = OA.target_dist(zpm[0], 1.0)
    qm, _ = OA.target_dist(zqm[0], 1.0)
    counts = np.zeros(V)
    acc = 0
    ud = rng.random(N)
    uu = rng.random((N, 2))
    cq = np.cumsum(qm)
    xs = np.minimum(np.searchsorted(cq, ud * cq[-1], side="right"), V - 1)
    for k in range(N):
        r = OA.accept(zpm, qm[None, :], [int(xs[k])], uu[k], 1.0)
        counts[r.tokens[0]] += 1
        acc += r.n_accepted
    assert counts[~a[0]].sum() == 0
    keep = a[0]
    assert stats.chisquare(counts[keep], pm[keep] * N).pvalue > 1e-3
    alpha = np.minimum(pm, qm).sum()
    se = np.sqrt(alpha * (1 - alpha) / N)
    assert abs(acc / N - alpha) < 4 * se


def test_mask_on_the_draft_side_only_breaks_the_rule():
    """The target unmasked, the draft masked: residual and bonus draws come
    from the unmasked p, so disallowed tokens are emitted and the output is
    no longer the masked target."""
    rng = np.random.default_rng(4)
    V, N = 8, 20000
    zp = rng.normal(0, 1.5, size=(2, V))
    a = np.array([[1, 0, 1, 1, 0, 1, 0, 1]] * 2, dtype=bool)
    qm, _ = OA.target_dist(OC.apply_mask(zp + rng.normal(0, 1.0, size=(2, V)), a)[0], 1.0)
    cq = np.cumsum(qm)
    bad = 0
    for k in range(N):
        x = int(min(np.searchsorted(cq, rng.random() * cq[-1], side="right"), V - 1))
        r = OA.accept(zp, qm[None, :], [x], rng.random(2), 1.0)
        bad += not a[0, r.tokens[0]]
    assert bad > 0.05 * N


def test_greedy_with_a_mask_takes_the_allowed_argmax():
    z = np.array([[5.0, 1.0, 3.0, 2.0], [0.0, 4.0, 1.0, 9.0]])
    a = np.array([[0, 1, 1, 1], [1, 1, 1, 0]], dtype=bool)
    r = OA.accept(OC.apply_mask(z, a), None, [2], None, 0.0)
    assert r.tokens == [2, 1] and r.n_accepted == 1


def test_all_allowed_is_identity_and_empty_rows_are_refused():
    rng = np.random.default_rng(5)
    z = rng.normal(size=(3, 17))
    np.testing.assert_array_equal(OC.apply_mask(z, np.ones_like(z, dtype=bool)), z)
    a = np.ones((3, 17), dtype=bool)
    a[1] = False
    with pytest.raises(ValueError):
        OC.apply_mask(z, a)
    with pytest.raises(ValueError):
        OC.apply_mask(z, np.ones((3, 16), dtype=bool))
