"""The pins against the mistakes the pages name (the engine guide's guardrail
list: resampling from p instead of the residual, a temperature mismatch
between the draft's sampling and the q given to the rule, a KV cache off by
one slot after rollback, seeds that do not propagate).

CPU only.  Each mistake is planted in the oracle (or in the inputs it is
given), and the test checks that the pin which guards against it — the
chi-square of the emitted tokens against p, the rollback-then-reverify
invariant, determinism in the uniforms — fails with the mistake and holds
without it.  The pins are thereby shown to have the power to catch them.
"""
import numpy as np
import pytest
from scipy import stats

from oracle import accept as A
from oracle import model as Mo
from oracle import weights as W

TINY = Mo.Config(n_layers=2, d_model=64, n_heads=4, n_kv_heads=2, d_ffn=96, vocab=50)


def _first_tokens(P, Q_sampled, Q_given, trials, seed, T=1.0):
    """First emitted token of one-draft passes: the draft x ~ Q_sampled (the
    oracle's own inverse CDF), the rule told that q = Q_given."""
    g = np.random.default_rng(seed)
    z = np.log(np.stack([P, P]))              # the scored row and the bonus row
    out = np.empty(trials, dtype=np.int64)
    for t in range(trials):
        x = A.inverse_cdf(Q_sampled, g.random()).token
        out[t] = A.accept(z, Q_given[None, :], [x], g.random(2), T).tokens[0]
    return out


def _pvalue(tokens, P):
    obs = np.bincount(tokens, minlength=P.size)
    return stats.chisquare(obs, P * tokens.size).pvalue


def _pq(seed, V=8):
    g = np.random.default_rng(seed)
    P = g.dirichlet(np.ones(V))
    Q = g.dirichlet(np.ones(V))
    return P, Q


def test_resampling_from_p_instead_of_the_residual_is_caught(monkeypatch):
    """Lattice notes: drawing the correction from p instead of
    norm(max(0, p - q)) silently biases the output.  Planted by raising the
    oracle's residual-fallback threshold above any residual mass, so every
    rejection draws from p: the first emitted token then follows
    min(p, q) + (1 - alpha) p, and the chi-square against p fails."""
    P, Q = _pq(21)
    trials = 40_000
    good = _first_tokens(P, Q, Q, trials, seed=1)
    assert _pvalue(good, P) > 1e-3
    monkeypatch.setattr(A, "RESIDUAL_FALLBACK", np.inf)
    bad = _first_tokens(P, Q, Q, trials, seed=1)
    assert _pvalue(bad, P) < 1e-9
    # the planted law, exactly
    alpha = np.minimum(P, Q).sum()
    law = np.minimum(P, Q) + (1 - alpha) * P
    assert _pvalue(bad, law) > 1e-3


def test_temperature_mismatch_is_caught():
    """Pigeon guide, *When it breaks*: the q given to the rule must be the
    distribution the draft sampled from, after the same temperature.  Drafts
    sampled at T = 1 but scored with q at T = 0.6 break the output law."""
    g = np.random.default_rng(33)
    zq = g.normal(0, 1.5, size=8)
    P = A.softmax_t(zq + g.normal(0, 0.7, size=8), 1.0)
    q_true = A.softmax_t(zq, 1.0)
    q_claimed = A.softmax_t(zq, 0.6)
    trials = 40_000
    assert _pvalue(_first_tokens(P, q_true, q_true, trials, seed=2), P) > 1e-3
    assert _pvalue(_first_tokens(P, q_true, q_claimed, trials, seed=2), P) < 1e-9


def _prefilled(Wt, L, seed):
    kv = Mo.KVState(TINY, 1, 32)
    toks = np.random.default_rng(seed).integers(0, TINY.vocab, size=(1, L))
    Mo.forward(TINY, Wt, toks, kv)
    return kv


@pytest.mark.parametrize("slip", [-1, 1])
def test_kv_length_off_by_one_after_rollback_is_caught(slip):
    """Engine guide, *Rollback Protocol*: after n accepted of gamma drafts the
    cache keeps t_last and the n drafts.  A length one slot short (drops the
    last accepted draft) or one long (keeps the first rejected draft) makes
    the next pass differ from a cache that only ever saw the accepted tokens
    — the rollback-then-reverify invariant fails."""
    Wt = W.Weights(TINY, 79)
    block = np.array([[7, 11, 13, 17, 19]])
    nxt = np.array([[23, 29, 31]])
    fresh = _prefilled(Wt, 6, 4)
    Mo.forward(TINY, Wt, block[:, :3], fresh)                   # t_last, x1, x2 accepted
    ref = Mo.forward(TINY, Wt, nxt, fresh)
    for s, expect_equal in ((0, True), (slip, False)):
        kv = _prefilled(Wt, 6, 4)
        Mo.forward(TINY, Wt, block, kv)
        kv.lens = Mo.truncate(kv.lens, [2], gamma=4) + s          # planted slip
        got = Mo.forward(TINY, Wt, nxt, kv)
        assert np.allclose(got, ref, rtol=1e-12, atol=1e-12) == expect_equal, (s, slip)


def test_outcome_is_a_function_of_the_uniforms():
    """Engine guide, *Quality, Evaluation, and Guardrails*: with the seeds
    propagated, a step is reproducible.  The rule is a pure function of its
    inputs: the same uniforms give the same tokens, other uniforms (another
    seed) give other tokens somewhere in a long run."""
    V, gamma = 16, 4
    g = np.random.default_rng(8)
    z = g.normal(0, 2, size=(gamma + 1, V))
    Q = A.softmax_t(z[:gamma] + g.normal(0, 1, size=(gamma, V)), 1.0)

    def run(seed):
        r = np.random.default_rng(seed)
        outs = []
        for _ in range(200):
            xs = [A.inverse_cdf(Q[i], r.random()).token for i in range(gamma)]
            outs.append(tuple(A.accept(z, Q, xs, r.random(gamma + 1), 1.0).tokens))
        return outs

    assert run(5) == run(5)
    assert run(5) != run(6)


def _tree_first_tokens(trials, seed):
    from oracle import tree as Tr
    rng = np.random.default_rng(seed)
    V = 6
    parents = [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3]
    n = len(parents)
    P = rng.dirichlet(np.ones(V), size=n)
    Q = np.clip(P + rng.normal(0, 0.12, size=(n, V)), 0.02, None)
    Q /= Q.sum(1, keepdims=True)
    z = np.log(P)
    first = np.zeros(V)
    for _ in range(trials):
        toks = [0] * n
        for c in range(1, n):
            toks[c] = int(rng.choice(V, p=Q[parents[c]]))
        first[Tr.tree_accept(z, Q, toks, parents, rng.random(n), 1.0).tokens[0]] += 1
    return first, P[0]


def test_tree_siblings_without_the_carried_residual_is_caught(monkeypatch):
    """Aci, *Tree-Based Drafting* (the per-node test): after a rejected child
    the next sibling is tested against norm(max(0, p' - q)), not against p.
    Planted by raising the tree oracle's residual-fallback threshold above any
    mass, so p' never changes: the root's first emitted token no longer
    follows p and the chi-square pin fails."""
    from oracle import tree as Tr
    trials = 20_000
    first, p0 = _tree_first_tokens(trials, seed=21)
    assert stats.chisquare(first, p0 * trials).pvalue > 1e-3
    monkeypatch.setattr(Tr, "RESIDUAL_FALLBACK", np.inf)
    first, p0 = _tree_first_tokens(trials, seed=21)
    assert stats.chisquare(first, p0 * trials).pvalue < 1e-9
