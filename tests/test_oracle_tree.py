"""Pins of the tree-verification oracle (CPU only).

The pages print the tree mask and depth list of a 6-node example and the
expected accepted depths of a binary tree and a chain; those are checked
here (tests/golden/tree_mask.json), the expected-depth formula is checked
against a simulation of independent per-candidate coins, a chain written as
a tree must reproduce the chain forward and the chain accept rule exactly,
every root-to-leaf path of a tree must reproduce a chain pass over that path
(what the ancestor mask and depth positions are for), and the acceptance
walk must emit the target distribution (chi-square).
"""
import json
import os

import numpy as np
import pytest
from scipy import stats

from oracle import accept as OA
from oracle import model as Mo
from oracle import tree as Tr
from oracle import weights as W

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "tree_mask.json")
TINY = Mo.Config(n_layers=2, d_model=64, n_heads=4, n_kv_heads=2, d_ffn=96, vocab=50)


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_mask_and_depths_match_printed_example():
    g = _golden()
    names = g["nodes"]
    # the pages' nodes under a root (node 0 = the last accepted token)
    parents = [-1] + [0 if p is None else names.index(p) + 1 for p in g["parents"]]
    depth, vis = Tr.tree_structure(parents)
    np.testing.assert_array_equal(vis[1:, 1:], np.array(g["mask"]))
    assert (vis[1:, 0] == 1).all()            # the prefix column the page prepends
    assert depth[1:].tolist() == g["depths"]
    assert depth[0] == 0


def test_chain_mask_is_lower_triangular():
    for n in (1, 2, 5, 9):
        depth, vis = Tr.tree_structure(Tr.chain_parents(n))
        np.testing.assert_array_equal(vis, np.tril(np.ones((n, n), dtype=np.int64)))
        assert depth.tolist() == list(range(n))


def test_bad_parents_rejected():
    for bad in ([0, 0], [-1, 1], [-1, 0, 3, 1], []):
        with pytest.raises(ValueError):
            Tr.tree_structure(bad)


def test_expected_depth_printed_values():
    g = _golden()
    for e in g["expected"]:
        assert round(Tr.expected_depth(e["p"], e["b"], e["D"]), 3) == e["E"]
    for key, p in (("p0.6", 0.6), ("p0.8", 0.8)):
        tree = Tr.expected_depth(p, 2, 3) + 1
        chain = Tr.expected_depth(p, 1, 3) + 1
        assert [round(tree, 3), round(chain, 3)] == g["totals_with_bonus"][key]
        assert round(tree / chain, 2) == round(g["ratio_tree_over_chain"][key], 2)


def test_expected_depth_against_simulated_coins():
    """Independent coins per candidate, walk down while some child's coin
    succeeds: the mean depth matches sum_d q^d within 4 standard errors."""
    rng = np.random.default_rng(5)
    for p, b in ((0.6, 2), (0.6, 1), (0.8, 2), (0.35, 3)):
        D, N = 3, 200000
        ok = rng.random((N, D, b)) < p
        level_ok = ok.any(axis=2)
        depth = np.cumprod(level_ok, axis=1).sum(axis=1)
        se = depth.std() / np.sqrt(N)
        assert abs(depth.mean() - Tr.expected_depth(p, b, D)) < 4 * se


def _cache(cfg, Wt, B, L, cap, seed):
    kv = Mo.KVState(cfg, B, cap)
    prefix = np.random.default_rng(seed).integers(0, cfg.vocab, size=(B, L))
    Mo.forward(cfg, Wt, prefix, kv)
    return kv


def _copy(kv):
    c = Mo.KVState.__new__(Mo.KVState)
    c.K = [k.copy() for k in kv.K]
    c.V = [v.copy() for v in kv.V]
    c.lens = kv.lens.copy()
    c.capacity = kv.capacity
    return c


def test_chain_tree_forward_equals_forward():
    Wt = W.Weights(TINY, 81)
    kv = _cache(TINY, Wt, 2, 7, 40, 1)
    kv2 = _copy(kv)
    toks = np.random.default_rng(3).integers(0, TINY.vocab, size=(2, 5))
    a = Mo.forward(TINY, Wt, toks, kv)
    b = Tr.forward_tree(TINY, Wt, toks, Tr.chain_parents(5), kv2)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-12)
    for l in range(TINY.n_layers):
        np.testing.assert_array_equal(kv.K[l], kv2.K[l])


@pytest.mark.parametrize("parents", [
    Tr.full_tree_parents(2, 2),                 # the pages' 6-node tree under a root
    Tr.full_tree_parents(2, 3),                 # 14 nodes + root
    [-1, 0, 0, 0, 1, 1, 3, 6, 2],               # ragged branching
])
def test_every_path_equals_a_chain_pass(parents):
    """Each node's logits equal those of a chain pass over its root-to-node
    path on the same cache: ancestors only, rotary position = depth."""
    Wt = W.Weights(TINY, 82)
    kv = _cache(TINY, Wt, 1, 6, 64, 2)
    n = len(parents)
    toks = np.random.default_rng(4).integers(0, TINY.vocab, size=(1, n))
    zt = Tr.forward_tree(TINY, Wt, toks, parents, _copy(kv))
    for i in range(n):
        path = []
        j = i
        while j != -1:
            path.append(j)
            j = parents[j]
        path = path[::-1]
        zc = Mo.forward(TINY, Wt, toks[:, path], _copy(kv))
        np.testing.assert_allclose(zt[0, i], zc[0, -1], rtol=1e-10, atol=1e-10)


def test_chain_tree_accept_equals_chain_rule():
    """A chain as a tree: tree child c uses u[c], the final draw u[0]; the
    chain rule uses u[c-1] and u[gamma]."""
    rng = np.random.default_rng(11)
    V, gamma = 40, 4
    for trial in range(300):
        zq = rng.normal(0, 2, size=(gamma, V))
        zp = rng.normal(0, 2, size=(gamma + 1, V))
        zp[:gamma] = zq + rng.normal(0, 0.5, size=(gamma, V))
        q, x, _ = OA.draft_sample(zq, rng.random(gamma), 1.0)
        uc = rng.random(gamma + 1)
        r = OA.accept(zp, q, x, uc, 1.0)
        qt = np.vstack([q, np.zeros((1, V))])
        ut = np.concatenate([[uc[gamma]], uc[:gamma]])
        t = Tr.tree_accept(zp, qt, [0] + list(x), Tr.chain_parents(gamma + 1), ut, 1.0)
        assert t.n_accepted == r.n_accepted
        assert t.tokens == r.tokens[:r.n_accepted + 1]
        assert t.path == list(range(1, r.n_accepted + 1))
    # greedy
    zp = rng.normal(size=(gamma + 1, V))
    x = zp[:gamma].argmax(1)
    x[2] = (x[2] + 1) % V
    r = OA.accept(zp, None, x, None, 0.0)
    t = Tr.tree_accept(zp, None, [0] + list(x), Tr.chain_parents(gamma + 1), None, 0.0)
    assert t.n_accepted == r.n_accepted == 2 and t.tokens == r.tokens[:3]


def test_tree_accept_emits_the_target_distribution():
    """Root with 3 children, each child with 2 children, children drawn i.i.d.
    from their parent's q: over 30000 trials the first emitted token follows
    p_root (chi-square p-value > 1e-3)."""
    rng = np.random.default_rng(21)
    V, N = 6, 30000
    parents = [-1, 0, 0, 0, 1, 1, 2, 2, 3, 3]
    n = len(parents)
    P = rng.dirichlet(np.ones(V), size=n)
    Q = np.clip(P + rng.normal(0, 0.12, size=(n, V)), 0.02, None)
    Q /= Q.sum(1, keepdims=True)
    z = np.log(P)
    first = np.zeros(V)
    for _ in range(N):
        toks = [0] * n
        for c in range(1, n):
            toks[c] = int(rng.choice(V, p=Q[parents[c]]))
        res = Tr.tree_accept(z, Q, toks, parents, rng.random(n), 1.0)
        first[res.tokens[0]] += 1
    Pf = np.exp(z) / np.exp(z).sum(1, keepdims=True)
    assert stats.chisquare(first, Pf[0] * N).pvalue > 1e-3


def test_tree_accept_second_token_conditional():
    """Given the walk moved to child c, the next emitted token follows c's
    own target distribution (chi-square per child reached > 500 times)."""
    rng = np.random.default_rng(22)
    V, N = 5, 20000
    parents = [-1, 0, 0, 1, 1, 2, 2]
    n = len(parents)
    P = rng.dirichlet(np.ones(V), size=n)
    Q = np.clip(P + rng.normal(0, 0.15, size=(n, V)), 0.02, None)
    Q /= Q.sum(1, keepdims=True)
    z = np.log(P)
    Pf = np.exp(z) / np.exp(z).sum(1, keepdims=True)
    counts = {}
    for _ in range(N):
        toks = [0] * n
        for c in range(1, n):
            toks[c] = int(rng.choice(V, p=Q[parents[c]]))
        res = Tr.tree_accept(z, Q, toks, parents, rng.random(n), 1.0)
        if res.n_accepted >= 1:
            node = res.path[0]
            counts.setdefault(node, np.zeros(V))[res.tokens[1]] += 1
    for node, cnt in counts.items():
        if cnt.sum() > 500:
            assert stats.chisquare(cnt, Pf[node] * cnt.sum()).pvalue > 1e-3, node


def test_commit_moves_the_accepted_path():
    cfg = TINY
    kv = Mo.KVState(cfg, 2, 32)
    rng = np.random.default_rng(9)
    for l in range(cfg.n_layers):
        kv.K[l][:] = rng.normal(size=kv.K[l].shape)
        kv.V[l][:] = rng.normal(size=kv.V[l].shape)
    kv.lens[:] = [10 + 7, 4 + 7]
    before = [k.copy() for k in kv.K]
    Tr.commit(kv, 0, 10, [2, 5, 6])
    assert kv.lens[0] == 14 and kv.lens[1] == 11
    for l in range(cfg.n_layers):
        for d, node in enumerate([2, 5, 6], start=1):
            np.testing.assert_array_equal(kv.K[l][0, :, 10 + d], before[l][0, :, 10 + node])
        np.testing.assert_array_equal(kv.K[l][1], before[l][1])
