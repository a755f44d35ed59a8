"""fp64 oracle of tree verification: one target pass over a draft tree.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

Sources (page title, section):

* "Speculative Decoding: Speeding Sequential Generation" (aci),
  *Tree-Based Drafting: Testing More Than One Guess*: several candidates per
  position, one verification pass over the whole tree, the accept/reject test
  "applied per node"; *Constructing the Tree Attention Mask in Code*: a node
  attends to itself and its ancestors (plus the shared prefix), never to a
  sibling branch, and its rotary position id is its depth in the tree, not its
  offset in the flattened buffer; the printed 6-node mask and depth list;
  *Expected Tokens per Verification Round: Chain vs. Tree*: with per-node
  acceptance p and branching b, a level survives with q = 1 - (1 - p)^b and
  depth d is reached with q^d; E = sum_{d=1..D} q^d (2.138 for the binary
  tree of depth 3 at p = 0.6, 1.176 for the chain; 2.766 / 1.952 at p = 0.8),
  plus one bonus token per round; *Active Recall* 3: a chain is the tree with
  one child per node, whose mask is the lower-triangular causal mask.
* "Build a Speculative Decoding Engine to Cut LLM Latency by 3x",
  *Speculation Depth Tuning and Tree Drafting*: the mask from parent pointers,
  the root being the last accepted token; each candidate attends over its own
  ancestor chain.
* "Speculative Decoding: How to Make an LLM 3x Faster..." (kishorek): verify
  the whole tree in one pass and accept the longest valid root-to-node path.

Readings where the pages leave a step open:

* Node 0 is the root: the previous pass's emitted token t_last, not yet in
  the cache, at position L_b (depth 0).  Node i > 0 has a parent p(i) < i, so
  the flattened order lists every parent before its children.  A node's new
  key/value goes to slot L_b + i (flattened), rotated at position
  L_b + depth(i); logits row i scores the token after node i.
* Siblings are independent draws from their parent's draft distribution
  q_parent (one q row per node; a leaf's row is unused).  At a node the
  children are tried in index order: child c is accepted iff
  u[c] < min(1, p'(x_c) / q(x_c)), where p' is the node's target
  distribution (after T / top-p) and, after each rejected child, is replaced
  by the residual norm(max(0, p' - q)) (kept as it is when that mass is at or
  below 1e-8, the chain rule's numerical fallback).  This is the per-node
  accept/reject test applied with the same q the siblings were drawn from; it
  emits each token with the target's probability (the chain rule is the case
  of one child per node).  The first accepted child becomes the current node;
  when no child is accepted (or the node is a leaf) one token is drawn from
  p' with u[0] by the inverse CDF in id order, and the round ends.
* Greedy (T = 0): at each node take the first child whose token is the
  target's argmax (lowest id on ties); else emit that argmax and stop.
* After the round the accepted path's keys/values are moved to the
  contiguous slots L_b + 1 .. L_b + m (m accepted nodes) and the length
  becomes L_b + 1 + m; the other slots are left as they are.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

from . import model as om
from . import weights as wts
from .accept import (CDF_MARGIN, RATIO_MARGIN, RESIDUAL_FALLBACK, TOPP_MARGIN, argmax_lowest,
                     inverse_cdf, target_dist)
from .bf16 import round_bf16


def tree_structure(parents):
    """(depth [n], visible [n][n]) of a tree given by parent indices.

    parents[0] = -1 (the root); parents[i] < i for i > 0.  visible[i][j] = 1
    iff j == i or j is an ancestor of i (the root included)."""
    par = [int(p) for p in parents]
    n = len(par)
    if n == 0 or par[0] != -1:
        raise ValueError("node 0 must be the root (parent -1)")
    for i in range(1, n):
        if not 0 <= par[i] < i:
            raise ValueError("parent must precede its child")
    depth = np.zeros(n, dtype=np.int64)
    vis = np.zeros((n, n), dtype=np.int64)
    for i in range(n):
        j = i
        while j != -1:
            vis[i, j] = 1
            j = par[j]
        depth[i] = vis[i].sum() - 1
    return depth, vis


def chain_parents(n: int) -> list:
    """The chain of n nodes as a tree: node i's parent is i - 1."""
    return [-1] + list(range(n - 1))


def full_tree_parents(b: int, D: int) -> list:
    """Root plus a full b-ary tree of depth D, nodes in level order."""
    par = [-1]
    level = [0]
    for _ in range(D):
        nxt = []
        for p in level:
            for _ in range(b):
                par.append(p)
                nxt.append(len(par) - 1)
        level = nxt
    return par


def expected_depth(p: float, b: int, D: int) -> float:
    """Expected accepted depth of a full b-ary tree of depth D when every
    candidate is accepted independently with probability p: sum_d q^d with
    q = 1 - (1 - p)^b (per-level survival)."""
    q = 1.0 - (1.0 - p) ** b
    return float(sum(q ** d for d in range(1, D + 1)))


def attention_tree(q, K, V, L0: int, vis) -> np.ndarray:
    """GQA attention of the n tree nodes of one sequence.

    q [n][H][hd] (rotated), K/V [Hkv][T][hd] with the new entries at slots
    L0 .. L0+n-1; node i reads the cached keys 0..L0-1 and the new slots
    L0 + j with vis[i][j] = 1."""
    n, H, hd = q.shape
    G = H // K.shape[0]
    o = np.zeros((n, H, hd))
    scale = 1.0 / np.sqrt(hd)
    for i in range(n):
        idx = np.concatenate([np.arange(L0), L0 + np.flatnonzero(vis[i])])
        for h in range(H):
            kh = h // G
            s = K[kh, idx] @ q[i, h] * scale
            a = np.exp(s - s.max())
            a /= a.sum()
            o[i, h] = a @ V[kh, idx]
    return o


def forward_tree(cfg: om.Config, W: "wts.Weights", tokens, parents, kv: om.KVState,
                 round_kv: bool = True) -> np.ndarray:
    """One verification pass over a draft tree per sequence.

    tokens [B][n] (node 0 = t_last), parents [B][n] (or one list shared by
    every sequence) -> logits [B][n][V] (fp64).  Node i's key/value goes to
    slot len_b + i at rotary position len_b + depth(i); len_b advances by n
    (``commit`` moves the accepted path afterwards)."""
    toks = np.asarray(tokens, dtype=np.int64)
    B, n = toks.shape
    par = np.asarray(parents, dtype=np.int64)
    if par.ndim == 1:
        par = np.broadcast_to(par, (B, n))
    struct = [tree_structure(par[b]) for b in range(B)]
    d, H, Hkv, hd = cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.head_dim
    L0 = kv.lens.copy()
    if np.any(L0 + n > kv.capacity):
        raise ValueError("cache capacity exceeded")
    if np.any(toks < 0) or np.any(toks >= cfg.vocab):
        raise ValueError("token id out of range")
    h = W.embed_rows(toks.reshape(-1)).astype(np.float64).reshape(B, n, d)
    g = W.norm_gain()
    store = round_bf16 if round_kv else (lambda a: a)
    for l in range(cfg.n_layers):
        w = W.layer(l)
        x = om.rmsnorm(h, g, cfg.rms_eps)
        q = (x @ w[wts.WQ].astype(np.float64).T).reshape(B, n, H, hd)
        k = (x @ w[wts.WK].astype(np.float64).T).reshape(B, n, Hkv, hd)
        v = (x @ w[wts.WV].astype(np.float64).T).reshape(B, n, Hkv, hd)
        o = np.zeros((B, n, H, hd))
        for b in range(B):
            depth, vis = struct[b]
            pos = L0[b] + depth
            qb = om.rope(q[b].transpose(1, 0, 2), pos, cfg.rope_theta).transpose(1, 0, 2)
            kb = om.rope(k[b].transpose(1, 0, 2), pos, cfg.rope_theta)
            kv.K[l][b, :, L0[b]:L0[b] + n] = store(kb)
            kv.V[l][b, :, L0[b]:L0[b] + n] = store(v[b].transpose(1, 0, 2))
            o[b] = attention_tree(qb, kv.K[l][b], kv.V[l][b], int(L0[b]), vis)
        h = h + o.reshape(B, n, H * hd) @ w[wts.WO].astype(np.float64).T
        x = om.rmsnorm(h, g, cfg.rms_eps)
        h = h + om.swiglu(x, w[wts.WG], w[wts.WU], w[wts.WD])
    x = om.rmsnorm(h, g, cfg.rms_eps)
    kv.lens += n
    return x @ W.head().astype(np.float64).T


@dataclass
class TreeResult:
    path: list                         # accepted nodes, root excluded, in depth order
    tokens: list                       # their tokens, then the emitted token
    n_accepted: int
    emitted: int
    ratio_boundary: bool = False
    cdf_boundary: bool = False
    topp_boundary: bool = False
    fallback_boundary: bool = False

    @property
    def boundary(self) -> bool:
        return (self.ratio_boundary or self.cdf_boundary or self.topp_boundary
                or self.fallback_boundary)


def tree_accept(z_target, q_draft, node_tokens, parents, uniforms, temperature: float,
                top_p: float = 1.0, margins: tuple | None = None) -> TreeResult:
    """The acceptance walk of one sequence's tree (readings in the header).

    z_target [n][V] target logits per node; q_draft [n][V] the distribution
    each node's children were drawn from (after the same T / top-p; unused
    for T = 0 and for leaves); node_tokens [n]; parents [n]; uniforms [n]:
    u[c] (c >= 1) is the coin of child c, u[0] drives the final draw."""
    z = np.asarray(z_target, dtype=np.float64)
    n, V = z.shape
    par = [int(p) for p in parents]
    tree_structure(par)
    toks = [int(t) for t in node_tokens]
    children = [[c for c in range(1, n) if par[c] == i] for i in range(n)]
    res = TreeResult([], [], 0, -1)
    cur = 0
    if temperature == 0:
        while True:
            a = argmax_lowest(z[cur])
            nxt = next((c for c in children[cur] if toks[c] == a), None)
            if nxt is None:
                res.tokens.append(a)
                res.emitted = a
                return res
            res.path.append(nxt)
            res.tokens.append(a)
            res.n_accepted += 1
            cur = nxt
    rm, cm, tm = margins if margins is not None else (RATIO_MARGIN, CDF_MARGIN, TOPP_MARGIN)
    q = np.asarray(q_draft, dtype=np.float64)
    u = np.asarray(uniforms, dtype=np.float64)
    while True:
        P, info = target_dist(z[cur], temperature, top_p, tm)
        res.topp_boundary |= info.boundary
        nxt = None
        for c in children[cur]:
            x = toks[c]
            if not 0 <= x < V:
                raise ValueError("draft token out of range")
            if not q[cur, x] > 0:
                raise ValueError("q(x) = 0 for a drafted token")
            a = min(1.0, P[x] / q[cur, x])
            if abs(u[c] - a) < rm:
                res.ratio_boundary = True
            if u[c] < a:
                nxt = c
                break
            r = np.maximum(P - q[cur], 0.0)
            S = r.sum()
            if RESIDUAL_FALLBACK * 0.1 < S < RESIDUAL_FALLBACK * 10:
                res.fallback_boundary = True
            if S > RESIDUAL_FALLBACK:
                P = r / S
        if nxt is None:
            d = inverse_cdf(P, u[0], cm)
            res.cdf_boundary = d.boundary
            res.tokens.append(d.token)
            res.emitted = d.token
            return res
        res.path.append(nxt)
        res.tokens.append(toks[nxt])
        res.n_accepted += 1
        cur = nxt


def commit(kv: om.KVState, b: int, L0: int, path) -> None:
    """After a tree round of sequence b (pass started at length L0): move the
    accepted path's entries (flattened slots L0 + node) to the contiguous
    slots L0 + 1 .. L0 + m, in depth order, and set the length L0 + 1 + m."""
    for d, node in enumerate(path, start=1):
        for l in range(len(kv.K)):
            kv.K[l][b, :, L0 + d] = kv.K[l][b, :, L0 + node]
            kv.V[l][b, :, L0 + d] = kv.V[l][b, :, L0 + node]
    kv.lens[b] = L0 + 1 + len(path)
