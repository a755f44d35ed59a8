"""GPU parity of draft-tree verification against the fp64 oracle.

Forward: the device model and the oracle share a seed; after a chain prefill
both run one pass over a draft tree per sequence (spec_tree_masks +
spec_verify_forward_tree vs oracle.tree.forward_tree) and the logits must
agree within |d| <= 1e-2 * (1 + |logit|), under the persistent and the
per-step schedules and with trees wide enough for the split-KV attention.
A chain written as a tree must give the chain call's logits.  Commit: after
spec_kv_tree_commit of an accepted path the next chain pass must agree with
the oracle's (oracle.tree.commit); the moved cache rows must equal the
sources bit for bit.  Accept: spec_tree_accept vs oracle.tree.tree_accept on
the same fp32 inputs: path, tokens and count equal exactly except where the
oracle flags a decision inside its fp32/fp64 margin.
"""
import numpy as np
import pytest
import torch

import parity
from oracle import accept as OA
from oracle import model as OM
from oracle import tree as Tr
from oracle import weights as OW
from speculative_decoding_verification_pass_gb300 import binding as sb
from speculative_decoding_verification_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

TOL = 1e-2

CFGS = [
    sb.ModelConfig(2, 256, 4, 2, 256, 1000),        # hd 64, 2 query heads per KV head
    sb.ModelConfig(2, 512, 4, 1, 384, 4099),        # hd 128, 4 query heads per KV head
]

RAGGED = [-1, 0, 0, 0, 1, 1, 3, 6, 2]


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _close(got, ref, tol=TOL):
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert err.max() <= tol, f"max rel err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    return err.max()


def _masks(parents_b):
    """Device (anc, depth) tensors [B][n] from per-sequence parent lists."""
    anc, dep = [], []
    for par in parents_b:
        a, d = sb.spec_tree_masks(par)
        anc.append(a)
        dep.append(d)
    anc = np.array(anc, dtype=np.uint64).view(np.int64)
    return _dev(anc), _dev(np.array(dep, dtype=np.int32))


def _ancestor_path(par, node):
    p = []
    while node > 0:
        p.append(node)
        node = par[node]
    return p[::-1]


class Pair:
    """A device model + cache and the oracle's model + cache, same seed."""

    def __init__(self, cfg, seed, B, cap):
        self.cfg, self.B, self.cap = cfg, B, cap
        self.model = sb.Model(cfg, seed)
        self.kv = sb.KVCache(cfg, B, cap)
        self.ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, 127, cap))
        self.ocfg = OM.Config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.d_ffn,
                              cfg.vocab, cfg.rms_eps, cfg.rope_theta)
        self.W = OW.Weights(self.ocfg, seed)
        self.okv = OM.KVState(self.ocfg, B, cap)

    def chain(self, toks):
        B, n = toks.shape
        out = torch.empty(B, n, self.cfg.vocab, device="cuda")
        sb.spec_verify_forward(self.model.handle, _dev(toks.astype(np.int32)), B, n - 1, self.kv,
                               out, self.ws)
        g = out.double().cpu().numpy()
        o = OM.forward(self.ocfg, self.W, toks, self.okv)
        _close(g, o)
        return g

    def tree(self, toks, parents_b):
        B, n = toks.shape
        anc, dep = _masks(parents_b)
        out = torch.empty(B, n, self.cfg.vocab, device="cuda")
        sb.spec_verify_forward_tree(self.model.handle, _dev(toks.astype(np.int32)), anc, dep, B, n,
                                    self.kv, out, self.ws)
        g = out.double().cpu().numpy()
        o = Tr.forward_tree(self.ocfg, self.W, toks, np.array(parents_b), self.okv)
        _close(g, o)
        return g

    def status_ok(self):
        st, bits = sb.spec_device_status(self.ws)
        assert st == sb.SPEC_OK, hex(bits)


def _trees(name, n_seq, seed):
    if name == "binary_d2":
        base = Tr.full_tree_parents(2, 2)        # the pages' 6-node tree under a root
    elif name == "ragged":
        base = RAGGED
    elif name == "binary_d4":
        base = Tr.full_tree_parents(2, 4)        # 31 nodes: split-KV attention
    elif name == "random64":
        base = wl.random_tree(seed, 64)          # the largest tree
    else:
        raise KeyError(name)
    # sequence 0 takes the named tree, the others random trees of the same size
    return [base] + [wl.random_tree(seed + 1 + b, len(base)) for b in range(n_seq - 1)]


@pytest.mark.parametrize("schedule", ["persistent", "per_step"])
@pytest.mark.parametrize("ci", range(len(CFGS)))
@pytest.mark.parametrize("tree", ["binary_d2", "ragged", "binary_d4", "random64"])
def test_tree_forward_and_commit(schedule, ci, tree, monkeypatch):
    if schedule == "per_step":
        monkeypatch.setenv("SPEC_FORWARD_PERSISTENT", "0")
    cfg = CFGS[ci]
    B, cap = 3, 192
    seed = 300 + 10 * ci + len(tree)
    P = Pair(cfg, seed, B, cap)
    # ragged prefixes: two chain passes, then a rollback keeping 31 / 10 / 20
    # of the second pass's 31 drafts (lengths 37, 16, 26)
    pre = wl.tokens(seed, B, 37, cfg.vocab)
    P.chain(pre[:, :5])
    P.chain(pre[:, 5:])
    keep = np.array([31, 10, 20], np.int32)
    sb.spec_kv_truncate(P.kv, _dev(keep), 31, P.ws)
    P.okv.lens -= 31 - keep
    parents_b = _trees(tree, B, seed)
    n = len(parents_b[0])
    toks = wl.tokens(seed, B, n, cfg.vocab, stream=11)
    L0 = P.kv.len.cpu().numpy().copy()
    P.tree(toks, parents_b)
    np.testing.assert_array_equal(P.kv.len.cpu().numpy(), L0 + n)
    # commit a root-to-node path per sequence (the last node's ancestors, cut
    # to a sequence-dependent depth; sequence 1 accepts nothing)
    paths = []
    for b in range(B):
        full = _ancestor_path(parents_b[b], n - 1)
        m = 0 if b == 1 else max(1, len(full) - b)
        paths.append(full[:m])
    path_t = np.full((B, n), -1, np.int32)
    nacc = np.zeros(B, np.int32)
    for b, p in enumerate(paths):
        path_t[b, :len(p)] = p
        nacc[b] = len(p)
    k_before = P.kv.k.clone()
    sb.spec_kv_tree_commit(P.model.handle, P.kv, _dev(path_t), _dev(nacc), n, P.ws)
    for b, p in enumerate(paths):
        Tr.commit(P.okv, b, int(L0[b]), p)
    np.testing.assert_array_equal(P.kv.len.cpu().numpy(), P.okv.lens)
    for b, p in enumerate(paths):
        for d, node in enumerate(p, start=1):
            assert torch.equal(P.kv.k[:, b, :, L0[b] + d], k_before[:, b, :, L0[b] + node])
    # the next chain pass reads the committed cache
    P.chain(wl.tokens(seed, B, 4, cfg.vocab, stream=12))
    P.status_ok()


def test_chain_written_as_tree_equals_chain():
    cfg = CFGS[1]
    B, cap, n = 2, 96, 6
    m = sb.Model(cfg, 5)
    kvs = [sb.KVCache(cfg, B, cap) for _ in range(2)]
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, 127, cap))
    pre = _dev(wl.tokens(5, B, 30, cfg.vocab).astype(np.int32))
    tmp = torch.empty(B, 30, cfg.vocab, device="cuda")
    for kv in kvs:
        sb.spec_verify_forward(m.handle, pre, B, 29, kv, tmp, ws)
    toks = _dev(wl.tokens(5, B, n, cfg.vocab, stream=11).astype(np.int32))
    a = torch.empty(B, n, cfg.vocab, device="cuda")
    b = torch.empty_like(a)
    sb.spec_verify_forward(m.handle, toks, B, n - 1, kvs[0], a, ws)
    anc, dep = _masks([Tr.chain_parents(n)] * B)
    sb.spec_verify_forward_tree(m.handle, toks, anc, dep, B, n, kvs[1], b, ws)
    err = ((a - b).abs() / (1 + a.abs())).max().item()
    assert err <= 1e-5, err
    assert torch.equal(kvs[0].len, kvs[1].len)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)


# ------------------------------------------------------------------ accept
def _tree_inputs(seed, B, parents, V, T, top_p):
    """Target logits, per-node draft distributions q (fp32) and node tokens:
    every child is drawn from its parent's q with its own uniform."""
    n = len(parents)
    zq, zp = wl.accept_logits(seed, B, n - 1, V)
    ud = wl.uniforms(seed, B, n, stream=8)
    Tq = T if T > 0 else 1.0
    q = np.zeros((B, n, V), np.float32)
    toks = np.zeros((B, n), np.int32)
    par = np.array(parents)
    for b in range(B):
        qs, _, _ = OA.draft_sample(zq[b], ud[b], Tq, top_p)
        q[b] = qs.astype(np.float32)
        _, xs, _ = OA.draft_sample(zq[b][par[1:]], ud[b][1:], Tq, top_p)
        toks[b, 1:] = xs
    toks[:, 0] = wl.tokens(seed, B, 1, V, stream=13)[:, 0]
    if T == 0:
        # greedy: some children carry the target's argmax at their parent
        agree = wl.uniforms(seed, B, n, stream=9) < 0.6
        am = zp.argmax(-1)[:, par[1:]]
        toks[:, 1:] = np.where(agree[:, 1:], am, toks[:, 1:])
    u = wl.uniforms(seed, B, n)
    return zp, q, toks, u


def _run_tree_accept(zp, q, toks, parents, u, T, top_p):
    B, n, V = zp.shape
    out = torch.full((B, n), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, n), -7, dtype=torch.int32, device="cuda")
    nacc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ws = sb.workspace(sb.spec_tree_accept_workspace_bytes(B, V))
    par = np.broadcast_to(np.array(parents, np.int32), (B, n))
    sb.spec_tree_accept(_dev(zp), _dev(q), _dev(toks), _dev(par), _dev(u), B, n, V, T, top_p, out,
                        path, nacc, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    return out.cpu().numpy(), path.cpu().numpy(), nacc.cpu().numpy()


@pytest.mark.parametrize("B,V,T,top_p,tree", [
    (64, 4096, 1.0, 1.0, "binary_d2"),
    (64, 4096, 0.8, 0.9, "ragged"),
    (32, 1000, 1.0, 1.0, "random64"),
    (64, 4096, 0.0, 1.0, "binary_d2"),     # greedy
    (32, 4096, 0.0, 1.0, "random64"),      # greedy, wide nodes
    (8, 128256, 1.0, 1.0, "binary_d2"),    # llama3 vocabulary
    (16, 3, 1.0, 1.0, "ragged"),           # tiny vocabulary: residuals empty out
])
def test_tree_accept_matches_oracle(B, V, T, top_p, tree):
    seed = 900 + B + V + len(tree)
    parents = _trees(tree, 1, seed)[0]
    n = len(parents)
    zp, q, toks, u = _tree_inputs(seed, B, parents, V, T, top_p)
    out, path, nacc = _run_tree_accept(zp, q, toks, parents, u, T, top_p)
    excused = near = 0
    for b in range(B):
        r = Tr.tree_accept(zp[b], q[b] if T > 0 else None, toks[b], parents,
                           u[b] if T > 0 else None, T, top_p)
        m = r.n_accepted
        same = (int(nacc[b]) == m and out[b, :m + 1].tolist() == r.tokens
                and (out[b, m + 1:] == -1).all() and path[b, :m].tolist() == r.path
                and (path[b, m:] == -1).all())
        near += r.boundary
        if not same:
            assert r.boundary, (b, out[b].tolist(), r.tokens, path[b].tolist(), r.path)
            excused += 1
    parity.check(f"tree accept B={B} V={V} T={T} top_p={top_p} {tree}", B, near, excused)
    if T > 0:
        assert (nacc > 0).any()
    if T == 0:
        assert (nacc > 0).any()


def test_chain_tree_accept_equals_chain_accept():
    """The chain as a tree (u[c] for child c, u[0] for the final draw) gives
    spec_accept's tokens and counts on the same device inputs."""
    B, gamma, V = 128, 4, 4096
    n = gamma + 1
    zq, zp = wl.accept_logits(41, B, gamma, V)
    ud = wl.uniforms(41, B, gamma, stream=8)
    uc = wl.uniforms(41, B, n)
    q = np.zeros((B, gamma, V), np.float32)
    x = np.zeros((B, gamma), np.int32)
    for b in range(B):
        qs, ts, _ = OA.draft_sample(zq[b, :gamma], ud[b], 1.0, 1.0)
        q[b] = qs.astype(np.float32)
        x[b] = ts
    out = torch.empty((B, n), dtype=torch.int32, device="cuda")
    nacc = torch.empty((B,), dtype=torch.int32, device="cuda")
    ws = sb.workspace(sb.spec_accept_workspace_bytes(B, gamma, V))
    sb.spec_accept(_dev(zp), _dev(q), _dev(x), _dev(uc), B, gamma, V, 1.0, 1.0, out, nacc, ws)
    qt = np.concatenate([q, np.zeros((B, 1, V), np.float32)], axis=1)
    tt = np.concatenate([np.zeros((B, 1), np.int32), x], axis=1)
    ut = np.concatenate([uc[:, gamma:], uc[:, :gamma]], axis=1)
    to, tp, tn = _run_tree_accept(zp, qt, tt, Tr.chain_parents(n), ut, 1.0, 1.0)
    np.testing.assert_array_equal(tn, nacc.cpu().numpy())
    np.testing.assert_array_equal(to, out.cpu().numpy())
    for b in range(B):
        assert tp[b, :tn[b]].tolist() == list(range(1, tn[b] + 1))


def test_tree_accept_rejects_bad_parents():
    V, n = 64, 4
    zp = wl.accept_logits(3, 2, n - 1, V)[1]
    q = np.full((2, n, V), 1.0 / V, np.float32)
    toks = np.zeros((2, n), np.int32)
    par = np.array([[-1, 0, 0, 1], [-1, 0, 2, 1]], np.int32)   # sequence 1: parent after child
    out = torch.full((2, n), -7, dtype=torch.int32, device="cuda")
    path = torch.full((2, n), -7, dtype=torch.int32, device="cuda")
    nacc = torch.full((2,), -7, dtype=torch.int32, device="cuda")
    ws = sb.workspace(sb.spec_tree_accept_workspace_bytes(2, V))
    u = wl.uniforms(3, 2, n)
    sb.spec_tree_accept(_dev(zp), _dev(q), _dev(toks), _dev(par), _dev(u), 2, n, V, 1.0, 1.0, out,
                        path, nacc, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_EDEVICE and bits == sb.DEV_BAD_TREE
    assert int(nacc[1]) == 0 and (out[1] == -1).all() and (path[1] == -1).all()
    assert int(nacc[0]) >= 0 and int(out[0, int(nacc[0])]) >= 0


def test_tree_commit_moves_rows_and_checks_paths():
    cfg = CFGS[0]
    B, cap, n = 4, 40, 7
    kv = sb.KVCache(cfg, B, cap)
    g = torch.Generator(device="cuda").manual_seed(7)
    kv.k.copy_(torch.randn(kv.k.shape, generator=g, device="cuda").to(torch.bfloat16))
    kv.v.copy_(torch.randn(kv.v.shape, generator=g, device="cuda").to(torch.bfloat16))
    L0 = np.array([3, 10, 0, 20], np.int32)
    kv.len.copy_(_dev(L0 + n))
    paths = [[2, 5, 6], [1, 2, 3, 4, 5, 6], [], [3, 2]]        # sequence 3: not increasing
    path_t = np.full((B, n), -1, np.int32)
    nacc = np.array([len(p) for p in paths], np.int32)
    for b, p in enumerate(paths):
        path_t[b, :len(p)] = p
    k0, v0 = kv.k.clone(), kv.v.clone()
    m = sb.Model(cfg, 1)
    ws = sb.workspace(256)
    sb.spec_kv_tree_commit(m.handle, kv, _dev(path_t), _dev(nacc), n, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_EDEVICE and bits == sb.DEV_BAD_TREE
    np.testing.assert_array_equal(kv.len.cpu().numpy(), [3 + 1 + 3, 10 + 1 + 6, 0 + 1, 20 + n])
    for b in range(3):
        ek, ev = k0[:, b].clone(), v0[:, b].clone()
        for d, node in enumerate(paths[b], start=1):
            ek[:, :, L0[b] + d] = k0[:, b, :, L0[b] + node]
            ev[:, :, L0[b] + d] = v0[:, b, :, L0[b] + node]
        assert torch.equal(kv.k[:, b], ek) and torch.equal(kv.v[:, b], ev)
    assert torch.equal(kv.k[:, 3], k0[:, 3]) and torch.equal(kv.v[:, 3], v0[:, 3])
