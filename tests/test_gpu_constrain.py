"""GPU parity of constrained acceptance (one allowed-token mask per row,
applied alike to the target and the draft logits).

spec_mask_logits must set exactly the disallowed positions to -inf and leave
every other logit bit-identical; spec_accept / spec_draft_sample /
spec_tree_accept on masked logits must agree with the oracle on the same
masked inputs (oracle.constrain.apply_mask): emitted tokens and counts
exactly, except where the oracle flags a decision inside its fp32/fp64
margin, and never a disallowed token.
"""
import numpy as np
import pytest
import torch

import parity
from oracle import accept as OA
from oracle import constrain as OC
from oracle import tree as Tr
from speculative_decoding_verification_pass_gb300 import binding as sb
from speculative_decoding_verification_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _mask_on_device(z, allowed):
    """Masked copy of fp32 logits [..][V] through spec_mask_logits."""
    V = z.shape[-1]
    rows = int(np.prod(z.shape[:-1]))
    t = _dev(z.reshape(rows, V).astype(np.float32))
    ws = sb.workspace(256)
    sb.spec_mask_logits(t, _dev(wl.pack_allowed(allowed.reshape(rows, V))), rows, V, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    return t.cpu().numpy().reshape(z.shape)


def test_mask_logits_exact():
    rng = np.random.default_rng(1)
    rows, V = 37, 4099
    z = rng.normal(0, 3, size=(rows, V)).astype(np.float32)
    a = wl.allowed_sets(1, rows, V, 0.3)
    got = _mask_on_device(z, a)
    np.testing.assert_array_equal(np.isneginf(got), ~a)
    np.testing.assert_array_equal(got[a], z[a])


def test_mask_logits_empty_row_is_flagged_and_untouched():
    rows, V = 3, 100
    z = np.arange(rows * V, dtype=np.float32).reshape(rows, V)
    a = np.ones((rows, V), dtype=bool)
    a[1] = False
    a[2, ::2] = False
    t = _dev(z)
    ws = sb.workspace(256)
    sb.spec_mask_logits(t, _dev(wl.pack_allowed(a)), rows, V, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_EDEVICE and bits == sb.DEV_EMPTY_MASK
    out = t.cpu().numpy()
    np.testing.assert_array_equal(out[:2], z[:2])
    np.testing.assert_array_equal(np.isneginf(out[2]), ~a[2])


def _masked_draft(zq, a, ud, T, top_p):
    B, gamma, V = zq.shape
    q = np.zeros((B, gamma, V), np.float32)
    x = np.zeros((B, gamma), np.int32)
    for b in range(B):
        qs, ts, _ = OA.draft_sample(OC.apply_mask(zq[b], a[b]), ud[b], T, top_p)
        q[b] = qs.astype(np.float32)
        x[b] = ts
    return q, x


@pytest.mark.parametrize("grid", ["1", "0"])
@pytest.mark.parametrize("B,gamma,V,T,top_p,frac", [
    (200, 4, 4096, 1.0, 1.0, 0.3),
    (64, 4, 4096, 0.8, 0.9, 0.5),
    (64, 4, 4096, 0.0, 1.0, 0.3),       # greedy over the allowed tokens
    (8, 4, 128256, 1.0, 1.0, 0.01),     # llama3 vocabulary, a narrow (JSON-like) allowed set
])
def test_masked_accept_matches_oracle(B, gamma, V, T, top_p, frac, grid, monkeypatch):
    monkeypatch.setenv("SPEC_ACCEPT_GRID", grid)
    seed = 500 + B + V
    n = gamma + 1
    zq, zp = wl.accept_logits(seed, B, gamma, V)
    a = wl.allowed_sets(seed, B * n, V, frac).reshape(B, n, V)
    ud = wl.uniforms(seed, B, gamma, stream=8)
    u = wl.uniforms(seed, B, n)
    Tq = T if T > 0 else 1.0
    q, x = _masked_draft(zq[:, :gamma], a[:, :gamma], ud, Tq, top_p)
    if T == 0:
        zpm = np.where(a, zp, -np.inf)
        agree = wl.uniforms(seed, B, gamma, stream=9) < 0.7
        x = np.where(agree, zpm[:, :gamma].argmax(-1), x).astype(np.int32)
    zp_dev = _mask_on_device(zp, a)
    out = torch.full((B, n), -7, dtype=torch.int32, device="cuda")
    nacc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ws = sb.workspace(sb.spec_accept_workspace_bytes(B, gamma, V))
    sb.spec_accept(_dev(zp_dev), _dev(q), _dev(x), _dev(u), B, gamma, V, T, top_p, out, nacc, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    out, nacc = out.cpu().numpy(), nacc.cpu().numpy()
    excused = near = 0
    for b in range(B):
        r = OA.accept(OC.apply_mask(zp[b], a[b]), q[b] if T > 0 else None, x[b],
                      u[b] if T > 0 else None, T, top_p)
        near += r.boundary
        m = int(nacc[b])
        emitted = out[b, :m + 1]
        assert all(a[b, i, t] for i, t in enumerate(emitted)), (b, emitted.tolist())
        same = m == r.n_accepted and out[b].tolist() == r.tokens
        if not same:
            assert r.boundary, (b, out[b].tolist(), r.tokens)
            excused += 1
    parity.check(f"masked accept B={B} V={V} T={T} top_p={top_p}", B, near, excused)
    assert (nacc > 0).any()


def test_masked_draft_sample_probs():
    R, V, T, top_p = 16, 32000, 0.8, 0.9
    z = wl.accept_logits(9, R, 0, V)[0][:, 0]
    a = wl.allowed_sets(9, R, V, 0.05)
    u = wl.uniforms(9, R)
    zd = _mask_on_device(z, a)
    probs = torch.empty(R, V, device="cuda")
    toks = torch.empty(R, dtype=torch.int32, device="cuda")
    ws = sb.workspace(sb.spec_accept_workspace_bytes(R, 0, V))
    sb.spec_draft_sample(_dev(zd), R, V, T, top_p, _dev(u), probs, toks, ws)
    p = probs.cpu().numpy()
    t = toks.cpu().numpy()
    assert (p[~a] == 0).all()
    excused = near = 0
    for r in range(R):
        qs, ts, bnd = OA.draft_sample(OC.apply_mask(z[r:r + 1], a[r:r + 1]), u[r:r + 1], T, top_p)
        near += bool(bnd[0])
        np.testing.assert_allclose(p[r], qs[0], rtol=1e-5, atol=1e-9)
        if t[r] != ts[0]:
            assert bnd[0], r
            excused += 1
        assert a[r, t[r]]
    parity.check("masked draft sample", R, int(near), excused)


def test_masked_tree_accept_matches_oracle():
    B, V = 32, 4096
    parents = Tr.full_tree_parents(2, 2)
    n = len(parents)
    zq, zp = wl.accept_logits(77, B, n - 1, V)
    a = wl.allowed_sets(77, B * n, V, 0.4).reshape(B, n, V)
    ud = wl.uniforms(77, B, n, stream=8)
    par = np.array(parents)
    q = np.zeros((B, n, V), np.float32)
    toks = np.zeros((B, n), np.int32)
    for b in range(B):
        zqm = OC.apply_mask(zq[b], a[b])
        qs, _, _ = OA.draft_sample(zqm, ud[b], 1.0, 1.0)
        q[b] = qs.astype(np.float32)
        _, xs, _ = OA.draft_sample(zqm[par[1:]], ud[b][1:], 1.0, 1.0)
        toks[b, 1:] = xs
    u = wl.uniforms(77, B, n)
    zp_dev = _mask_on_device(zp, a)
    out = torch.full((B, n), -7, dtype=torch.int32, device="cuda")
    path = torch.full((B, n), -7, dtype=torch.int32, device="cuda")
    nacc = torch.full((B,), -7, dtype=torch.int32, device="cuda")
    ws = sb.workspace(sb.spec_tree_accept_workspace_bytes(B, V))
    sb.spec_tree_accept(_dev(zp_dev), _dev(q), _dev(toks), _dev(np.broadcast_to(par.astype(np.int32), (B, n))),
                        _dev(u), B, n, V, 1.0, 1.0, out, path, nacc, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    out, path, nacc = out.cpu().numpy(), path.cpu().numpy(), nacc.cpu().numpy()
    excused = near = 0
    for b in range(B):
        r = Tr.tree_accept(OC.apply_mask(zp[b], a[b]), q[b], toks[b], parents, u[b], 1.0)
        near += r.boundary
        m = int(nacc[b])
        same = m == r.n_accepted and out[b, :m + 1].tolist() == r.tokens and path[b, :m].tolist() == r.path
        # the emitted token is allowed at the node it follows
        node = 0 if m == 0 else int(path[b, m - 1])
        assert a[b, node, out[b, m]]
        if not same:
            assert r.boundary, (b, out[b].tolist(), r.tokens)
            excused += 1
    parity.check("masked tree accept", B, near, excused)
