"""The 8B-shaped decoder (32 layers, d 4096, 32/8 heads of 128, SwiGLU 14336,
vocab 128256) against the fp64 oracle, in every configuration the
benchmark and the batched workload run:

* batch 1, 2048 cached tokens, gamma in {2, 4, 8}: every logit of the pass,
  then the acceptance step at T = 1 and at T = 0 (greedy) on identical
  fp32 inputs (the oracle's logits) and end to end (each side on its own
  logits, graded outside margins widened to the logits difference);
* batch 16 and 64, per-sequence cached lengths uniform in [512, 4096],
  gamma 4, T 0.8 and top-p 0.9 on p and q: every logit, the acceptance step
  on identical inputs with drafts independent of the target and with drafts
  from noisy copies of the target (noise sigma 0.3 and 1.0, which set the
  acceptance rate), end to end, and the rollback.

The oracle generates the model's weights itself from the seed, once for the
module, and keeps them as bf16 when the host has room.  Batched caches take
their rows from a seeded pool (workloads.kv_pool), so the oracle rebuilds any
(layer, sequence) slice instead of holding the whole fp64 cache.
"""
import numpy as np
import pytest
import torch

import parity
from oracle import accept as OA
from oracle import model as OM
from oracle import weights as OW
from oracle.bf16 import from_bits
from speculative_decoding_verification_pass_gb300 import binding as sb
from speculative_decoding_verification_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu

SEED = 1003
TOL = 1e-2
POOL = 65536


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _mem_available_gb() -> float:
    try:
        with open("/proc/meminfo") as f:
            for line in f:
                if line.startswith("MemAvailable:"):
                    return int(line.split()[1]) / 2 ** 20
    except OSError:
        pass
    return 0.0


@pytest.fixture(scope="module")
def eight():
    cfg = sb.LLAMA_8B
    ocfg = OM.Config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.d_ffn, cfg.vocab)
    mem = _mem_available_gb()
    cache = True if mem > 80 else ("bf16" if mem > 40 else False)
    m = sb.Model(cfg, SEED)
    W = OW.Weights(ocfg, SEED, cache_layers=cache)
    yield cfg, ocfg, m, W
    m.close()


def _rel(got, ref):
    return np.abs(got - ref) / (1.0 + np.abs(ref))


def _dev(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _device_accept(z, q, x, u, T, top_p):
    B, n, V = z.shape
    out = torch.empty(B, n, dtype=torch.int32, device="cuda")
    nacc = torch.empty(B, dtype=torch.int32, device="cuda")
    ws = sb.workspace(sb.spec_accept_workspace_bytes(B, n - 1, V))
    zz = z if torch.is_tensor(z) else _dev(z)
    sb.spec_accept(zz, _dev(q) if q is not None else None, _dev(x),
                   _dev(u) if u is not None else None, B, n - 1, V, T, top_p, out, nacc, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    return out.cpu().numpy(), nacc.cpu().numpy()


def _greedy_near(z, rows, margin):
    """A greedy decision is ungraded end to end when one of the rows it reads
    has its two largest logits closer than the logits difference allows."""
    for r in rows:
        top2 = np.partition(z[r], -2)[-2:]
        if top2[1] - top2[0] <= margin:
            return True
    return False


# ------------------------------------------------------------ batch 1 sweep
@pytest.fixture(scope="module")
def ctx_cache(eight):
    cfg = eight[0]
    ctx = 2048
    K, V = wl.kv_prefix(SEED, cfg.n_layers, 1, cfg.n_kv_heads, ctx, cfg.head_dim)
    return ctx, K, V


def _pass_b1(eight, ctx_cache, toks):
    """One verify pass over toks [1][n] on a fresh copy of the 2048-token
    context on both sides: (device fp32 logits, oracle fp64 logits)."""
    cfg, ocfg, m, W = eight
    ctx, K, V = ctx_cache
    n = toks.shape[1]
    kv = sb.KVCache(cfg, 1, ctx + 16)
    kv.k[:, :, :, :ctx].copy_(torch.from_numpy(K.view(np.int16)).view(torch.bfloat16))
    kv.v[:, :, :, :ctx].copy_(torch.from_numpy(V.view(np.int16)).view(torch.bfloat16))
    kv.len.fill_(ctx)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, 1, n - 1, ctx + 16))
    z = torch.empty(1, n, cfg.vocab, device="cuda")
    sb.spec_verify_forward(m.handle, _dev(toks.astype(np.int32)), 1, n - 1, kv, z, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    assert int(kv.len[0]) == ctx + n
    okv = OM.PrefixKV([ctx], lambda l, b: (from_bits(K[l][b]), from_bits(V[l][b])), extra=16)
    ref = OM.forward(ocfg, W, toks, okv)
    zd = z.double().cpu().numpy()
    del kv
    return zd, ref


@pytest.mark.parametrize("gamma", [2, 4, 8])
def test_8b_gamma_sweep_matches_oracle(eight, ctx_cache, gamma):
    cfg = eight[0]
    V = cfg.vocab
    n = gamma + 1
    seed = 3000 + gamma
    # T = 1: drafts drawn from independent noisy logits by the oracle's own
    # draft rule, then verified
    zq = wl.gauss(seed, (gamma, V), 2.0)
    ud = wl.uniforms(seed, 1, gamma, stream=8)[0]
    q, x, _ = OA.draft_sample(zq, ud, 1.0)
    toks = np.concatenate([wl.tokens(seed, 1, 1, V), x[None].astype(np.int32)], axis=1)
    zd, ref = _pass_b1(eight, ctx_cache, toks)
    err = _rel(zd, ref).max()
    print(f"[8B gamma={gamma}] logits max rel err {err:.2e}")
    assert err <= TOL, err
    q32 = q.astype(np.float32)[None]
    u = wl.uniforms(seed, 1, n)
    ref32 = ref.astype(np.float32)
    out, nacc = _device_accept(ref32, q32, x[None].astype(np.int32), u, 1.0, 1.0)
    r = OA.accept(ref32[0], q32[0], x, u[0], 1.0)
    same = int(nacc[0]) == r.n_accepted and out[0].tolist() == r.tokens
    assert same or r.boundary
    out2, nacc2 = _device_accept(zd.astype(np.float32), q32, x[None].astype(np.int32), u, 1.0, 1.0)
    re = OA.accept(ref32[0], q32[0], x, u[0], 1.0, margins=(5e-3, 5e-3, 5e-3))
    if not re.boundary:
        assert int(nacc2[0]) == re.n_accepted and out2[0].tolist() == re.tokens
    parity.check(f"8B gamma={gamma} T=1 accept", 1, int(r.boundary), int(not same), int(re.boundary))

    # T = 0: the first draft is the target's argmax after t_last (row 0
    # depends on t_last and the context only), the others the argmax of the
    # previous pass's rows, so the walk accepts at least one draft and
    # usually stops at a mismatch
    am = ref[0].argmax(-1)
    xg = np.concatenate([[am[0]], am[1:gamma]]).astype(np.int32)
    tg = np.concatenate([toks[:, :1], xg[None]], axis=1)
    zd, ref = _pass_b1(eight, ctx_cache, tg)
    derr = np.abs(zd - ref).max()
    assert _rel(zd, ref).max() <= TOL
    ref32 = ref.astype(np.float32)
    out, nacc = _device_accept(ref32, None, xg[None], None, 0.0, 1.0)
    r = OA.accept(ref32[0], None, xg, None, 0.0)
    assert int(nacc[0]) == r.n_accepted and out[0].tolist() == r.tokens
    assert r.n_accepted >= 1
    out2, nacc2 = _device_accept(zd.astype(np.float32), None, xg[None], None, 0.0, 1.0)
    skipped = _greedy_near(ref[0], range(min(r.n_accepted, gamma) + 1), 2 * derr)
    if not skipped:
        assert int(nacc2[0]) == r.n_accepted and out2[0].tolist() == r.tokens
    print(f"[8B gamma={gamma} T=0] n_accepted {r.n_accepted}, max |dz| {derr:.2e}")
    parity.check(f"8B gamma={gamma} T=0 accept", 1, 0, 0, int(skipped))


# ------------------------------------------------------------ batched
def _pool_prefix(seed, cfg, lens, Kp, Vp):
    def prefix(l, b):
        idx = wl.kv_pool_index(seed, l, b, cfg.n_kv_heads, int(lens[b]), POOL)
        return from_bits(Kp[idx[0]]), from_bits(Vp[idx[1]])
    return prefix


def _fill_device_cache(seed, cfg, kv, lens, Kp, Vp):
    kd = torch.from_numpy(Kp.view(np.int16)).cuda().view(torch.bfloat16)
    vd = torch.from_numpy(Vp.view(np.int16)).cuda().view(torch.bfloat16)
    for l in range(cfg.n_layers):
        for b in range(len(lens)):
            L = int(lens[b])
            idx = torch.from_numpy(wl.kv_pool_index(seed, l, b, cfg.n_kv_heads, L, POOL)).cuda()
            kv.k[l, b, :, :L] = kd[idx[0]]
            kv.v[l, b, :, :L] = vd[idx[1]]
    kv.len.copy_(torch.from_numpy(lens.astype(np.int32)))


@pytest.mark.parametrize("B", [16, 64])
def test_8b_batched_topp_matches_oracle(eight, B):
    cfg, ocfg, m, W = eight
    V, gamma, T, top_p = cfg.vocab, 4, 0.8, 0.9
    n = gamma + 1
    seed = 4000 + B
    lens = wl.context_lengths(seed, B, 512, 4096).astype(np.int64)
    cap = 4096 + 16
    Kp, Vp = wl.kv_pool(seed, POOL, cfg.head_dim)
    kv = sb.KVCache(cfg, B, cap)
    _fill_device_cache(seed, cfg, kv, lens, Kp, Vp)
    okv = OM.PrefixKV(lens, _pool_prefix(seed, cfg, lens, Kp, Vp), extra=16)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, gamma, cap))
    # drafts from independent noisy logits (no device output enters the oracle)
    zq = wl.gauss(seed, (B, gamma, V), 2.0)
    ud = wl.uniforms(seed, B, gamma, stream=8)
    q = np.zeros((B, gamma, V), np.float32)
    x = np.zeros((B, gamma), np.int32)
    for b in range(B):
        qs, ts, _ = OA.draft_sample(zq[b], ud[b], T, top_p)
        q[b], x[b] = qs.astype(np.float32), ts
    t_last = wl.tokens(seed, B, 1, V)
    block = np.concatenate([t_last, x], axis=1).astype(np.int32)
    z = torch.empty(B, n, V, device="cuda")
    sb.spec_verify_forward(m.handle, _dev(block), B, gamma, kv, z, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    zd = z.double().cpu().numpy()
    ref = OM.forward(ocfg, W, block, okv)
    err = _rel(zd, ref).max()
    print(f"[8B B={B}] logits max rel err {err:.2e}")
    assert err <= TOL, err
    np.testing.assert_array_equal(kv.len.cpu().numpy(), okv.lens)
    ref32 = ref.astype(np.float32)
    u = wl.uniforms(seed, B, n)
    # accept on identical (oracle) logits with the pass's own drafts
    out, nacc = _device_accept(ref32, q, x, u, T, top_p)
    excused = near = 0
    oracle_n = np.zeros(B, np.int64)
    for b in range(B):
        r = OA.accept(ref32[b], q[b], x[b], u[b], T, top_p)
        oracle_n[b] = r.n_accepted
        near += r.boundary
        if not (int(nacc[b]) == r.n_accepted and out[b].tolist() == r.tokens):
            assert r.boundary, b
            excused += 1
    parity.check(f"8B B={B} accept, independent drafts", B, near, excused)
    # end to end: each side on its own logits
    out2, nacc2 = _device_accept(z, q, x, u, T, top_p)
    skipped = 0
    for b in range(B):
        r = OA.accept(ref32[b], q[b], x[b], u[b], T, top_p, margins=(5e-3, 5e-3, 5e-3))
        skipped += r.boundary
        if not r.boundary:
            assert int(nacc2[b]) == r.n_accepted and out2[b].tolist() == r.tokens, b
    parity.check(f"8B B={B} accept end to end", B, 0, 0, skipped)
    # drafts from noisy copies of the target's rows (sigma sets the
    # acceptance rate), accept on identical logits
    for sigma in (0.3, 1.0):
        zs = ref32[:, :gamma] + wl.gauss(seed + int(10 * sigma), (B, gamma, V), sigma)
        us = wl.uniforms(seed + int(10 * sigma), B, gamma, stream=8)
        qs = np.zeros((B, gamma, V), np.float32)
        xs = np.zeros((B, gamma), np.int32)
        for b in range(B):
            qq, tt, _ = OA.draft_sample(zs[b], us[b], T, top_p)
            qs[b], xs[b] = qq.astype(np.float32), tt
        uu = wl.uniforms(seed + int(10 * sigma), B, n)
        o3, n3 = _device_accept(ref32, qs, xs, uu, T, top_p)
        excused = near = 0
        for b in range(B):
            r = OA.accept(ref32[b], qs[b], xs[b], uu[b], T, top_p)
            near += r.boundary
            if not (int(n3[b]) == r.n_accepted and o3[b].tolist() == r.tokens):
                assert r.boundary, (sigma, b)
                excused += 1
        print(f"[8B B={B} sigma={sigma}] mean accepted drafts {n3.mean():.2f} of {gamma}")
        parity.check(f"8B B={B} accept, sigma {sigma} drafts", B, near, excused)
        if sigma == 0.3:
            assert n3.mean() > 1.0
    # rollback by the oracle's decisions
    sb.spec_kv_truncate(kv, _dev(oracle_n.astype(np.int32)), gamma, ws)
    okv.lens = OM.truncate(okv.lens, oracle_n, gamma)
    np.testing.assert_array_equal(kv.len.cpu().numpy(), okv.lens)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    del kv
    torch.cuda.empty_cache()
