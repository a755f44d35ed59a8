"""The decoder workloads at their full sizes.

* 1B-shaped decoder (16 layers, d 2048, 32/8 heads of 64, SwiGLU 8192, vocab
  32000): a 512-token prefix uniform over the vocabulary is prefilled through
  spec_verify_forward, then a gamma=4 pass is verified; every logit of every
  pass is compared with the fp64 oracle running on its own weights and cache;
  accept + rollback follow, then a second pass is compared again.
* Batched workload at the 1B shape (batch 16 and 64, ragged cached lengths,
  T 0.8, top-p 0.9): logits, accept and rollback against the oracle.
* 8B-shaped decoder (32 layers, d 4096, 32/8 heads of 128, SwiGLU 14336,
  vocab 128256) with 2048 cached tokens, the launch configuration the
  benchmark times: properties that hold at any size (one pass over gamma+1
  equals gamma+1 single-token passes; rollback then re-verify equals a fresh
  pass).  Its logits and accept decisions against the oracle, for every
  gamma, temperature and batch the workloads name, are in
  test_gpu_8b_oracle.py.
"""
import numpy as np
import pytest
import torch

import parity
from oracle import accept as OA
from oracle import model as OM
from oracle import weights as OW
from speculative_decoding_verification_pass_gb300 import binding as sb
from speculative_decoding_verification_pass_gb300 import workloads as wl

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _rel(got, ref):
    return (np.abs(got - ref) / (1.0 + np.abs(ref))).max()


def test_1b_workload_matches_oracle():
    cfg = sb.LLAMA_1B
    ocfg = OM.Config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.d_ffn, cfg.vocab)
    seed, B, gamma, L0 = 1002, 1, 4, 512
    cap = L0 + 2 * (gamma + 1) + 8
    m = sb.Model(cfg, seed)
    kv = sb.KVCache(cfg, B, cap)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, 127, cap))
    W = OW.Weights(ocfg, seed)
    okv = OM.KVState(ocfg, B, cap)
    prefix = wl.tokens(seed, B, L0, cfg.vocab)
    worst = 0.0
    for c0 in range(0, L0, 128):
        blk = prefix[:, c0:c0 + 128]
        z = torch.empty(B, blk.shape[1], cfg.vocab, device="cuda")
        sb.spec_verify_forward(m.handle, torch.from_numpy(np.ascontiguousarray(blk)).cuda(), B,
                               blk.shape[1] - 1, kv, z, ws)
        ref = OM.forward(ocfg, W, blk, okv)
        worst = max(worst, _rel(z.double().cpu().numpy(), ref))
    assert worst <= 1e-2, worst
    # the verify pass: t_last + 4 drafts drawn as in the accept-only workload
    zq, _ = wl.accept_logits(seed, B, gamma, cfg.vocab)
    ud = wl.uniforms(seed, B, gamma, stream=8)
    q, x, _ = OA.draft_sample(zq[0, :gamma], ud[0], 1.0)
    t_last = wl.tokens(seed + 1, B, 1, cfg.vocab)
    block = np.concatenate([t_last, x[None].astype(np.int32)], axis=1)
    z = torch.empty(B, gamma + 1, cfg.vocab, device="cuda")
    sb.spec_verify_forward(m.handle, torch.from_numpy(block).cuda(), B, gamma, kv, z, ws)
    ref = OM.forward(ocfg, W, block, okv)
    zg = z.cpu().numpy()
    err = _rel(zg.astype(np.float64), ref)
    assert err <= 1e-2, err
    u = wl.uniforms(seed, B, gamma + 1)
    out = torch.empty(B, gamma + 1, dtype=torch.int32, device="cuda")
    nacc = torch.empty(B, dtype=torch.int32, device="cuda")
    aws = sb.workspace(sb.spec_accept_workspace_bytes(B, gamma, cfg.vocab))
    q32 = q.astype(np.float32)
    dq = torch.from_numpy(q32[None]).cuda()
    dx = torch.from_numpy(x.astype(np.int32)[None]).cuda()
    du = torch.from_numpy(u).cuda()
    # the accept on identical (oracle) fp32 logits: exact outside the margins
    ref32 = ref[0].astype(np.float32)
    sb.spec_accept(torch.from_numpy(ref32[None]).cuda(), dq, dx, du, B, gamma, cfg.vocab, 1.0, 1.0,
                   out, nacc, aws)
    r = OA.accept(ref32, q32, x, u[0], 1.0)
    same = int(nacc[0]) == r.n_accepted and out[0].tolist() == r.tokens
    assert same or r.boundary
    # end to end: each side's accept on its own logits, graded outside
    # margins widened to the logits tolerance
    sb.spec_accept(z, dq, dx, du, B, gamma, cfg.vocab, 1.0, 1.0, out, nacc, aws)
    re = OA.accept(ref32, q32, x, u[0], 1.0, margins=(5e-3, 5e-3, 5e-3))
    n_dev = int(nacc[0])
    if not re.boundary:
        assert n_dev == re.n_accepted and out[0].tolist() == re.tokens
    parity.check("1B verify step accept", 1, int(r.boundary), int(not same), int(re.boundary))
    sb.spec_kv_truncate(kv, nacc, gamma, ws)
    okv.lens = OM.truncate(okv.lens, [n_dev], gamma)
    assert kv.len.cpu().tolist() == okv.lens.tolist() == [L0 + 1 + n_dev]
    # next pass from the device's emitted token
    nxt = np.array([[int(out[0, n_dev])] + list(wl.tokens(seed + 2, 1, gamma, cfg.vocab)[0])],
                   np.int32)
    sb.spec_verify_forward(m.handle, torch.from_numpy(nxt).cuda(), B, gamma, kv, z, ws)
    ref = OM.forward(ocfg, W, nxt, okv)
    assert _rel(z.double().cpu().numpy(), ref) <= 1e-2
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, bits
    m.close()


@pytest.fixture(scope="module")
def big():
    cfg = sb.LLAMA_8B
    seed, B, ctx = 1003, 1, 2048
    cap = ctx + 64
    m = sb.Model(cfg, seed)
    K, V = wl.kv_prefix(seed, cfg.n_layers, B, cfg.n_kv_heads, ctx, cfg.head_dim)
    kv = sb.KVCache(cfg, B, cap)
    kv.k[:, :, :, :ctx].copy_(torch.from_numpy(K.view(np.int16)).view(torch.bfloat16))
    kv.v[:, :, :, :ctx].copy_(torch.from_numpy(V.view(np.int16)).view(torch.bfloat16))
    del K, V
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, 8, cap))
    yield cfg, m, kv, ws, ctx
    m.close()


def _run(cfg, m, kv, ws, toks):
    B, n = toks.shape
    z = torch.empty(B, n, cfg.vocab, device="cuda")
    sb.spec_verify_forward(m.handle, torch.from_numpy(np.ascontiguousarray(toks)).cuda(), B, n - 1,
                           kv, z, ws)
    return z


@pytest.mark.parametrize("gamma", [2, 4, 8])
def test_8b_one_pass_equals_sequential(big, gamma):
    cfg, m, kv, ws, ctx = big
    toks = wl.tokens(50 + gamma, 1, gamma + 1, cfg.vocab)
    kv.len.fill_(ctx)
    one = _run(cfg, m, kv, ws, toks).double().cpu().numpy()
    kv.len.fill_(ctx)
    seq = np.concatenate([_run(cfg, m, kv, ws, toks[:, j:j + 1]).double().cpu().numpy()
                          for j in range(gamma + 1)], axis=1)
    assert np.isfinite(one).all()
    assert _rel(one, seq) <= 1e-3
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, bits


def test_8b_rollback_then_reverify_equals_fresh(big):
    cfg, m, kv, ws, ctx = big
    gamma = 4
    blk = wl.tokens(60, 1, gamma + 1, cfg.vocab)
    nxt = wl.tokens(61, 1, gamma + 1, cfg.vocab)
    kv.len.fill_(ctx)
    _run(cfg, m, kv, ws, blk)
    sb.spec_kv_truncate(kv, torch.tensor([2], dtype=torch.int32, device="cuda"), gamma, ws)
    assert int(kv.len[0]) == ctx + 3
    a = _run(cfg, m, kv, ws, nxt).double().cpu().numpy()
    kv.len.fill_(ctx)
    _run(cfg, m, kv, ws, blk[:, :3])
    b = _run(cfg, m, kv, ws, nxt).double().cpu().numpy()
    assert _rel(a, b) <= 1e-5


def _batched_topp(B, steps, seed, lo, hi):
    """The batched workload (ragged cached lengths ~ U{lo..hi}, capacity
    hi+16, gamma 4, T 0.8, top-p 0.9 on p and q; draft logits independent
    N(0, 2^2), so that no device output enters the oracle) at the 1B shape:
    every logit of every pass against the fp64 oracle on its own weights and
    the same cache bytes; the accept kernel against the oracle on identical
    (oracle) logits, and end to end outside margins widened to the logits
    tolerance; rollback by the oracle's decisions."""
    cfg = sb.LLAMA_1B
    gamma, T, top_p, cap = 4, 0.8, 0.9, hi + 16
    n = gamma + 1
    ocfg = OM.Config(cfg.n_layers, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.d_ffn, cfg.vocab)
    lens = wl.context_lengths(seed, B, lo, hi)
    Lmax = int(lens.max())
    m = sb.Model(cfg, seed)
    kv = sb.KVCache(cfg, B, cap)
    W = OW.Weights(ocfg, seed)
    okv = OM.KVState(ocfg, B, cap)
    K, V = wl.kv_prefix(seed, cfg.n_layers, B, cfg.n_kv_heads, Lmax, cfg.head_dim)
    from oracle.bf16 import from_bits
    okv.load_prefix([from_bits(K[l]) for l in range(cfg.n_layers)],
                    [from_bits(V[l]) for l in range(cfg.n_layers)], lens)
    kv.k[:, :, :, :Lmax].copy_(torch.from_numpy(K.view(np.int16)).view(torch.bfloat16))
    kv.v[:, :, :, :Lmax].copy_(torch.from_numpy(V.view(np.int16)).view(torch.bfloat16))
    del K, V
    kv.len.copy_(torch.from_numpy(lens))
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, gamma, cap))
    aws = sb.workspace(sb.spec_accept_workspace_bytes(B, gamma, cfg.vocab))
    t_last = wl.tokens(seed + 1, B, 1, cfg.vocab)[:, 0]
    excused = near = skipped = 0
    for step in range(steps):
        x = np.zeros((B, gamma), np.int32)
        q = np.zeros((B, gamma, cfg.vocab), np.float32)
        ud = wl.uniforms(seed + 10 * step, B, gamma, stream=8)
        # drafts from independent noisy logits (no device output enters the oracle)
        zq = wl.gauss(seed + 10 * step, (B, gamma, cfg.vocab), 2.0)
        for b in range(B):
            qs, ts, _ = OA.draft_sample(zq[b], ud[b], T, top_p)
            q[b] = qs.astype(np.float32)
            x[b] = ts
        block = np.concatenate([t_last[:, None], x], axis=1).astype(np.int32)
        z = torch.empty(B, n, cfg.vocab, device="cuda")
        sb.spec_verify_forward(m.handle, torch.from_numpy(block).cuda(), B, gamma, kv, z, ws)
        st, bits = sb.spec_device_status(ws)
        assert st == sb.SPEC_OK, hex(bits)
        zd = z.double().cpu().numpy()
        ref = OM.forward(ocfg, W, block, okv)
        assert _rel(zd, ref) <= 1e-2, (step, _rel(zd, ref))
        np.testing.assert_array_equal(kv.len.cpu().numpy(), okv.lens)
        u = wl.uniforms(seed + 10 * step, B, n)
        # accept on identical (oracle) fp32 logits: exact except boundary cases
        ref32 = ref.astype(np.float32)
        out = torch.empty(B, n, dtype=torch.int32, device="cuda")
        nacc = torch.empty(B, dtype=torch.int32, device="cuda")
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        sb.spec_accept(dev(ref32), dev(q), dev(x), dev(u), B, gamma, cfg.vocab, T, top_p, out, nacc, aws)
        o, na = out.cpu().numpy(), nacc.cpu().numpy()
        oracle_n = np.zeros(B, np.int32)
        for b in range(B):
            r = OA.accept(ref32[b], q[b], x[b], u[b], T, top_p)
            oracle_n[b] = r.n_accepted
            near += r.boundary
            if not (int(na[b]) == r.n_accepted and o[b].tolist() == r.tokens):
                assert r.boundary, (step, b)
                excused += 1
        # end to end: the device's accept on the device's logits
        sb.spec_accept(z, dev(q), dev(x), dev(u), B, gamma, cfg.vocab, T, top_p, out, nacc, aws)
        o2, na2 = out.cpu().numpy(), nacc.cpu().numpy()
        for b in range(B):
            r = OA.accept(ref32[b], q[b], x[b], u[b], T, top_p, margins=(5e-3, 5e-3, 5e-3))
            skipped += r.boundary
            if not r.boundary:
                assert int(na2[b]) == r.n_accepted and o2[b].tolist() == r.tokens, (step, b)
        # roll both caches back by the oracle's decisions; emitted token = next t_last
        sb.spec_kv_truncate(kv, dev(oracle_n), gamma, ws)
        okv.lens = OM.truncate(okv.lens, oracle_n, gamma)
        np.testing.assert_array_equal(kv.len.cpu().numpy(), okv.lens)
        t_last = np.array([OA.accept(ref32[b], q[b], x[b], u[b], T, top_p).tokens[oracle_n[b]]
                           for b in range(B)], np.int32)
    parity.check(f"1B batched accept B={B} steps={steps}", B * steps, near, excused, skipped)
    m.close()


def test_batched_topp_workload_b16_two_steps():
    """Batch 16, cached lengths U{512..4096} (80 token rows: the persistent
    kernel), two verify steps."""
    _batched_topp(16, 2, 2016, 512, 4096)


def test_batched_topp_workload_b64():
    """Batch 64 (320 token rows: one kernel per step), cached lengths
    U{512..1024} (the oracle's fp64 cache at 4096 slots would need ~34 GB of
    host memory), one verify step."""
    _batched_topp(64, 1, 2064, 512, 1024)
