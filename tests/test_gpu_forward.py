"""GPU parity of the verification forward, the LM head and the KV rollback.

The oracle generates its own weights from the same seed with its own
Philox4x64-10 + Box-Muller implementation and runs the fp64 decoder with its
own cache; the device runs spec_model_create + spec_verify_forward.  Logits
must agree within |d| <= 1e-2 * (1 + |logit|); the generator must agree
bit-exactly on sampled elements (1-ulp slips allowed on at most 1e-4 of them,
from last-bit differences in fp64 log/sin/cos).
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

TOL = 1e-2


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


def _ocfg(c: sb.ModelConfig) -> OM.Config:
    return OM.Config(c.n_layers, c.d_model, c.n_heads, c.n_kv_heads, c.d_ffn, c.vocab,
                     c.rms_eps, c.rope_theta)


def _close(got, ref, tol=TOL):
    err = np.abs(got - ref) / (1.0 + np.abs(ref))
    assert err.max() <= tol, f"max rel err {err.max():.3e} at {np.unravel_index(err.argmax(), err.shape)}"
    return err.max()


class Pair:
    """A device model + cache and the oracle's model + cache, same seed."""

    def __init__(self, cfg, seed, B, cap):
        self.cfg, self.B, self.cap = cfg, B, cap
        self.model = sb.Model(cfg, seed)
        self.kv = sb.KVCache(cfg, B, cap)
        self.ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, 127, cap))
        self.ocfg = _ocfg(cfg)
        self.W = OW.Weights(self.ocfg, seed)
        self.okv = OM.KVState(self.ocfg, B, cap)

    def gpu(self, toks):
        B, n = toks.shape
        out = torch.empty(B, n, self.cfg.vocab, device="cuda")
        sb.spec_verify_forward(self.model.handle, torch.from_numpy(np.ascontiguousarray(toks)).cuda(),
                               B, n - 1, self.kv, out, self.ws)
        return out.double().cpu().numpy()

    def oracle(self, toks):
        return OM.forward(self.ocfg, self.W, toks, self.okv)

    def prefill(self, toks, chunk=100):
        for c0 in range(0, toks.shape[1], chunk):
            blk = toks[:, c0:c0 + chunk]
            g = self.gpu(blk)
            o = self.oracle(blk)
            _close(g, o)

    def status_ok(self):
        st, bits = sb.spec_device_status(self.ws)
        assert st == sb.SPEC_OK, hex(bits)


SMALL = [
    sb.ModelConfig(2, 256, 4, 2, 256, 1000),        # hd 64, G 2, ragged vocab
    sb.ModelConfig(2, 512, 4, 1, 384, 4099),        # hd 128, G 4, ragged vocab
    sb.ModelConfig(3, 1024, 8, 8, 2048, 2048),      # hd 128, G 1 (MHA), several K tiles
]


@pytest.mark.parametrize("cfg", SMALL, ids=["hd64", "hd128", "mha"])
def test_generator_matches_oracle(cfg):
    m = sb.Model(cfg, 9)
    W = OW.Weights(_ocfg(cfg), 9)
    torch.cuda.synchronize()
    checks = [(-1, 0, None), (-1, 1, None)] + [(l, k, None) for l in range(cfg.n_layers) for k in range(7)]
    slips = total = 0
    for layer, which, _ in checks:
        dev = m.tensor(layer, which).view(torch.int16).cpu().numpy().view(np.uint16)
        if layer == -1:
            ref = OW.tensor(9, which, cfg.vocab, cfg.d_model)
        else:
            ref = W.layer(layer)[which]
        got = from_bits(dev)
        diff = got != ref
        total += got.size
        if diff.any():
            # at most one bf16 ulp apart
            ulp = np.abs(got[diff] - ref[diff]) / np.maximum(np.abs(ref[diff]), 1e-30)
            assert (ulp <= 2 ** -7 + 1e-12).all()
            slips += int(diff.sum())
    assert slips <= max(1, total // 10000), (slips, total)
    m.close()


@pytest.mark.parametrize("cfg", SMALL, ids=["hd64", "hd128", "mha"])
def test_forward_matches_oracle_ragged_batch(cfg):
    """Prefill 2 sequences (300 tokens: 3 key chunks, ragged), verify a
    gamma=4 block, roll back different amounts per sequence, verify again."""
    B, cap, gamma = 2, 320, 4
    pr = Pair(cfg, 21, B, cap)
    pr.prefill(wl.tokens(3, B, 300, cfg.vocab))
    blk = wl.tokens(4, B, gamma + 1, cfg.vocab)
    _close(pr.gpu(blk), pr.oracle(blk))
    n_acc = np.array([1, 4], np.int32)[:B]
    sb.spec_kv_truncate(pr.kv, torch.from_numpy(n_acc).cuda(), gamma, pr.ws)
    pr.okv.lens = OM.truncate(pr.okv.lens, n_acc, gamma)
    np.testing.assert_array_equal(pr.kv.len.cpu().numpy(), pr.okv.lens)
    blk = wl.tokens(5, B, gamma + 1, cfg.vocab)
    _close(pr.gpu(blk), pr.oracle(blk))
    # the cache contents (bf16) agree with the oracle's cache
    for l in range(cfg.n_layers):
        for b in range(B):
            Lb = int(pr.okv.lens[b])
            kd = pr.kv.k[l, b, :, :Lb].double().cpu().numpy()
            vd = pr.kv.v[l, b, :, :Lb].double().cpu().numpy()
            _close(kd, pr.okv.K[l][b, :, :Lb])
            _close(vd, pr.okv.V[l][b, :, :Lb])
    pr.status_ok()
    pr.model.close()


ATT_PATHS = [("1", "1"), ("1", "0"), ("0", "1")]
ATT_IDS = ["tcgen05_tma", "tcgen05_copies", "mma_sync"]


@pytest.mark.parametrize("tc,tma", ATT_PATHS, ids=ATT_IDS)
def test_attention_paths_match_oracle(tc, tma, monkeypatch):
    """Head dim 128 has these attention paths in the persistent forward: S^T
    and O^T as tcgen05 MMAs with TMEM accumulators (the default where the
    shape fits), its key blocks loaded by TMA or by per-thread copies, and
    warp-level MMAs.  Each matches the oracle on a ragged batch of 2 (300
    cached tokens: 3 key blocks) verifying a gamma=4 block, before and after a
    rollback."""
    monkeypatch.setenv("SPEC_ATTENTION_TC", tc)
    monkeypatch.setenv("SPEC_ATTENTION_TMA", tma)
    cfg = SMALL[1]
    B, cap, gamma = 2, 320, 4
    pr = Pair(cfg, 23, B, cap)
    pr.prefill(wl.tokens(13, B, 300, cfg.vocab))
    blk = wl.tokens(14, B, gamma + 1, cfg.vocab)
    _close(pr.gpu(blk), pr.oracle(blk))
    n_acc = np.array([0, 3], np.int32)
    sb.spec_kv_truncate(pr.kv, torch.from_numpy(n_acc).cuda(), gamma, pr.ws)
    pr.okv.lens = OM.truncate(pr.okv.lens, n_acc, gamma)
    blk = wl.tokens(15, B, gamma + 1, cfg.vocab)
    _close(pr.gpu(blk), pr.oracle(blk))
    pr.status_ok()
    pr.model.close()


@pytest.mark.parametrize("tc,tma", ATT_PATHS, ids=ATT_IDS)
def test_stale_cache_slots_do_not_leak(tc, tma, monkeypatch):
    """Cache slots past a sequence's length hold whatever the buffer held
    (a rolled-back pass, never-written memory): fill them with NaN in every
    layer, K and V, and a verify pass still matches the oracle.  The key
    blocks of a chunk's end are read whole, so this pins the visibility mask
    on K and the zeroed V rows."""
    monkeypatch.setenv("SPEC_ATTENTION_TC", tc)
    monkeypatch.setenv("SPEC_ATTENTION_TMA", tma)
    cfg = SMALL[1]
    B, cap, gamma = 2, 320, 4
    pr = Pair(cfg, 29, B, cap)
    pr.prefill(wl.tokens(17, B, 203, cfg.vocab))
    nan = torch.tensor(0x7FC0, dtype=torch.int16).view(torch.bfloat16)
    lens = pr.kv.len.cpu().numpy()
    for b in range(B):
        pr.kv.k[:, b, :, int(lens[b]):] = nan
        pr.kv.v[:, b, :, int(lens[b]):] = nan
    blk = wl.tokens(18, B, gamma + 1, cfg.vocab)
    got = pr.gpu(blk)
    assert np.isfinite(got).all()
    _close(got, pr.oracle(blk))
    pr.status_ok()
    pr.model.close()


def _bf16_ulp(x):
    """Spacing of bf16 values at |x| (8 significant bits)."""
    a = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(a)) - 7)


@pytest.mark.parametrize("L0", [4091, 32003])
def test_rope_cache_rows_at_large_positions(L0):
    """Keys written at cached positions L0 .. L0+4 (up to 32007 of a
    32768-slot cache) agree with the oracle's bf16 keys to within one bf16
    ulp, and all but a small fraction agree exactly: the rotation angle is
    reduced by whole turns before the sine is taken, so its error stays near
    1e-7 rad at any position (an unreduced fast sine loses ~|angle| * 2^-22).
    Layer 0's keys depend only on the token, its position and the weights,
    so the cache below L0 can stay empty."""
    cfg = sb.ModelConfig(1, 512, 4, 2, 256, 1000)   # hd 128
    B, cap, n = 1, 32768, 5
    m = sb.Model(cfg, 77)
    kv = sb.KVCache(cfg, B, cap)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, n - 1, cap))
    kv.len.fill_(L0)
    toks = wl.tokens(78 + L0, B, n, cfg.vocab)
    out = torch.empty(B, n, cfg.vocab, device="cuda")
    sb.spec_verify_forward(m.handle, torch.from_numpy(toks).cuda(), B, n - 1, kv, out, ws)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    ocfg = _ocfg(cfg)
    W = OW.Weights(ocfg, 77)
    w = W.layer(0)
    x = OM.rmsnorm(W.embed_rows(toks[0]).astype(np.float64), W.norm_gain(), ocfg.rms_eps)
    hd = ocfg.head_dim
    k = (x @ w[OW.WK].astype(np.float64).T).reshape(n, ocfg.n_kv_heads, hd).transpose(1, 0, 2)
    v = (x @ w[OW.WV].astype(np.float64).T).reshape(n, ocfg.n_kv_heads, hd).transpose(1, 0, 2)
    pos = L0 + np.arange(n)
    from oracle.bf16 import round_bf16
    kref = round_bf16(OM.rope(k, pos, ocfg.rope_theta))
    vref = round_bf16(v)
    kd = kv.k[0, 0, :, L0:L0 + n].double().cpu().numpy()
    vd = kv.v[0, 0, :, L0:L0 + n].double().cpu().numpy()
    for got, ref in ((kd, kref), (vd, vref)):
        diff = np.abs(got - ref)
        assert (diff <= _bf16_ulp(ref) * (1 + 1e-9)).all(), diff.max()
        frac = float((diff > 0).mean())
        print("bf16 rows differing by one ulp: %.4f" % frac)
        assert frac < 0.02, frac
    m.close()


def test_one_pass_equals_sequential_passes_on_device():
    cfg = SMALL[1]
    B, cap, gamma = 2, 200, 4
    a = Pair(cfg, 8, B, cap)
    b = Pair(cfg, 8, B, cap)
    pre = wl.tokens(6, B, 150, cfg.vocab)
    a.gpu(pre[:, :100]); a.gpu(pre[:, 100:])
    b.gpu(pre[:, :100]); b.gpu(pre[:, 100:])
    blk = wl.tokens(7, B, gamma + 1, cfg.vocab)
    one = a.gpu(blk)
    seq = np.concatenate([b.gpu(blk[:, j:j + 1]) for j in range(gamma + 1)], axis=1)
    np.testing.assert_allclose(one, seq, rtol=1e-4, atol=1e-4)
    np.testing.assert_array_equal(a.kv.len.cpu().numpy(), b.kv.len.cpu().numpy())


def test_rollback_then_reverify_equals_fresh_pass_on_device():
    cfg = SMALL[0]
    B, cap, gamma = 1, 128, 4
    a = Pair(cfg, 12, B, cap)
    b = Pair(cfg, 12, B, cap)
    pre = wl.tokens(9, B, 40, cfg.vocab)
    a.gpu(pre)
    b.gpu(pre)
    blk = np.array([[7, 11, 13, 17, 19]], np.int32)
    a.gpu(blk)
    sb.spec_kv_truncate(a.kv, torch.tensor([1], dtype=torch.int32, device="cuda"), gamma, a.ws)
    b.gpu(blk[:, :2])
    nxt = np.array([[23, 29, 31, 37, 41]], np.int32)
    np.testing.assert_allclose(a.gpu(nxt), b.gpu(nxt), rtol=1e-5, atol=1e-5)


def test_device_status_on_overflow_and_bad_token():
    cfg = SMALL[0]
    B, cap = 2, 16
    pr = Pair(cfg, 3, B, cap)
    pr.kv.len.copy_(torch.tensor([10, 14], dtype=torch.int32))
    toks = np.array([[1, 2, 3], [4, 5, cfg.vocab + 5]], np.int32)   # seq 1 overflows, bad id
    pr.gpu(toks)
    st, bits = sb.spec_device_status(pr.ws)
    assert st == sb.SPEC_EDEVICE
    assert bits & sb.DEV_KV_OVERFLOW and bits & sb.DEV_BAD_TOKEN
    assert pr.kv.len.cpu().tolist() == [13, 14]
    st, bits = sb.spec_device_status(pr.ws)      # cleared by the read
    assert st == sb.SPEC_OK and bits == 0
    # truncate with n_accepted out of range leaves len alone and flags it
    sb.spec_kv_truncate(pr.kv, torch.tensor([5, -1], dtype=torch.int32, device="cuda"), 2, pr.ws)
    st, bits = sb.spec_device_status(pr.ws)
    assert bits & sb.DEV_BAD_NACC and pr.kv.len.cpu().tolist() == [13, 14]


def test_lm_head_workload_and_accept():
    """LM head 4096 x 32000 on 5 activation rows ~ N(0,1) (bf16), draft
    probabilities from the same head on activations + N(0, 0.3^2), T = 1:
    skinny GEMM then fused accept, checked against the oracle."""
    cfg = sb.ModelConfig(0, 4096, 32, 8, 128, 32000)
    seed = 41
    m = sb.Model(cfg, seed)
    head = OW.tensor(seed, OW.HEAD, cfg.vocab, cfg.d_model)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, 5, 0, 1))
    hb = wl.hidden_bf16(seed, 5, cfg.d_model)
    h = from_bits(hb)
    z = torch.empty(5, cfg.vocab, device="cuda")
    sb.spec_lm_head(m.handle, torch.from_numpy(hb.view(np.int16)).cuda(), 5, z, ws)
    zp = z.cpu().numpy()
    ref = OM.lm_head(h, head)
    _close(zp.astype(np.float64), ref, 1e-4)
    # draft: the same head on noisy activations (oracle side, fp64)
    noisy = h[:4] + wl.gauss(seed, (4, cfg.d_model), 0.3)
    zq = OM.lm_head(noisy, head)
    ud = wl.uniforms(seed, 1, 4, stream=8)[0]
    q, x, _ = OA.draft_sample(zq, ud, 1.0)
    u = wl.uniforms(seed, 1, 5)
    out = torch.empty(1, 5, dtype=torch.int32, device="cuda")
    nacc = torch.empty(1, dtype=torch.int32, device="cuda")
    aws = sb.workspace(sb.spec_accept_workspace_bytes(1, 4, cfg.vocab))
    q32 = q.astype(np.float32)
    dq = torch.from_numpy(q32[None]).cuda()
    dx = torch.from_numpy(x.astype(np.int32)[None]).cuda()
    du = torch.from_numpy(u).cuda()
    ref32 = ref.astype(np.float32)
    # identical (oracle) fp32 logits on both sides: exact outside the margins
    sb.spec_accept(torch.from_numpy(ref32[None]).cuda(), dq, dx, du, 1, 4, cfg.vocab, 1.0, 1.0,
                   out, nacc, aws)
    r = OA.accept(ref32, q32, x, u[0], 1.0)
    same = int(nacc[0]) == r.n_accepted and out[0].tolist() == r.tokens
    assert same or r.boundary
    # end to end: the device decides on its own logits, the oracle on its
    # own; decisions closer to a boundary than the logits tolerance are
    # counted, not graded
    sb.spec_accept(z.view(1, 5, -1), dq, dx, du, 1, 4, cfg.vocab, 1.0, 1.0, out, nacc, aws)
    re = OA.accept(ref32, q32, x, u[0], 1.0, margins=(5e-3, 5e-3, 5e-3))
    if not re.boundary:
        assert int(nacc[0]) == re.n_accepted and out[0].tolist() == re.tokens
    parity.check("LM-head workload accept", 1, int(r.boundary), int(not same), int(re.boundary))
    m.close()


def _device_pass(cfg, seed, B, cap, prompt, blk, persistent, monkeypatch):
    """Prefill `prompt` (per-step schedule: more than 32 query rows per KV
    head), then verify `blk` under the chosen schedule; returns the block's
    logits, the caches and the per-kind launch counts of the block's pass."""
    monkeypatch.setenv("SPEC_FORWARD_PERSISTENT", "1" if persistent else "0")
    m = sb.Model(cfg, seed)
    kv = sb.KVCache(cfg, B, cap)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, 127, cap))

    def run(toks):
        Bn, n = toks.shape
        out = torch.empty(Bn, n, cfg.vocab, device="cuda")
        sb.spec_verify_forward(m.handle, torch.from_numpy(np.ascontiguousarray(toks)).cuda(), Bn,
                               n - 1, kv, out, ws)
        return out.double().cpu().numpy()

    run(prompt)
    sb.spec_timing_enable(m.handle, True)
    sb.spec_timing_read(m.handle)
    z = run(blk)
    _, launches, _ = sb.spec_timing_read(m.handle)
    sb.spec_timing_enable(m.handle, False)
    st, bits = sb.spec_device_status(ws)
    assert st == sb.SPEC_OK, hex(bits)
    res = (z, kv.k.double().cpu().numpy(), kv.v.double().cpu().numpy(), kv.len.cpu().numpy(),
           launches)
    m.close()
    return res


@pytest.mark.parametrize("cfg", SMALL, ids=["hd64", "hd128", "mha"])
def test_persistent_and_per_step_schedules_agree(cfg, monkeypatch):
    """A decode-shaped pass runs as ONE persistent kernel (timing kind 2);
    forcing the per-step schedule on an identical model and cache gives the
    same logits up to fp32 summation order (the two split the GEMMs'
    K dimension differently) and the same cache up to one bf16 rounding."""
    B, cap, gamma = 3, 200, 4
    prompt = wl.tokens(51, B, 97, cfg.vocab)
    blk = wl.tokens(52, B, gamma + 1, cfg.vocab)
    zp, kp, vp, lp, np_ = _device_pass(cfg, 61, B, cap, prompt, blk, True, monkeypatch)
    zs, ks, vs, ls, ns_ = _device_pass(cfg, 61, B, cap, prompt, blk, False, monkeypatch)
    assert np_[2] == 1 and np_[0] == 0 and np_[1] == 0, np_
    assert ns_[2] == 0 and ns_[0] == 4 * cfg.n_layers + 1 and ns_[1] == cfg.n_layers, ns_
    np.testing.assert_array_equal(lp, ls)
    _close(zp, zs, tol=1e-3)
    _close(kp, ks, tol=8e-3)
    _close(vp, vs, tol=8e-3)


def test_graph_replays_recompute_every_pass():
    """The persistent kernel tags its stream-K words with a launch epoch kept
    in the workspace, so replays of one captured graph (frozen parameters)
    never take an earlier replay's words as current: every replay with new
    tokens in place must give the eager pass's logits exactly."""
    cfg = SMALL[1]
    B, cap, n = 2, 96, 5
    m = sb.Model(cfg, 12)
    kv_g = sb.KVCache(cfg, B, cap)
    kv_e = sb.KVCache(cfg, B, cap)
    ws_g = sb.workspace(sb.spec_workspace_bytes(cfg, B, n - 1, cap))
    ws_e = sb.workspace(sb.spec_workspace_bytes(cfg, B, n - 1, cap))
    toks = torch.zeros(B, n, dtype=torch.int32, device="cuda")
    out_g = torch.empty(B, n, cfg.vocab, device="cuda")
    out_e = torch.empty_like(out_g)
    for kv in (kv_g, kv_e):
        kv.len.fill_(20)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        sb.spec_verify_forward(m.handle, toks, B, n - 1, kv_g, out_g, ws_g, st)   # warm-up
        kv_g.len.fill_(20)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            sb.spec_verify_forward(m.handle, toks, B, n - 1, kv_g, out_g, ws_g, st)
    for it in range(4):
        toks.copy_(torch.from_numpy(wl.tokens(100 + it, B, n, cfg.vocab).astype(np.int32)))
        kv_g.len.fill_(20 + it)
        kv_e.len.fill_(20 + it)
        g.replay()
        sb.spec_verify_forward(m.handle, toks, B, n - 1, kv_e, out_e, ws_e)
        torch.cuda.synchronize()
        assert torch.equal(out_g, out_e), it
    for ws in (ws_g, ws_e):
        stt, bits = sb.spec_device_status(ws)
        assert stt == sb.SPEC_OK, hex(bits)


def test_bounded_wait_gives_up_and_the_context_stays_usable():
    """The persistent forward's grid-barrier wait on a counter that nothing
    advances: it gives up after its limit, sets the timeout bit, the kernel
    returns, and afterwards a verify pass gives the same logits as before."""
    import time
    cfg = SMALL[1]
    B, cap, n = 1, 64, 5
    m = sb.Model(cfg, 21)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, n - 1, cap))
    toks = torch.from_numpy(wl.tokens(31, B, n, cfg.vocab).astype(np.int32)).cuda()

    def verify():
        kv = sb.KVCache(cfg, B, cap)
        kv.len.fill_(7)
        out = torch.empty(B, n, cfg.vocab, device="cuda")
        sb.spec_verify_forward(m.handle, toks, B, n - 1, kv, out, ws)
        assert sb.spec_device_status(ws) == (sb.SPEC_OK, 0)
        return out

    before = verify()
    ctr = torch.full((1,), 3, dtype=torch.int32, device="cuda")
    sb.spec_wait_selftest(ctr, 3, 50.0, ws)            # already reached: no timeout
    assert sb.spec_device_status(ws) == (sb.SPEC_OK, 0)
    ctr.zero_()                                        # nothing advances it
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    sb.spec_wait_selftest(ctr, 1, 50.0, ws)
    st, bits = sb.spec_device_status(ws)
    waited = time.perf_counter() - t0
    assert st == sb.SPEC_ETIMEOUT and bits == sb.DEV_TIMEOUT, (st, hex(bits))
    assert waited >= 0.045, waited
    assert sb.spec_device_status(ws) == (sb.SPEC_OK, 0)   # read and cleared
    assert torch.equal(verify(), before)
    with pytest.raises(sb.SpecError):
        sb.spec_wait_selftest(ctr, 1, 0.0, ws)
