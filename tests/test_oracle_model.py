"""Pins of the forward / rollback / weight-generator oracle.

CPU only.  The pages print no logits, so the forward is pinned by library
routines (torch fp64 CPU ops) for each sublayer, by mathematical invariants
(RoPE is a rotation that depends only on relative position; one key makes
attention return its value) and by the two properties the pages rely on:
one pass over gamma+1 positions equals gamma+1 single-token passes, and a
rollback followed by a new pass equals a fresh pass over the accepted prefix.
"""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import model as Mo
from oracle import weights as W
from oracle.bf16 import round_bf16, to_bits, from_bits

TINY = Mo.Config(n_layers=2, d_model=64, n_heads=4, n_kv_heads=2, d_ffn=96, vocab=50)


# ---------------------------------------------------------------- generator
def test_philox4x64_known_answers():
    """Published Philox4x64-10 known-answer vectors (Random123 kat_vectors):
    counter 0 / key 0 and counter all-ones / key all-ones."""
    m = 2 ** 64 - 1
    bg = np.random.Philox(counter=[m, m, m, m], key=[0, 0])        # emits counter 0
    assert [hex(x) for x in bg.random_raw(4)] == [
        "0x16554d9eca36314c", "0xdb20fe9d672d0fdc", "0xd7e772cee186176b", "0x7e68b68aec7ba23b"]
    bg = np.random.Philox(counter=[m - 1, m, m, m], key=[m, m])   # emits counter all-ones
    assert [hex(x) for x in bg.random_raw(4)] == [
        "0x87b092c3013fe90b", "0x438c3c67be8d0224", "0x9cc7d7c69cd777b6", "0xa09caebf594f0ba0"]


def test_block_addressing_is_random_access():
    a = W.normals(5, 9, 0, 64)
    b = W.normals(5, 9, 13, 30)
    np.testing.assert_array_equal(a[13:43], b)
    c = W.normals(6, 9, 0, 64)
    assert not np.allclose(a, c)


def test_box_muller_moments():
    z = W.normals(123, 3, 0, 1 << 20)
    n = z.size
    assert abs(z.mean()) < 4 / np.sqrt(n)
    assert abs(z.var() - 1) < 4 * np.sqrt(2 / n)
    # tails of a normal: P(|z| > 3) = 0.0026998
    frac = np.mean(np.abs(z) > 3)
    assert abs(frac - 0.0026998) < 4 * np.sqrt(0.0027 / n)


def test_weight_scale():
    w = W.tensor(1, W.tensor_id(0, W.WG), 256, 512)
    assert abs(w.std() - 0.02) < 4 * 0.02 / np.sqrt(2 * w.size) + 0.02 * 2 ** -8
    np.testing.assert_array_equal(round_bf16(w), w)


def test_bf16_rounding_cases_and_library():
    e = 2.0 ** -8
    x = np.array([1 + e, 1 + 3 * e, 1 + e + 2 ** -30, -(1 + e), 0.0, 3.0])
    np.testing.assert_array_equal(round_bf16(x), [1, 1 + 4 * e, 1 + 2 * e, -1, 0, 3])
    g = np.random.default_rng(0)
    f = (g.standard_normal(100_000) * 10.0 ** g.integers(-6, 6, 100_000)).astype(np.float32)
    lib = torch.from_numpy(f).to(torch.bfloat16).to(torch.float64).numpy()
    np.testing.assert_array_equal(round_bf16(f.astype(np.float64)), lib)
    np.testing.assert_array_equal(from_bits(to_bits(lib)), lib)


# ---------------------------------------------------------------- sublayers
def test_rmsnorm_matches_torch():
    g = np.random.default_rng(1)
    x = g.normal(size=(5, 64)) * 3
    gain = g.normal(size=64)
    ref = F.rms_norm(torch.from_numpy(x), (64,), torch.from_numpy(gain), eps=1e-5).numpy()
    np.testing.assert_allclose(Mo.rmsnorm(x, gain, 1e-5), ref, rtol=1e-12, atol=1e-12)


def test_rope_is_complex_rotation():
    """Rotate-half RoPE equals multiplying (a_i + i b_i) by exp(i P f_i)."""
    g = np.random.default_rng(2)
    hd, n = 16, 7
    x = g.normal(size=(3, n, hd))
    pos = g.integers(0, 5000, size=n)
    f = 10000.0 ** (-2.0 * np.arange(hd // 2) / hd)
    zc = (x[..., :hd // 2] + 1j * x[..., hd // 2:]) * np.exp(1j * pos[:, None] * f[None, :])
    ref = np.concatenate([zc.real, zc.imag], axis=-1)
    np.testing.assert_allclose(Mo.rope(x, pos, 10000.0), ref, rtol=1e-10, atol=1e-10)


def test_rope_invariants():
    g = np.random.default_rng(3)
    q = g.normal(size=(1, 1, 32))
    k = g.normal(size=(1, 1, 32))
    np.testing.assert_allclose(Mo.rope(q, [0], 500000.0), q)
    np.testing.assert_allclose(np.linalg.norm(Mo.rope(q, [123], 5e5)), np.linalg.norm(q))
    d1 = (Mo.rope(q, [40], 5e5) * Mo.rope(k, [17], 5e5)).sum()
    d2 = (Mo.rope(q, [1040], 5e5) * Mo.rope(k, [1017], 5e5)).sum()
    assert d1 == pytest.approx(d2, rel=1e-9)


def test_attention_matches_torch_sdpa():
    g = np.random.default_rng(4)
    n, H, Hkv, hd, L = 5, 8, 2, 16, 37
    T = L + n
    q = g.normal(size=(n, H, hd))
    K = g.normal(size=(Hkv, T, hd))
    V = g.normal(size=(Hkv, T, hd))
    pos = L + np.arange(n)
    got = Mo.attention(q, K, V, pos)
    Kr = torch.from_numpy(K).repeat_interleave(H // Hkv, 0)
    Vr = torch.from_numpy(V).repeat_interleave(H // Hkv, 0)
    mask = torch.from_numpy(np.arange(T)[None, :] <= pos[:, None])
    ref = F.scaled_dot_product_attention(torch.from_numpy(q).transpose(0, 1), Kr, Vr,
                                         attn_mask=mask).transpose(0, 1).numpy()
    np.testing.assert_allclose(got, ref, rtol=1e-10, atol=1e-12)


def test_attention_single_key_returns_value():
    g = np.random.default_rng(5)
    q = g.normal(size=(1, 4, 8))
    K = g.normal(size=(1, 1, 8))
    V = g.normal(size=(1, 1, 8))
    np.testing.assert_allclose(Mo.attention(q, K, V, [0]), np.broadcast_to(V[0, 0], (1, 4, 8)))


def test_silu_matches_torch():
    x = np.linspace(-30, 30, 1001)
    np.testing.assert_allclose(Mo.silu(x), F.silu(torch.from_numpy(x)).numpy(), rtol=1e-13, atol=1e-300)


# ---------------------------------------------------------------- whole pass
def _prefilled(cfg, Wt, B, L, cap, seed, round_kv):
    kv = Mo.KVState(cfg, B, cap)
    toks = np.random.default_rng(seed).integers(0, cfg.vocab, size=(B, L))
    Mo.forward(cfg, Wt, toks, kv, round_kv=round_kv)
    return kv


@pytest.mark.parametrize("round_kv,tol", [(False, 1e-9), (True, 1e-6)])
def test_one_pass_equals_sequential_passes(round_kv, tol):
    cfg = TINY
    Wt = W.Weights(cfg, 77)
    kv1 = _prefilled(cfg, Wt, 2, 9, 32, 1, round_kv)
    kv2 = _prefilled(cfg, Wt, 2, 9, 32, 1, round_kv)
    toks = np.random.default_rng(2).integers(0, cfg.vocab, size=(2, 5))
    one = Mo.forward(cfg, Wt, toks, kv1, round_kv=round_kv)
    seq = np.concatenate([Mo.forward(cfg, Wt, toks[:, j:j + 1], kv2, round_kv=round_kv)
                          for j in range(5)], axis=1)
    np.testing.assert_allclose(one, seq, rtol=tol, atol=tol)
    np.testing.assert_array_equal(kv1.lens, kv2.lens)


def test_rollback_then_reverify_equals_fresh_pass():
    """Verify [t, x1..x4], keep t and x1 (n_accepted = 1), then verify a new
    block: must equal a cache that only ever saw the accepted tokens."""
    cfg = TINY
    Wt = W.Weights(cfg, 78)
    kvA = _prefilled(cfg, Wt, 1, 6, 32, 3, True)
    kvB = _prefilled(cfg, Wt, 1, 6, 32, 3, True)
    block = np.array([[7, 11, 13, 17, 19]])
    Mo.forward(cfg, Wt, block, kvA)
    kvA.lens = Mo.truncate(kvA.lens, [1], gamma=4)
    assert kvA.lens[0] == 6 + 1 + 1
    Mo.forward(cfg, Wt, block[:, :2], kvB)
    nxt = np.array([[23, 29, 31]])
    np.testing.assert_allclose(Mo.forward(cfg, Wt, nxt, kvA), Mo.forward(cfg, Wt, nxt, kvB),
                               rtol=1e-12, atol=1e-12)


def test_without_rollback_the_stale_slots_change_the_result():
    """The invariant above is not vacuous: skipping the rollback changes the
    next pass (the stale drafts are attended)."""
    cfg = TINY
    Wt = W.Weights(cfg, 78)
    kvA = _prefilled(cfg, Wt, 1, 6, 32, 3, True)
    kvB = _prefilled(cfg, Wt, 1, 6, 32, 3, True)
    Mo.forward(cfg, Wt, np.array([[7, 11, 13, 17, 19]]), kvA)
    Mo.forward(cfg, Wt, np.array([[7, 11]]), kvB)
    nxt = np.array([[23, 29, 31]])
    assert not np.allclose(Mo.forward(cfg, Wt, nxt, kvA), Mo.forward(cfg, Wt, nxt, kvB))


def test_truncate_rule():
    np.testing.assert_array_equal(Mo.truncate([10, 10, 10], [0, 2, 4], 4), [6, 8, 10])
    with pytest.raises(ValueError):
        Mo.truncate([10], [5], 4)
    with pytest.raises(ValueError):
        Mo.truncate([2], [0], 4)


def test_forward_rejects_bad_inputs():
    cfg = TINY
    Wt = W.Weights(cfg, 1)
    kv = Mo.KVState(cfg, 1, 4)
    with pytest.raises(ValueError):
        Mo.forward(cfg, Wt, np.array([[1, 2, 3, 4, 5]]), kv)
    with pytest.raises(ValueError):
        Mo.forward(cfg, Wt, np.array([[cfg.vocab]]), kv)


def test_prefix_cache_equals_stored_cache():
    """The streamed cache (prefix rebuilt from the row pool on demand, only
    the written slots kept) gives the stored cache's logits and new cache
    rows, over a pass, a rollback and a second pass, with ragged lengths."""
    from speculative_decoding_verification_pass_gb300 import workloads as wl
    B, n, gamma = 3, 5, 4
    lens = np.array([17, 40, 9])
    Kp, Vp = wl.kv_pool(4, 64, TINY.head_dim)

    def prefix(l, b):
        idx = wl.kv_pool_index(4, l, b, TINY.n_kv_heads, int(lens[b]), 64)
        return from_bits(Kp[idx[0]]), from_bits(Vp[idx[1]])

    Wt = W.Weights(TINY, 3)
    stored = Mo.KVState(TINY, B, 64)
    for l in range(TINY.n_layers):
        for b in range(B):
            K0, V0 = prefix(l, b)
            stored.K[l][b, :, :lens[b]] = K0
            stored.V[l][b, :, :lens[b]] = V0
    stored.lens[:] = lens
    streamed = Mo.PrefixKV(lens, prefix, extra=16)
    t1 = np.random.default_rng(0).integers(0, TINY.vocab, (B, n))
    t2 = np.random.default_rng(1).integers(0, TINY.vocab, (B, n))
    np.testing.assert_array_equal(Mo.forward(TINY, Wt, t1, stored), Mo.forward(TINY, Wt, t1, streamed))
    n_acc = np.array([0, 4, 2])
    stored.lens = Mo.truncate(stored.lens, n_acc, gamma)
    streamed.lens = Mo.truncate(streamed.lens, n_acc, gamma)
    np.testing.assert_array_equal(Mo.forward(TINY, Wt, t2, stored), Mo.forward(TINY, Wt, t2, streamed))
    for l in range(TINY.n_layers):
        for b in range(B):
            K, V = streamed.seq(l, b)
            L = int(streamed.lens[b])
            np.testing.assert_array_equal(K[:, :L], stored.K[l][b, :, :L])
            np.testing.assert_array_equal(V[:, :L], stored.V[l][b, :, :L])
    with pytest.raises(ValueError):             # passes beyond the kept slots
        streamed.lens = streamed.base + 14
        Mo.forward(TINY, Wt, t1, streamed)


def test_bf16_layer_cache_returns_the_generated_values():
    a = W.Weights(TINY, 8, cache_layers="bf16")
    b = W.Weights(TINY, 8, cache_layers=False)
    for k, v in b.layer(1).items():
        np.testing.assert_array_equal(a.layer(1)[k], v)
        np.testing.assert_array_equal(a.layer(1)[k], v)   # from the cache


# ---------------------------------------------------------------- LM head
def test_lm_head_pins():
    """The LM head is hidden @ head^T: equal to torch's fp64 linear; the
    identity head returns the hidden states; a one-hot hidden state picks one
    column of the head; the logits are linear in the head."""
    g = np.random.default_rng(41)
    h = g.normal(size=(5, 64))
    Hd = g.normal(size=(300, 64))
    Hd2 = g.normal(size=(300, 64))
    z = Mo.lm_head(h, Hd)
    assert z.shape == (5, 300)
    ref = torch.nn.functional.linear(torch.from_numpy(h), torch.from_numpy(Hd)).numpy()
    np.testing.assert_allclose(z, ref, rtol=1e-13, atol=1e-12)
    np.testing.assert_allclose(Mo.lm_head(h, np.eye(64)), h, rtol=0, atol=0)
    e3 = np.zeros((1, 64))
    e3[0, 3] = 1.0
    np.testing.assert_allclose(Mo.lm_head(e3, Hd)[0], Hd[:, 3], rtol=0, atol=0)
    np.testing.assert_allclose(Mo.lm_head(h, Hd + Hd2), Mo.lm_head(h, Hd) + Mo.lm_head(h, Hd2), rtol=1e-12, atol=1e-12)
