"""fp64 oracle of the target verification forward and the KV rollback rule.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

What the pages fix:

* One target pass scores the gamma drafted positions plus the next-token slot
  (lattice-ai-eng "Speculative decoding" notes, the reference loop: the target
  is run once on the current sequence and its last k+1 logits rows are kept;
  pigeon guide *How it works* step 2: "gamma + 1 positions" in one pass).
  So the input of a pass is [t_last, x_1 .. x_gamma] where t_last is the
  previous pass's emitted token, not yet in the cache, and logits row j
  predicts the token after input j.
* The cache holds bf16 keys/values and a valid length; rollback moves that
  length and clears nothing ("Build a Speculative Decoding Engine ...",
  *KV Cache Management for Dual Models* and *Rollback Protocol*).

The decoder itself is the "Llama-style" model the workloads name; the pages
say nothing of its layers, so these readings are used:
RMSNorm with eps 1e-5 and unit gains; rotate-half RoPE over pairs
(i, i + hd/2) with frequency theta^(-2i/hd), theta = 500000, positions from 0;
grouped-query attention with group n_heads / n_kv_heads and scale
1/sqrt(hd), causal (a query at position P sees keys 0..P); SwiGLU MLP
silu(x W_g^T) * (x W_u^T) then W_d; no biases; untied LM head.

Everything is fp64 except that keys and values are rounded to bf16 when
stored (the cache's defined format); ``round_kv=False`` stores them in fp64.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np

from .bf16 import round_bf16
from . import weights as wts


@dataclass(frozen=True)
class Config:
    n_layers: int
    d_model: int
    n_heads: int
    n_kv_heads: int
    d_ffn: int
    vocab: int
    rms_eps: float = 1e-5
    rope_theta: float = 500000.0

    @property
    def head_dim(self) -> int:
        return self.d_model // self.n_heads

    @property
    def group(self) -> int:
        return self.n_heads // self.n_kv_heads


def rmsnorm(x, g, eps: float) -> np.ndarray:
    """x / sqrt(mean(x^2) + eps) * g over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(g, dtype=np.float64)


def rope(x, positions, theta: float) -> np.ndarray:
    """Rotate-half RoPE.  x [..., n, hd] with positions [n]; the pair
    (i, i + hd/2) is rotated by positions * theta^(-2i/hd)."""
    x = np.asarray(x, dtype=np.float64)
    hd = x.shape[-1]
    half = hd // 2
    freq = theta ** (-2.0 * np.arange(half) / hd)
    ang = np.asarray(positions, dtype=np.float64)[:, None] * freq[None, :]
    c, s = np.cos(ang), np.sin(ang)
    a, b = x[..., :half], x[..., half:]
    return np.concatenate([a * c - b * s, a * s + b * c], axis=-1)


def attention(q, K, V, q_pos) -> np.ndarray:
    """Causal GQA attention for one sequence.

    q [n][H][hd] (already rotated), K/V [Hkv][T][hd] (cache incl. the new
    entries), q_pos [n] absolute positions; query j of head h reads keys
    0..q_pos[j] of kv head h // (H / Hkv)."""
    n, H, hd = q.shape
    Hkv = K.shape[0]
    G = H // Hkv
    o = np.zeros((n, H, hd))
    scale = 1.0 / np.sqrt(hd)
    for j in range(n):
        P = int(q_pos[j])
        for h in range(H):
            kh = h // G
            s = K[kh, :P + 1] @ q[j, h] * scale
            a = np.exp(s - s.max())
            a /= a.sum()
            o[j, h] = a @ V[kh, :P + 1]
    return o


def silu(x):
    return x / (1.0 + np.exp(-x))


def swiglu(x, wg, wu, wd) -> np.ndarray:
    """(silu(x W_g^T) * (x W_u^T)) W_d^T."""
    x = np.asarray(x, dtype=np.float64)
    a = silu(x @ np.asarray(wg, np.float64).T) * (x @ np.asarray(wu, np.float64).T)
    return a @ np.asarray(wd, np.float64).T


class KVState:
    """The oracle's own cache: K[l], V[l] of shape [B][Hkv][cap][hd] (fp64
    arrays holding bf16 values unless round_kv is off) and lengths [B]."""

    def __init__(self, cfg: Config, batch: int, capacity: int):
        shape = (batch, cfg.n_kv_heads, capacity, cfg.head_dim)
        self.K = [np.zeros(shape) for _ in range(cfg.n_layers)]
        self.V = [np.zeros(shape) for _ in range(cfg.n_layers)]
        self.lens = np.zeros(batch, dtype=np.int64)
        self.capacity = capacity

    def load_prefix(self, K_prefix, V_prefix, lens):
        """Install given cache contents: K_prefix[l] [B][Hkv][L][hd]."""
        for l in range(len(self.K)):
            L = K_prefix[l].shape[2]
            self.K[l][:, :, :L] = K_prefix[l]
            self.V[l][:, :, :L] = V_prefix[l]
        self.lens[:] = lens

    def seq(self, l: int, b: int):
        """Layer l's keys and values of sequence b, [Hkv][cap][hd] (views)."""
        return self.K[l][b], self.V[l][b]

    def keep(self, l: int, b: int, K, V, start: int, n: int) -> None:
        """Slots start..start+n-1 were written into the views: nothing to do."""


class PrefixKV:
    """A cache for long batched contexts whose full fp64 copy would not fit
    in host memory.  The cached prefix of each (layer, sequence) is not
    stored: ``prefix(l, b)`` returns it, [Hkv][lens[b]][hd] fp64, whenever
    a pass needs it; only the slots that passes write after the prefix
    (at most ``extra`` per sequence) are kept.  The same cache contents as a
    KVState loaded with the same prefix, in another storage."""

    def __init__(self, lens, prefix, extra: int = 64):
        self.base = np.array(lens, dtype=np.int64)
        self.lens = self.base.copy()
        self.capacity = self.base + extra
        self.prefix = prefix
        self.extra = extra
        self.new = {}

    def seq(self, l: int, b: int):
        K0, V0 = self.prefix(l, b)
        Hkv, L, hd = K0.shape
        if L != self.base[b]:
            raise ValueError("prefix length differs from the cached length")
        K = np.zeros((Hkv, L + self.extra, hd))
        V = np.zeros_like(K)
        K[:, :L], V[:, :L] = K0, V0
        if (l, b) in self.new:
            K[:, L:], V[:, L:] = self.new[(l, b)]
        return K, V

    def keep(self, l: int, b: int, K, V, start: int, n: int) -> None:
        L = int(self.base[b])
        if start < L:
            raise ValueError("a pass may not rewrite the stored prefix")
        self.new[(l, b)] = (K[:, L:].copy(), V[:, L:].copy())


def forward(cfg: Config, W: "wts.Weights", tokens, kv,
            round_kv: bool = True) -> np.ndarray:
    """One verification pass: tokens [B][n] -> logits [B][n][V] (fp64).

    Writes keys/values of the n new positions at slots len_b .. len_b+n-1 and
    advances len_b by n (the rollback afterwards is ``truncate``).  ``kv`` is
    a KVState or a PrefixKV."""
    toks = np.asarray(tokens, dtype=np.int64)
    B, n = toks.shape
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
        x = rmsnorm(h, g, cfg.rms_eps)
        q = (x @ w[wts.WQ].astype(np.float64).T).reshape(B, n, H, hd)
        k = (x @ w[wts.WK].astype(np.float64).T).reshape(B, n, Hkv, hd)
        v = (x @ w[wts.WV].astype(np.float64).T).reshape(B, n, Hkv, hd)
        o = np.zeros((B, n, H, hd))
        for b in range(B):
            pos = L0[b] + np.arange(n)
            qb = rope(q[b].transpose(1, 0, 2), pos, cfg.rope_theta).transpose(1, 0, 2)
            kb = rope(k[b].transpose(1, 0, 2), pos, cfg.rope_theta)       # [Hkv][n][hd]
            Kb, Vb = kv.seq(l, b)
            Kb[:, pos[0]:pos[0] + n] = store(kb)
            Vb[:, pos[0]:pos[0] + n] = store(v[b].transpose(1, 0, 2))
            kv.keep(l, b, Kb, Vb, int(pos[0]), n)
            o[b] = attention(qb, Kb, Vb, pos)
        h = h + o.reshape(B, n, H * hd) @ w[wts.WO].astype(np.float64).T
        x = rmsnorm(h, g, cfg.rms_eps)
        h = h + swiglu(x, w[wts.WG], w[wts.WU], w[wts.WD])
    x = rmsnorm(h, g, cfg.rms_eps)
    kv.lens += n
    return x @ W.head().astype(np.float64).T


def lm_head(hidden, head) -> np.ndarray:
    """Logits of given hidden states: hidden [M][d] @ head[V][d]^T (the
    LM-head-only workload feeds activations straight to the head)."""
    return np.asarray(hidden, np.float64) @ np.asarray(head, np.float64).T


def truncate(lens, n_accepted, gamma: int) -> np.ndarray:
    """KV rollback after a pass that appended gamma+1 slots.

    The input t_last and the accepted drafts stay; the rejected drafts'
    slots are dropped: new length = (len_before_pass) + 1 + n_accepted, i.e.
    len -= gamma - n_accepted.  The rollback protocol's "N + (i - 1)" for a
    rejection at the 1-based draft i counts the same slots.  Pointer update
    only; slot contents are left as they are."""
    lens = np.asarray(lens, dtype=np.int64)
    n_acc = np.asarray(n_accepted, dtype=np.int64)
    if np.any(n_acc < 0) or np.any(n_acc > gamma):
        raise ValueError("n_accepted out of range")
    if np.any(lens < gamma - n_acc):
        raise ValueError("length below the rollback")
    return lens - (gamma - n_acc)
