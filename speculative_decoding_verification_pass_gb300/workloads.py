"""Seeded synthetic inputs shared by the tests, the benchmark and the oracle.

This module holds no arithmetic of the method: it only draws random arrays
(numpy PCG64 from a SeedSequence) of the shapes and distributions the
workloads state.  Anything derived from them by the method (softmax, top-p,
draft sampling, forwards) is computed by the side that consumes them.

Recipes (numbers are the workloads' own):

* ``accept_logits``: draft logits z_q ~ N(0, 2^2) fp32 and target logits
  z_p = z_q + N(0, 0.5^2) for gamma+1 positions.
* ``uniforms``: U[0, 1) fp32 coins and draw variables.
* ``hidden_bf16``: activations ~ N(0, 1) rounded to bf16 (bit patterns).
* ``tokens``: token ids uniform over the vocabulary.
* ``kv_prefix``: cache contents ~ N(0, 1) rounded to bf16 (bit patterns).
* ``context_lengths``: per-sequence lengths uniform in [lo, hi].
* ``kv_pool`` / ``kv_pool_index``: cache rows ~ N(0, 1) in bf16 drawn from a
  seeded pool, for contexts too long to draw row by row.
* ``gauss``: plain N(0, sigma^2) fp32 noise.
"""
from __future__ import annotations

import numpy as np

BASE_SEED = 20261202


def rng(seed: int, *stream: int) -> np.random.Generator:
    """Independent generator for (seed, stream...)."""
    return np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, *stream])))


def f32_to_bf16_bits(x) -> np.ndarray:
    """Round fp32 to bf16 (nearest, ties to even) and return uint16 bits.
    A storage-format conversion for generated inputs."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16).reshape(x.shape)


def bf16_bits_to_f32(b) -> np.ndarray:
    b = np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32)


def accept_logits(seed: int, batch: int, gamma: int, vocab: int,
                  z_std: float = 2.0, noise_std: float = 0.5):
    """(z_q [B][gamma+1][V], z_p [B][gamma+1][V]) fp32."""
    g = rng(seed, 1)
    zq = (z_std * g.standard_normal((batch, gamma + 1, vocab))).astype(np.float32)
    zp = (zq + noise_std * g.standard_normal(zq.shape)).astype(np.float32)
    return zq, zp


def uniforms(seed: int, *shape: int, stream: int = 2) -> np.ndarray:
    return rng(seed, stream).random(shape, dtype=np.float32)


def hidden_bf16(seed: int, rows: int, dim: int, stream: int = 3) -> np.ndarray:
    return f32_to_bf16_bits(rng(seed, stream).standard_normal((rows, dim), dtype=np.float32))


def gauss(seed: int, shape, sigma: float, stream: int = 4) -> np.ndarray:
    return (sigma * rng(seed, stream).standard_normal(shape)).astype(np.float32)


def tokens(seed: int, batch: int, n: int, vocab: int, stream: int = 5) -> np.ndarray:
    return rng(seed, stream).integers(0, vocab, size=(batch, n), dtype=np.int32)


def kv_prefix(seed: int, n_layers: int, batch: int, n_kv_heads: int,
              length: int, head_dim: int, stream: int = 6):
    """(K, V) bf16 bit patterns, each [layers][B][Hkv][length][hd]."""
    g = rng(seed, stream)
    shape = (n_layers, batch, n_kv_heads, length, head_dim)
    K = f32_to_bf16_bits(g.standard_normal(shape, dtype=np.float32))
    V = f32_to_bf16_bits(g.standard_normal(shape, dtype=np.float32))
    return K, V


def kv_pool(seed: int, rows: int, head_dim: int, stream: int = 15):
    """(K, V) pools of cache rows: bf16 bit patterns [rows][hd] ~ N(0, 1).
    Long batched contexts take their cached rows from these pools (see
    kv_pool_index) instead of drawing every row: the contents keep the same
    distribution, and each side can rebuild any (layer, sequence) slice."""
    g = rng(seed, stream)
    K = f32_to_bf16_bits(g.standard_normal((rows, head_dim), dtype=np.float32))
    V = f32_to_bf16_bits(g.standard_normal((rows, head_dim), dtype=np.float32))
    return K, V


def kv_pool_index(seed: int, layer: int, seq: int, n_kv_heads: int, length: int,
                  pool_rows: int, stream: int = 16) -> np.ndarray:
    """Pool rows of the cached keys and values of one (layer, sequence):
    int64 [2][Hkv][length], [0] for K and [1] for V, uniform over the pool."""
    return rng(seed, stream, layer, seq).integers(0, pool_rows, size=(2, n_kv_heads, length))


def context_lengths(seed: int, batch: int, lo: int, hi: int, stream: int = 7) -> np.ndarray:
    return rng(seed, stream).integers(lo, hi + 1, size=batch, dtype=np.int32)


def random_tree(seed: int, n: int, stream: int = 10) -> list:
    """Parent pointers of a random n-node draft tree: node 0 is the root
    (parent -1), node i > 0 hangs under a uniformly chosen earlier node."""
    g = rng(seed, stream)
    return [-1] + [int(g.integers(0, i)) for i in range(1, n)]


def allowed_sets(seed: int, rows: int, vocab: int, frac: float, stream: int = 14) -> np.ndarray:
    """A random allowed-token set per row (bool [rows][vocab]), each token
    allowed with probability frac and at least one per row."""
    a = rng(seed, stream).random((rows, vocab)) < frac
    a[~a.any(axis=1), 0] = True
    return a


def pack_allowed(a) -> np.ndarray:
    """Bool [rows][vocab] -> uint32 [rows][ceil(vocab / 32)], token x at bit
    x % 32 of word x / 32."""
    a = np.asarray(a, dtype=bool)
    rows, V = a.shape
    W = (V + 31) // 32
    pad = np.zeros((rows, W * 32), dtype=bool)
    pad[:, :V] = a
    bits = pad.reshape(rows, W, 32).astype(np.uint64) << np.arange(32, dtype=np.uint64)
    return bits.sum(axis=2).astype(np.uint32)
