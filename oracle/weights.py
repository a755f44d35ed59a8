"""Seeded synthetic decoder weights, generated on the oracle side.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).

The weights are random numbers the method draws from a seed, so each side
implements the same counter-based generator from its published definition:

* Philox4x64-10 (Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as
  easy as 1, 2, 3", SC 2011).  numpy's ``Philox`` bit generator is that
  generator; it is pinned here by the paper's known-answer vectors (tests).
  Block i of logical tensor t uses counter (i + 1, t, 0, 0) and key
  (seed, 0); numpy increments the counter before each block, so a state with
  counter (i, t, 0, 0) emits block i.
* Box-Muller (1958) in fp64: each pair of 64-bit outputs (a, b) gives
  u = ((a >> 11) + 0.5) * 2^-53, v = ((b >> 11) + 0.5) * 2^-53 and the two
  normals sqrt(-2 ln u) * cos(2 pi v), sqrt(-2 ln u) * sin(2 pi v).  Element
  4i + {0,1} takes the first pair of block i, 4i + {2,3} the second.
* A weight is the bf16 rounding (to nearest, ties even) of 0.02 * normal:
  matrices ~ N(0, 0.02^2) as the decoder workloads state; RMSNorm gains are
  1.0 (a reading: gains drawn at std 0.02 would shrink every normalised
  activation fifty-fold).

Logical tensor ids: 0 embedding [V][d]; 1 LM head [V][d]; layer l uses
2 + 7l + k for k = 0 W_q [H*hd][d], 1 W_k [Hkv*hd][d], 2 W_v [Hkv*hd][d],
3 W_o [d][H*hd], 4 W_gate [ffn][d], 5 W_up [ffn][d], 6 W_down [d][ffn].
Matrices are [out][in], row-major.
"""
from __future__ import annotations

import atexit
import concurrent.futures as cf
import multiprocessing as mp
import os

import numpy as np

from .bf16 import round_bf16

SCALE = 0.02
TWO_M53 = 2.0 ** -53

EMBED, HEAD = 0, 1
WQ, WK, WV, WO, WG, WU, WD = range(7)
NAMES = ("wq", "wk", "wv", "wo", "wg", "wu", "wd")


def tensor_id(layer: int, k: int) -> int:
    return 2 + 7 * layer + k


def philox_blocks(seed: int, tid: int, first_block: int, n_blocks: int) -> np.ndarray:
    """Raw Philox4x64-10 output of blocks first_block .. first_block+n-1."""
    bg = np.random.Philox(counter=[first_block, tid, 0, 0], key=[seed, 0])
    return bg.random_raw(4 * n_blocks)


def normals(seed: int, tid: int, start: int, count: int) -> np.ndarray:
    """fp64 standard normals of elements [start, start+count) of tensor tid."""
    if count <= 0:
        return np.zeros(0)
    b0 = start // 4
    b1 = (start + count + 3) // 4
    raw = philox_blocks(seed, tid, b0, b1 - b0).reshape(-1, 2, 2)
    u = ((raw[:, :, 0] >> np.uint64(11)).astype(np.float64) + 0.5) * TWO_M53
    v = ((raw[:, :, 1] >> np.uint64(11)).astype(np.float64) + 0.5) * TWO_M53
    r = np.sqrt(-2.0 * np.log(u))
    th = 2.0 * np.pi * v
    z = np.stack([r * np.cos(th), r * np.sin(th)], axis=-1).reshape(-1)
    off = start - 4 * b0
    return z[off:off + count]


def _chunk(args):
    seed, tid, start, count = args
    return round_bf16(SCALE * normals(seed, tid, start, count)).astype(np.float32)


_POOL = None


def _pool():
    """Worker processes for large tensors (spawned, never forked, so they are
    safe to start after CUDA has been initialised in the parent)."""
    global _POOL
    if _POOL is None:
        n = int(os.environ.get("ORACLE_WORKERS", min(16, os.cpu_count() or 1)))
        if n > 1:
            _POOL = cf.ProcessPoolExecutor(n, mp_context=mp.get_context("spawn"))
            atexit.register(_POOL.shutdown, wait=True)
        else:
            _POOL = False
    return _POOL


def tensor(seed: int, tid: int, rows: int, cols: int,
           row0: int = 0, nrows: int | None = None,
           chunk: int = 1 << 22) -> np.ndarray:
    """Rows [row0, row0+nrows) of a [rows][cols] weight matrix as fp32
    arrays holding bf16-exact values (element order is independent of how
    the range is split into chunks)."""
    if nrows is None:
        nrows = rows - row0
    out = np.empty(nrows * cols, dtype=np.float32)
    start = row0 * cols
    n = nrows * cols
    jobs = [(seed, tid, start + c0, min(n, c0 + chunk) - c0) for c0 in range(0, n, chunk)]
    pool = _pool() if len(jobs) > 2 else False
    parts = None
    if pool:
        try:
            parts = list(pool.map(_chunk, jobs))
        except cf.process.BrokenProcessPool:     # e.g. a parent without a main file
            global _POOL
            _POOL = False
    if parts is None:
        parts = map(_chunk, jobs)
    for (_, _, s0, cnt), part in zip(jobs, parts):
        out[s0 - start:s0 - start + cnt] = part
    return out.reshape(nrows, cols)


def layer_shapes(cfg):
    """[out][in] shapes of the seven matrices of one layer."""
    hd = cfg.head_dim
    d = cfg.d_model
    return {
        WQ: (cfg.n_heads * hd, d), WK: (cfg.n_kv_heads * hd, d),
        WV: (cfg.n_kv_heads * hd, d), WO: (d, cfg.n_heads * hd),
        WG: (cfg.d_ffn, d), WU: (cfg.d_ffn, d), WD: (d, cfg.d_ffn),
    }


def _bits(a) -> np.ndarray:
    """uint16 bit patterns of fp32 arrays holding bf16-exact values."""
    return (np.ascontiguousarray(a, dtype=np.float32).view(np.uint32) >> np.uint32(16)).astype(np.uint16)


def _unbits(b) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


class Weights:
    """Lazily generated weights of one seeded model (fp32 holding bf16).

    cache_layers: True keeps generated layers as fp32, "bf16" keeps them as
    bf16 bit patterns (half the memory; the values are bf16 already), False
    regenerates a layer whenever it is asked for."""

    def __init__(self, cfg, seed: int, cache_layers=True):
        self.cfg, self.seed, self.cache = cfg, seed, cache_layers
        self._layers = {}
        self._head = None

    def layer(self, l: int) -> dict:
        if l in self._layers:
            w = self._layers[l]
            return {k: _unbits(v) for k, v in w.items()} if self.cache == "bf16" else w
        w = {k: tensor(self.seed, tensor_id(l, k), *shape)
             for k, shape in layer_shapes(self.cfg).items()}
        if self.cache == "bf16":
            self._layers[l] = {k: _bits(v) for k, v in w.items()}
        elif self.cache:
            self._layers[l] = w
        return w

    def embed_rows(self, toks) -> np.ndarray:
        d = self.cfg.d_model
        toks = np.asarray(toks).reshape(-1)
        out = np.empty((toks.size, d), dtype=np.float32)
        for i, t in enumerate(toks):
            out[i] = tensor(self.seed, EMBED, self.cfg.vocab, d, int(t), 1)[0]
        return out

    def head(self) -> np.ndarray:
        if self._head is None:
            self._head = tensor(self.seed, HEAD, self.cfg.vocab, self.cfg.d_model)
        return self._head

    def norm_gain(self) -> np.ndarray:
        return np.ones(self.cfg.d_model)
