"""ctypes binding of the C ABI in ``include/spec_verify.h``.

Argument marshalling only: every step of the verification pass runs in the
CUDA library.  PyTorch supplies device memory (tensors) and streams.  The
functions named ``spec_*`` mirror the C entry points one to one; the small
classes below (``Model``, ``KVCache``, ``Workspace``) own the torch buffers
those calls need.  Loading fails loudly when the library has not been built.
"""
from __future__ import annotations

import ctypes
import os
from dataclasses import dataclass

import numpy as np
import torch

from . import _build

SPEC_OK, SPEC_EINVAL, SPEC_ESIZE, SPEC_ECUDA, SPEC_EDEVICE, SPEC_ETIMEOUT, SPEC_ENOTSUP = (
    0, -1, -2, -3, -4, -5, -6)
DEV_BAD_TOKEN, DEV_KV_OVERFLOW, DEV_Q_ZERO, DEV_TIMEOUT, DEV_BAD_NACC, DEV_BAD_TREE = (
    0x1, 0x2, 0x4, 0x8, 0x10, 0x20)
DEV_EMPTY_MASK = 0x40
DEV_BAD_PAGE = 0x80


class SpecError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        msg = f"{where}: {lib().spec_status_string(status).decode()} ({status})"
        if status == SPEC_ECUDA:
            msg += ": " + lib().spec_last_cuda_error().decode()
        super().__init__(msg)


class spec_model_config(ctypes.Structure):
    _fields_ = [("n_layers", ctypes.c_int), ("d_model", ctypes.c_int), ("n_heads", ctypes.c_int),
                ("n_kv_heads", ctypes.c_int), ("d_ffn", ctypes.c_int), ("vocab", ctypes.c_int),
                ("rms_eps", ctypes.c_float), ("rope_theta", ctypes.c_float)]


class spec_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("len", ctypes.c_void_p),
                ("batch", ctypes.c_int), ("capacity", ctypes.c_int)]


class spec_paged_kv_cache(ctypes.Structure):
    _fields_ = [("k", ctypes.c_void_p), ("v", ctypes.c_void_p), ("len", ctypes.c_void_p),
                ("table", ctypes.c_void_p), ("batch", ctypes.c_int), ("n_pages", ctypes.c_int),
                ("max_pages", ctypes.c_int)]


PAGE_SLOTS = 64
_LIB = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t
_F = ctypes.c_float

_SIGS = {
    "spec_status_string": (ctypes.c_char_p, [_I]),
    "spec_last_cuda_error": (ctypes.c_char_p, []),
    "spec_model_weight_bytes": (_SZ, [ctypes.POINTER(spec_model_config)]),
    "spec_model_create": (_I, [ctypes.POINTER(spec_model_config), ctypes.c_uint64, _P, _SZ, _P,
                               ctypes.POINTER(_P)]),
    "spec_model_destroy": (_I, [_P]),
    "spec_model_tensor": (_I, [_P, _I, _I, ctypes.POINTER(_P), ctypes.POINTER(ctypes.c_int64),
                               ctypes.POINTER(_I), ctypes.POINTER(_I)]),
    "spec_kv_bytes": (_SZ, [ctypes.POINTER(spec_model_config), _I, _I]),
    "spec_workspace_bytes": (_SZ, [ctypes.POINTER(spec_model_config), _I, _I, _I]),
    "spec_verify_forward": (_I, [_P, _P, _I, _I, ctypes.POINTER(spec_kv_cache), _P, _P, _SZ, _P]),
    "spec_lm_head": (_I, [_P, _P, _I, _P, _P, _SZ, _P]),
    "spec_lm_head_noalloc": (_I, [_P, _P, _I, _P, _P]),
    "spec_accept_workspace_bytes": (_SZ, [_I, _I, _I]),
    "spec_accept": (_I, [_P, _P, _P, _P, _I, _I, _I, _F, _F, _P, _P, _P, _SZ, _P]),
    "spec_draft_sample": (_I, [_P, _I, _I, _F, _F, _P, _P, _P, _P, _SZ, _P]),
    "spec_kv_truncate": (_I, [ctypes.POINTER(spec_kv_cache), _P, _I, _P, _P]),
    "spec_mask_logits": (_I, [_P, _P, _I, _I, _P, _P]),
    "spec_paged_kv_bytes": (_SZ, [ctypes.POINTER(spec_model_config), _I]),
    "spec_verify_forward_paged": (_I, [_P, _P, _I, _I, ctypes.POINTER(spec_paged_kv_cache), _P, _P,
                                       _SZ, _P]),
    "spec_paged_kv_truncate": (_I, [ctypes.POINTER(spec_paged_kv_cache), _P, _I, _P, _P]),
    "spec_page_pool_create": (_I, [_I, _I, _I, ctypes.POINTER(_P)]),
    "spec_page_pool_destroy": (_I, [_P]),
    "spec_page_pool_reserve": (_I, [_P, _I, _I]),
    "spec_page_pool_release": (_I, [_P, _I, _I]),
    "spec_page_pool_table": (ctypes.POINTER(ctypes.c_int32), [_P]),
    "spec_page_pool_free_pages": (_I, [_P]),
    "spec_gamma_ctl_create": (_I, [_I, _I, _I, _I, _I, _I, ctypes.c_double, ctypes.c_double,
                                   ctypes.c_double, ctypes.POINTER(_P)]),
    "spec_gamma_ctl_destroy": (_I, [_P]),
    "spec_gamma_ctl_reset": (_I, [_P, _I]),
    "spec_gamma_ctl_step": (_I, [_P, _I, _P, _P, _P, _P]),
    "spec_gamma_ctl_state": (_I, [_P, _I, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int32),
                                  ctypes.POINTER(ctypes.c_int32)]),
    "spec_gamma_optimal": (_I, [ctypes.c_double, _I, _I, ctypes.c_double, ctypes.c_double,
                                ctypes.POINTER(ctypes.c_int32)]),
    "spec_tree_masks": (_I, [ctypes.POINTER(ctypes.c_int32), _I, ctypes.POINTER(ctypes.c_uint64),
                             ctypes.POINTER(ctypes.c_int32)]),
    "spec_verify_forward_tree": (_I, [_P, _P, _P, _P, _I, _I, ctypes.POINTER(spec_kv_cache), _P, _P,
                                      _SZ, _P]),
    "spec_tree_accept_workspace_bytes": (_SZ, [_I, _I]),
    "spec_tree_accept": (_I, [_P, _P, _P, _P, _P, _I, _I, _I, _F, _F, _P, _P, _P, _P, _SZ, _P]),
    "spec_kv_tree_commit": (_I, [_P, ctypes.POINTER(spec_kv_cache), _P, _P, _I, _P, _P]),
    "spec_device_status": (_I, [_P, _P, ctypes.POINTER(ctypes.c_int32)]),
    "spec_wait_selftest": (_I, [_P, ctypes.c_uint32, ctypes.c_double, _P, _SZ, _P]),
    "spec_timing_enable": (_I, [_P, _I]),
    "spec_timing_read": (_I, [_P, ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64),
                              ctypes.POINTER(ctypes.c_double)]),
}

EXPORTED = tuple(_SIGS)


def lib_path() -> str:
    return _build.LIB


def lib():
    """The loaded library (raises if it has not been built)."""
    global _LIB
    if _LIB is None:
        if not os.path.exists(_build.LIB):
            raise RuntimeError(f"CUDA library not built: {_build.LIB} is missing "
                               "(run __graft_entry__.build())")
        L = ctypes.CDLL(_build.LIB)
        for name, (res, args) in _SIGS.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _LIB = L
    return _LIB


def _check(status: int, where: str):
    if status != SPEC_OK:
        raise SpecError(status, where)


def _ptr(t) -> int | None:
    if t is None:
        return None
    if isinstance(t, int):
        return t
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return t.data_ptr()


def _stream(stream) -> int | None:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


# ----------------------------------------------------------------- configs
@dataclass(frozen=True)
class ModelConfig:
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

    def c(self) -> spec_model_config:
        return spec_model_config(self.n_layers, self.d_model, self.n_heads, self.n_kv_heads,
                                 self.d_ffn, self.vocab, self.rms_eps, self.rope_theta)


LLAMA_8B = ModelConfig(32, 4096, 32, 8, 14336, 128256)
LLAMA_1B = ModelConfig(16, 2048, 32, 8, 8192, 32000)


# ------------------------------------------------------------ raw entry points
def spec_model_weight_bytes(cfg: ModelConfig) -> int:
    return int(lib().spec_model_weight_bytes(ctypes.byref(cfg.c())))


def spec_model_create(cfg: ModelConfig, seed: int, weights: torch.Tensor, stream=None) -> int:
    h = _P()
    _check(lib().spec_model_create(ctypes.byref(cfg.c()), ctypes.c_uint64(seed), _ptr(weights),
                                   weights.numel() * weights.element_size(), _stream(stream),
                                   ctypes.byref(h)), "spec_model_create")
    return h.value


def spec_model_destroy(handle: int):
    _check(lib().spec_model_destroy(handle), "spec_model_destroy")


def spec_model_tensor(handle: int, layer: int, which: int):
    p = _P()
    shape = (ctypes.c_int64 * 2)()
    br, rs = _I(), _I()
    _check(lib().spec_model_tensor(handle, layer, which, ctypes.byref(p), shape, ctypes.byref(br),
                                   ctypes.byref(rs)), "spec_model_tensor")
    return p.value, (shape[0], shape[1]), br.value, rs.value


def spec_kv_bytes(cfg: ModelConfig, batch: int, capacity: int) -> int:
    return int(lib().spec_kv_bytes(ctypes.byref(cfg.c()), batch, capacity))


def spec_workspace_bytes(cfg: ModelConfig, batch: int, gamma: int, capacity: int) -> int:
    return int(lib().spec_workspace_bytes(ctypes.byref(cfg.c()), batch, gamma, capacity))


def spec_verify_forward(handle: int, tokens, batch: int, gamma: int, kv: "KVCache", logits, ws,
                        stream=None):
    _check(lib().spec_verify_forward(handle, _ptr(tokens), batch, gamma, ctypes.byref(kv.c()),
                                     _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)),
           "spec_verify_forward")


def spec_lm_head(handle: int, hidden, rows: int, logits, ws, stream=None):
    _check(lib().spec_lm_head(handle, _ptr(hidden), rows, _ptr(logits), _ptr(ws), ws.numel(),
                              _stream(stream)), "spec_lm_head")


def spec_lm_head_noalloc(handle: int, hidden, rows: int, logits, stream=None):
    """LM head with the library's own scratch (no workspace argument)."""
    _check(lib().spec_lm_head_noalloc(handle, _ptr(hidden), rows, _ptr(logits), _stream(stream)),
           "spec_lm_head_noalloc")


def spec_accept_workspace_bytes(batch: int, gamma: int, vocab: int) -> int:
    return int(lib().spec_accept_workspace_bytes(batch, gamma, vocab))


def spec_accept(target_logits, draft_probs, draft_tokens, uniforms, batch: int, gamma: int,
                vocab: int, temperature: float, top_p: float, out_tokens, n_accepted, ws,
                stream=None):
    _check(lib().spec_accept(_ptr(target_logits), _ptr(draft_probs), _ptr(draft_tokens),
                             _ptr(uniforms), batch, gamma, vocab, temperature, top_p,
                             _ptr(out_tokens), _ptr(n_accepted), _ptr(ws), ws.numel(),
                             _stream(stream)), "spec_accept")


def spec_draft_sample(logits, rows: int, vocab: int, temperature: float, top_p: float, uniforms,
                      probs, tokens, ws, stream=None):
    _check(lib().spec_draft_sample(_ptr(logits), rows, vocab, temperature, top_p, _ptr(uniforms),
                                   _ptr(probs), _ptr(tokens), _ptr(ws), ws.numel(),
                                   _stream(stream)), "spec_draft_sample")


def spec_kv_truncate(kv: "KVCache", n_accepted, gamma: int, ws, stream=None):
    _check(lib().spec_kv_truncate(ctypes.byref(kv.c()), _ptr(n_accepted), gamma, _ptr(ws),
                                  _stream(stream)), "spec_kv_truncate")


def spec_mask_logits(logits, allowed, rows: int, vocab: int, ws, stream=None):
    """logits[r][x] = -inf where bit x of row r's packed mask is clear (in place)."""
    _check(lib().spec_mask_logits(_ptr(logits), _ptr(allowed), rows, vocab, _ptr(ws), _stream(stream)),
           "spec_mask_logits")


class PagedKVCache:
    """Paged target cache: k, v bf16 [layers][n_pages][Hkv][64][hd], len int32
    [B], the device page table int32 [B][max_pages], and a host page pool
    (free list + host table) that `sync()` copies to the device."""

    def __init__(self, cfg: ModelConfig, batch: int, n_pages: int, max_pages: int, device="cuda"):
        self.cfg, self.batch, self.n_pages, self.max_pages = cfg, batch, n_pages, max_pages
        shape = (cfg.n_layers, n_pages, cfg.n_kv_heads, PAGE_SLOTS, cfg.head_dim)
        self.k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        assert self.k.numel() * 2 == int(lib().spec_paged_kv_bytes(ctypes.byref(cfg.c()), n_pages))
        self.len = torch.zeros(batch, dtype=torch.int32, device=device)
        self.table = torch.full((batch, max_pages), -1, dtype=torch.int32, device=device)
        h = ctypes.c_void_p()
        _check(lib().spec_page_pool_create(n_pages, batch, max_pages, ctypes.byref(h)),
               "spec_page_pool_create")
        self.pool = h.value

    @property
    def capacity(self) -> int:
        return self.max_pages * PAGE_SLOTS

    def c(self) -> spec_paged_kv_cache:
        return spec_paged_kv_cache(self.k.data_ptr(), self.v.data_ptr(), self.len.data_ptr(),
                                   self.table.data_ptr(), self.batch, self.n_pages, self.max_pages)

    def reserve(self, b: int, slots: int):
        _check(lib().spec_page_pool_reserve(self.pool, b, slots), "spec_page_pool_reserve")

    def release(self, b: int, slots: int):
        _check(lib().spec_page_pool_release(self.pool, b, slots), "spec_page_pool_release")

    def host_table(self) -> np.ndarray:
        ptr = lib().spec_page_pool_table(self.pool)
        return np.ctypeslib.as_array(ptr, shape=(self.batch * self.max_pages,)).reshape(
            self.batch, self.max_pages).copy()

    def free_pages(self) -> int:
        return int(lib().spec_page_pool_free_pages(self.pool))

    def sync(self):
        """Copy the host page table to the device table."""
        self.table.copy_(torch.from_numpy(self.host_table()))

    def close(self):
        if self.pool:
            lib().spec_page_pool_destroy(self.pool)
            self.pool = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spec_verify_forward_paged(handle: int, tokens, batch: int, gamma: int, kv: "PagedKVCache", logits,
                              ws, stream=None):
    _check(lib().spec_verify_forward_paged(handle, _ptr(tokens), batch, gamma, ctypes.byref(kv.c()),
                                           _ptr(logits), _ptr(ws), ws.numel(), _stream(stream)),
           "spec_verify_forward_paged")


def spec_paged_kv_truncate(kv: "PagedKVCache", n_accepted, gamma: int, ws, stream=None):
    _check(lib().spec_paged_kv_truncate(ctypes.byref(kv.c()), _ptr(n_accepted), gamma, _ptr(ws),
                                        _stream(stream)), "spec_paged_kv_truncate")


class GammaController:
    """Host-side speculation-depth controller (spec_gamma_ctl_*): one rolling
    acceptance window per slot, the depth maximising expected tokens/ms."""

    def __init__(self, slots: int, gamma_min: int = 2, gamma_max: int = 8, gamma_init: int = 4,
                 window: int = 20, min_records: int = 5, draft_ms_per_token: float = 2.0,
                 target_ms_per_pass: float = 20.0, alpha_prior: float = 0.80):
        h = ctypes.c_void_p()
        _check(lib().spec_gamma_ctl_create(slots, gamma_min, gamma_max, gamma_init, window,
                                           min_records, draft_ms_per_token, target_ms_per_pass,
                                           alpha_prior, ctypes.byref(h)), "spec_gamma_ctl_create")
        self.handle = h.value
        self.slots = slots

    def step(self, slots, gamma_used, n_accepted) -> list:
        n = len(slots)
        arr = lambda v: (ctypes.c_int32 * max(n, 1))(*[int(x) for x in v])
        s, g, a = arr(slots), arr(gamma_used), arr(n_accepted)
        out = (ctypes.c_int32 * max(n, 1))()
        _check(lib().spec_gamma_ctl_step(self.handle, n, s, g, a, out), "spec_gamma_ctl_step")
        return list(out)[:n]

    def state(self, slot: int):
        al, g, r = ctypes.c_double(), ctypes.c_int32(), ctypes.c_int32()
        _check(lib().spec_gamma_ctl_state(self.handle, slot, ctypes.byref(al), ctypes.byref(g),
                                          ctypes.byref(r)), "spec_gamma_ctl_state")
        return al.value, g.value, r.value

    def reset(self, slot: int):
        _check(lib().spec_gamma_ctl_reset(self.handle, slot), "spec_gamma_ctl_reset")

    def close(self):
        if self.handle:
            lib().spec_gamma_ctl_destroy(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def spec_gamma_optimal(alpha: float, gamma_min: int, gamma_max: int, draft_ms_per_token: float,
                       target_ms_per_pass: float) -> int:
    out = ctypes.c_int32()
    _check(lib().spec_gamma_optimal(alpha, gamma_min, gamma_max, draft_ms_per_token,
                                    target_ms_per_pass, ctypes.byref(out)), "spec_gamma_optimal")
    return out.value


def spec_tree_masks(parents) -> tuple[list, list]:
    """(ancestor masks, depths) of a tree given by parent pointers (host only)."""
    n = len(parents)
    par = (ctypes.c_int32 * max(n, 1))(*[int(x) for x in parents])
    anc = (ctypes.c_uint64 * max(n, 1))()
    depth = (ctypes.c_int32 * max(n, 1))()
    _check(lib().spec_tree_masks(par, n, anc, depth), "spec_tree_masks")
    return list(anc)[:n], list(depth)[:n]


def spec_verify_forward_tree(handle: int, tokens, anc, depth, batch: int, n_nodes: int,
                             kv: "KVCache", logits, ws, stream=None):
    _check(lib().spec_verify_forward_tree(handle, _ptr(tokens), _ptr(anc), _ptr(depth), batch,
                                          n_nodes, ctypes.byref(kv.c()), _ptr(logits), _ptr(ws),
                                          ws.numel(), _stream(stream)),
           "spec_verify_forward_tree")


def spec_tree_accept_workspace_bytes(batch: int, vocab: int) -> int:
    return int(lib().spec_tree_accept_workspace_bytes(batch, vocab))


def spec_tree_accept(target_logits, draft_probs, node_tokens, parents, uniforms, batch: int,
                     n_nodes: int, vocab: int, temperature: float, top_p: float, out_tokens,
                     out_path, n_accepted, ws, stream=None):
    _check(lib().spec_tree_accept(_ptr(target_logits), _ptr(draft_probs), _ptr(node_tokens),
                                  _ptr(parents), _ptr(uniforms), batch, n_nodes, vocab,
                                  temperature, top_p, _ptr(out_tokens), _ptr(out_path),
                                  _ptr(n_accepted), _ptr(ws), ws.numel(), _stream(stream)),
           "spec_tree_accept")


def spec_kv_tree_commit(handle: int, kv: "KVCache", path, n_accepted, n_nodes: int, ws,
                        stream=None):
    _check(lib().spec_kv_tree_commit(handle, ctypes.byref(kv.c()), _ptr(path), _ptr(n_accepted),
                                     n_nodes, _ptr(ws), _stream(stream)), "spec_kv_tree_commit")


def spec_wait_selftest(counter, target: int, limit_ms: float, ws, stream=None) -> None:
    """One bounded wait (the persistent forward's grid-barrier wait) on the
    uint32 device counter `counter` until it reaches `target`, giving up after
    `limit_ms`; a wait that gives up sets the timeout bit in `ws`'s status."""
    _check(lib().spec_wait_selftest(_ptr(counter), target, limit_ms, _ptr(ws), ws.numel(),
                                    _stream(stream)), "spec_wait_selftest")


def spec_device_status(ws, stream=None) -> tuple[int, int]:
    """(return status, device status bits); synchronises the stream."""
    out = ctypes.c_int32()
    r = lib().spec_device_status(_ptr(ws), _stream(stream), ctypes.byref(out))
    if r not in (SPEC_OK, SPEC_EDEVICE, SPEC_ETIMEOUT):
        raise SpecError(r, "spec_device_status")
    return r, out.value


def spec_timing_enable(handle: int, enable: bool):
    _check(lib().spec_timing_enable(handle, int(enable)), "spec_timing_enable")


def spec_timing_read(handle: int):
    ms = (ctypes.c_double * 3)()
    n = (ctypes.c_int64 * 3)()
    by = (ctypes.c_double * 3)()
    _check(lib().spec_timing_read(handle, ms, n, by), "spec_timing_read")
    return list(ms), list(n), list(by)


# ------------------------------------------------------------- owners
class Model:
    """Seeded synthetic weights in a torch-owned device buffer."""

    def __init__(self, cfg: ModelConfig, seed: int, device="cuda", stream=None):
        self.cfg = cfg
        self.seed = seed
        n = spec_model_weight_bytes(cfg)
        if n == 0:
            raise ValueError(f"unsupported config {cfg}")
        self.weights = torch.empty(n, dtype=torch.uint8, device=device)
        self.handle = spec_model_create(cfg, seed, self.weights, stream)

    def tensor(self, layer: int, which: int) -> torch.Tensor:
        """Logical weight matrix as a bf16 tensor (a copy for interleaved ones)."""
        ptr, (rows, cols), brows, stride = spec_model_tensor(self.handle, layer, which)
        off = ptr - self.weights.data_ptr()
        if brows == rows:
            return self.weights[off:off + rows * cols * 2].view(torch.bfloat16).view(rows, cols)
        nblk = rows // brows
        span = ((nblk - 1) * stride + brows) * cols * 2
        phys = self.weights[off:off + span].view(torch.bfloat16)
        out = torch.empty(rows, cols, dtype=torch.bfloat16, device=self.weights.device)
        for i in range(nblk):
            out[i * brows:(i + 1) * brows] = phys[i * stride * cols:(i * stride + brows) * cols].view(brows, cols)
        return out

    def close(self):
        if self.handle:
            spec_model_destroy(self.handle)
            self.handle = 0

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class KVCache:
    """Caller-owned target cache: k, v bf16 [layers][B][Hkv][cap][hd] and len int32 [B]."""

    def __init__(self, cfg: ModelConfig, batch: int, capacity: int, device="cuda"):
        self.cfg, self.batch, self.capacity = cfg, batch, capacity
        shape = (cfg.n_layers, batch, cfg.n_kv_heads, capacity, cfg.head_dim)
        self.k = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.v = torch.zeros(shape, dtype=torch.bfloat16, device=device)
        self.len = torch.zeros(batch, dtype=torch.int32, device=device)
        assert self.k.numel() * 2 == spec_kv_bytes(cfg, batch, capacity)

    def c(self) -> spec_kv_cache:
        return spec_kv_cache(self.k.data_ptr(), self.v.data_ptr(), self.len.data_ptr(),
                             self.batch, self.capacity)


def workspace(nbytes: int, device="cuda") -> torch.Tensor:
    """A device workspace (256-byte aligned, status word cleared)."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device)
