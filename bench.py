"""Benchmark of one speculative-decoding verification pass on GB300.

A step is the whole hot path on one batch: spec_verify_forward (the target's
single pass over [t_last, x_1..x_gamma]) + spec_accept + spec_kv_truncate.
Workload (default): 8B-shaped synthetic Llama decoder (32 layers, d 4096,
32/8 heads of 128, SwiGLU 14336, vocab 128256, bf16 weights ~ N(0, 0.02^2)
from seed), batch 1, gamma 4, 2048 cached tokens before every pass,
temperature 1.0.  Drafts come from a noisy copy of the target (its own
logits + N(0, 0.5^2) on the device, drawn with spec_draft_sample), produced
outside the timed region.  Weights (15 GB) stream from HBM every step, so
the inputs are larger than L2 and no flush is needed.

The value is the verify pass's algorithmic HBM bytes per second (weights +
KV read/write + logits + draft probabilities), with emitted tokens/s beside
it.  Multi-GPU runs are independent replicas (the pass does not shard).
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from speculative_decoding_verification_pass_gb300 import binding as sb  # noqa: E402
from speculative_decoding_verification_pass_gb300 import workloads as wl  # noqa: E402

METRIC = "verify-pass HBM GB/s (% of peak) and emitted tokens/s, 8B-shape γ=4, batch 1"

# DRAM bytes (read + write) per launch of the dominant kernel, from ncu
# captures summarised under profiles/, keyed by the sha1 of the kernel's
# source files (concatenated in the order listed): reported only while the
# sources are the ones that were measured.
TRAFFIC = {
    # batch 64 (each GEMM as two launches of 160 token rows): one 8B-dims
    # layer's eight GEMM launches x 32 + the LM head's two, / 258 launches
    "gemm_tc_kernel": {"files": ["gemm.cu", "gemm_common.cuh", "common.cuh", "internal.h"],
                       "source_sha1": "3b1ed332ec29f56b9421a63d49eda92c49aaa74c",
                       "bytes_per_launch": 125648430},
    # a 2-layer capture with the 8B dimensions, scaled to 32 layers by the
    # algorithmic bytes (weights, KV and logits each move once)
    "forward_kernel": {"files": ["forward.cu", "gemm_common.cuh", "attn_common.cuh", "common.cuh",
                                 "internal.h"],
                       "source_sha1": "3becae6f1076ad3e075db63ed1fe8ae0ccc51305",
                       "bytes_per_launch": 15426783985},
}


def kernel_traffic(kernel: str):
    import hashlib
    t = TRAFFIC[kernel]
    h = hashlib.sha1()
    for f in t["files"]:
        with open(os.path.join(ROOT, "speculative_decoding_verification_pass_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    ok = h.hexdigest() == t["source_sha1"]
    return t["bytes_per_launch"] if ok else None


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            p = json.load(f)
        return p["hbm_gbs"], p.get("bf16_tflops"), "measured"
    except Exception:
        return 6800.0, 1900.0, "fallback"


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during a region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu: int):
        self.gpu = gpu
        self.p = None

    def __enter__(self):
        try:
            self.p = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.Q}",
                                       "--format=csv,noheader,nounits", "-lms", "100"],
                                      stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.p = None
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.p:
            time.sleep(0.25)
            self.p.terminate()
            try:
                self.out, _ = self.p.communicate(timeout=5)
            except Exception:
                self.p.kill()

    def summary(self):
        rows = [r.split(", ") for r in self.out.strip().splitlines() if r.count(",") >= 8]
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sm = [float(r[1]) for r in rows]
        mx = max(float(r[2]) for r in rows)
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].strip() == "Active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": reasons,
                "samples": len(rows)}


class Workload:
    """One verify-step workload on the device: model, cache, drafts, outputs.

    ctx is one cached length for every sequence or an array of per-sequence
    lengths.  kv_init: "prefix" draws the cache contents on the host
    (N(0, 1) in bf16, seeded), "device" draws them on the device with a
    seeded torch generator (for caches too large to draw on the host),
    "prefill" runs spec_verify_forward over uniform random tokens (untimed).
    model / kv: share an existing Model / KVCache instead of creating one.""" 

    def __init__(self, cfg: sb.ModelConfig, B: int, gamma: int, ctx, T: float,
                 top_p: float, sigma: float, seed: int, steps_cap: int = 0,
                 model: "sb.Model | None" = None, kv_init: str = "prefix", cap: int = 0,
                 kv: "sb.KVCache | None" = None):
        self.cfg, self.B, self.gamma = cfg, B, gamma
        self.T, self.top_p, self.sigma = T, top_p, sigma
        self.n = gamma + 1
        self.lens = np.full(B, int(ctx), np.int64) if np.ndim(ctx) == 0 else np.asarray(ctx, np.int64)
        self.ctx = int(self.lens.max())
        self.cap = cap or self.ctx + self.n + 16
        dev = "cuda"
        self.own_model = model is None
        self.model = model if model is not None else sb.Model(cfg, 1000 + seed)
        if kv is not None:              # share a cache whose contents are already drawn
            self.cap = kv.capacity
            kv_init = "shared"
        self.kv = kv if kv is not None else sb.KVCache(cfg, B, self.cap)
        self.lens_dev = torch.from_numpy(self.lens.astype(np.int32)).to(dev)
        self.ws = sb.workspace(sb.spec_workspace_bytes(cfg, B, max(gamma, 127), self.cap))
        self.aws = sb.workspace(sb.spec_accept_workspace_bytes(B, gamma, cfg.vocab))
        hd = cfg.head_dim
        if kv_init == "prefix":
            ctx0 = self.ctx
            K, V = wl.kv_prefix(seed, cfg.n_layers, B, cfg.n_kv_heads, ctx0, hd)
            self.kv.k[:, :, :, :ctx0].copy_(torch.from_numpy(K.view(np.int16)).view(torch.bfloat16))
            self.kv.v[:, :, :, :ctx0].copy_(torch.from_numpy(V.view(np.int16)).view(torch.bfloat16))
            del K, V
        elif kv_init == "device":
            g = torch.Generator(device=dev)
            g.manual_seed(seed)
            self.kv.k.normal_(generator=g)
            self.kv.v.normal_(generator=g)
        elif kv_init == "prefill":
            toks = torch.from_numpy(wl.tokens(seed, B, self.ctx, cfg.vocab)).to(dev)
            for c0 in range(0, self.ctx, 128):
                blk = toks[:, c0:c0 + 128].contiguous()
                z = torch.empty(B, blk.shape[1], cfg.vocab, device=dev)
                sb.spec_verify_forward(self.model.handle, blk, B, blk.shape[1] - 1, self.kv, z, self.ws)
            torch.cuda.synchronize()
        self.kv.len.copy_(self.lens_dev)
        Vv = cfg.vocab
        self.tokens = torch.zeros(B, self.n, dtype=torch.int32, device=dev)
        self.logits = torch.empty(B, self.n, Vv, device=dev)
        self.q = torch.zeros(B, gamma, Vv, device=dev)
        self.x = torch.zeros(B, gamma, dtype=torch.int32, device=dev)
        self.u = torch.zeros(B, self.n, device=dev)
        self.out = torch.empty(B, self.n, dtype=torch.int32, device=dev)
        self.nacc = torch.empty(B, dtype=torch.int32, device=dev)
        self.zrow = torch.empty(B, 1, Vv, device=dev)
        self.qrow = torch.empty(B, Vv, device=dev)
        self.xrow = torch.empty(B, dtype=torch.int32, device=dev)
        self.gen = torch.Generator(device=dev)
        self.gen.manual_seed(seed)
        self.t_last = torch.from_numpy(wl.tokens(seed, B, 1, Vv)).to(dev).view(B)
        self.emitted = 0
        self.accepted = 0

    # ------------------------------------------------------------- harness
    def draft(self):
        """Untimed: gamma sequential single-token passes of the target give
        its logits at each draft position; the draft distribution is
        softmax((z + N(0, sigma^2)) / T) (+ top-p), x drawn from it."""
        B, g = self.B, self.gamma
        cur = self.t_last.view(B, 1).clone()
        self.tokens[:, 0] = self.t_last
        for i in range(g):
            sb.spec_verify_forward(self.model.handle, cur, B, 0, self.kv, self.zrow, self.ws)
            zq = self.zrow.view(B, -1) + self.sigma * torch.randn(B, self.cfg.vocab, device="cuda",
                                                                  generator=self.gen)
            ud = torch.rand(B, device="cuda", generator=self.gen)
            sb.spec_draft_sample(zq.contiguous(), B, self.cfg.vocab, self.T, self.top_p, ud,
                                 self.qrow, self.xrow, self.aws)
            self.q[:, i] = self.qrow
            self.x[:, i] = self.xrow
            self.tokens[:, i + 1] = self.xrow
            cur = self.xrow.view(B, 1).clone()
        self.kv.len.copy_(self.lens_dev)                          # back to the context
        self.u.copy_(torch.rand(B, self.n, device="cuda", generator=self.gen))

    def step(self, stream=None):
        """The timed hot path."""
        sb.spec_verify_forward(self.model.handle, self.tokens, self.B, self.gamma, self.kv,
                               self.logits, self.ws, stream)
        sb.spec_accept(self.logits, self.q, self.x, self.u, self.B, self.gamma, self.cfg.vocab,
                       self.T, self.top_p, self.out, self.nacc, self.aws, stream)
        sb.spec_kv_truncate(self.kv, self.nacc, self.gamma, self.ws, stream)

    def finish(self):
        """Untimed: count emitted tokens, take the last emitted token, and
        return the cache to the fixed context for the next pass."""
        n = self.nacc.cpu().numpy()
        o = self.out.cpu().numpy()
        self.emitted += int((n + 1).sum())
        self.accepted += int(n.sum())
        self.t_last = torch.from_numpy(o[np.arange(self.B), n].astype(np.int32)).cuda()
        self.kv.len.copy_(self.lens_dev)

    def close(self):
        if self.own_model:
            self.model.close()

    def check_status(self):
        for ws in (self.ws, self.aws):
            st, bits = sb.spec_device_status(ws)
            if st != sb.SPEC_OK:
                raise RuntimeError(f"device status {hex(bits)}")

    # ---------------------------------------------------------- accounting
    def bytes_per_step(self) -> float:
        c = self.cfg
        hd, d = c.head_dim, c.d_model
        qkv = (c.n_heads + 2 * c.n_kv_heads) * hd
        per_layer = (qkv * d + d * c.n_heads * hd + 2 * c.d_ffn * d + d * c.d_ffn) * 2
        M = self.B * self.n
        w = c.n_layers * per_layer + c.vocab * d * 2 + M * d * 2
        logits = M * c.vocab * 4 * 2
        q = self.B * self.gamma * c.vocab * 4
        return float(w + self.kv_bytes() + logits + q)

    def kv_bytes(self) -> float:
        """Keys/values read (each sequence's context + the new slots) and
        the new slots written, every layer."""
        c = self.cfg
        kv_tok = c.n_layers * c.n_kv_heads * c.head_dim * 2 * 2
        return float(sum((int(L) + self.n) * kv_tok + self.n * kv_tok for L in self.lens))

    def flops_per_step(self) -> float:
        """2 * M * weight parameters + the attention (scores and values,
        4 * keys * H * hd per new position and layer)."""
        c = self.cfg
        hd, d = c.head_dim, c.d_model
        qkv = (c.n_heads + 2 * c.n_kv_heads) * hd
        params = c.n_layers * (qkv * d + d * c.n_heads * hd + 3 * c.d_ffn * d) + c.vocab * d
        att = sum(4 * (int(L) + j + 1) * c.n_heads * hd for L in self.lens for j in range(self.n))
        return float(2 * self.B * self.n * params + c.n_layers * att)

    def gemm_bytes(self) -> float:
        c = self.cfg
        hd, d = c.head_dim, c.d_model
        qkv = (c.n_heads + 2 * c.n_kv_heads) * hd
        per_layer = (qkv * d + d * c.n_heads * hd + 2 * c.d_ffn * d + d * c.d_ffn) * 2
        return float(c.n_layers * per_layer + c.vocab * d * 2)

    def forward_bytes(self) -> float:
        """Algorithmic HBM bytes of one verify forward: every weight once, the
        new tokens' embedding rows, the attended keys/values (context + the
        gamma+1 new slots, every layer), the appended slots and the logits."""
        c = self.cfg
        M = self.B * self.n
        return float(self.gemm_bytes() + M * c.d_model * 2 + self.kv_bytes() + M * c.vocab * 4)


def time_steps(w: Workload, K: int):
    """Per-step device time (CUDA events on the launch stream), synchronised
    on both sides of each step; drafting happens between steps."""
    st = torch.cuda.current_stream()
    times = []
    for _ in range(K):
        w.draft()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        w.step()
        b.record(st)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
        w.finish()
    return times


def time_graph(w: Workload, K: int):
    """The same step captured once as a CUDA graph and replayed each step
    (one graph launch instead of the library's individual launches); inputs
    are refreshed in place between steps, as for the plain launches."""
    w.draft()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        w.step()
    torch.cuda.synchronize()
    w.kv.len.fill_(w.ctx)
    st = torch.cuda.current_stream()
    times = []
    for _ in range(K):
        w.draft()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        g.replay()
        b.record(st)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
        w.finish()
    del g
    return times


def time_e2e(w: Workload, K: int):
    """The same step through the C ABI with host buffers: pinned host inputs
    (tokens, draft probabilities, draft tokens, uniforms) copied in and the
    emitted tokens + n_accepted copied out inside the timed region."""
    st = torch.cuda.current_stream()
    h_tok = torch.empty_like(w.tokens, device="cpu").pin_memory()
    h_q = torch.empty_like(w.q, device="cpu").pin_memory()
    h_x = torch.empty_like(w.x, device="cpu").pin_memory()
    h_u = torch.empty_like(w.u, device="cpu").pin_memory()
    h_out = torch.empty_like(w.out, device="cpu").pin_memory()
    h_n = torch.empty_like(w.nacc, device="cpu").pin_memory()
    times = []
    for _ in range(K):
        w.draft()
        h_tok.copy_(w.tokens)
        h_q.copy_(w.q)
        h_x.copy_(w.x)
        h_u.copy_(w.u)
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        w.tokens.copy_(h_tok, non_blocking=True)
        w.q.copy_(h_q, non_blocking=True)
        w.x.copy_(h_x, non_blocking=True)
        w.u.copy_(h_u, non_blocking=True)
        w.step()
        h_out.copy_(w.out, non_blocking=True)
        h_n.copy_(w.nacc, non_blocking=True)
        b.record(st)
        torch.cuda.synchronize()
        times.append(a.elapsed_time(b))
        w.finish()
    h2d = sum(t.numel() * t.element_size() for t in (h_tok, h_q, h_x, h_u))
    d2h = h_out.numel() * h_out.element_size() + h_n.numel() * h_n.element_size()
    return times, h2d, d2h


def instrumented(w: Workload, K: int):
    """Per-kernel-kind device time of the GEMM and attention launches (events
    around each launch, so launches are serialised; separate from the
    headline timing)."""
    sb.spec_timing_enable(w.model.handle, True)
    sb.spec_timing_read(w.model.handle)
    for _ in range(K):
        w.draft()
        sb.spec_timing_read(w.model.handle)     # drop the draft passes
        w.step()
        ms, n, by = sb.spec_timing_read(w.model.handle)
        w.finish()
        yield ms, n, by
    sb.spec_timing_enable(w.model.handle, False)


def accept_time(w: Workload, K: int):
    st = torch.cuda.current_stream()
    ts = []
    for _ in range(K):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record(st)
        sb.spec_accept(w.logits, w.q, w.x, w.u, w.B, w.gamma, w.cfg.vocab, w.T, w.top_p, w.out,
                       w.nacc, w.aws)
        b.record(st)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts)


def mask_time(w: Workload, K: int, frac: float = 0.05):
    """Constrained rows: spec_mask_logits on the step's target logits (a copy)
    with one allowed-token set per row (a narrow, JSON-like set), then the
    accept on the masked rows.  Median device microseconds of each."""
    rows, V = w.B * w.n, w.cfg.vocab
    allowed = torch.from_numpy(wl.pack_allowed(wl.allowed_sets(17, rows, V, frac))).cuda()
    z = w.logits.clone()
    st = torch.cuda.current_stream()
    tm, ta = [], []
    for _ in range(K):
        z.copy_(w.logits)
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        c = torch.cuda.Event(enable_timing=True)
        a.record(st)
        sb.spec_mask_logits(z, allowed, rows, V, w.aws)
        b.record(st)
        sb.spec_accept(z, w.q, w.x, w.u, w.B, w.gamma, V, w.T, w.top_p, w.out, w.nacc, w.aws)
        c.record(st)
        torch.cuda.synchronize()
        tm.append(a.elapsed_time(b))
        ta.append(b.elapsed_time(c))
    stt, bits = sb.spec_device_status(w.aws)   # drafts outside the mask read as q(x) = 0
    if stt not in (sb.SPEC_OK, sb.SPEC_EDEVICE) or (bits & ~sb.DEV_Q_ZERO):
        raise RuntimeError(f"mask device status {hex(bits)}")
    return statistics.median(tm) * 1e3, statistics.median(ta) * 1e3


def gamma_ctl_probe(w: Workload, alpha: float, step_ms: float):
    """The host-side depth controller: its cost per recorded step for 64
    slots, and the depth it picks at the measured acceptance rate with the
    page's costs (2.0 ms per draft token, 20.0 ms per target pass) and with
    this run's own costs (one single-token pass of the drafting harness,
    one verify step)."""
    B = w.B
    cur = w.t_last.view(B, 1).clone()
    ts = []
    for _ in range(5):
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        sb.spec_verify_forward(w.model.handle, cur, B, 0, w.kv, w.zrow, w.ws)
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
        w.kv.len.fill_(w.ctx)
    draft_ms = statistics.median(ts)
    ctl = sb.GammaController(64)
    rng = np.random.default_rng(0)
    slots = list(range(64))
    used = [4] * 64
    accs = [rng.integers(0, 5, size=64).tolist() for _ in range(200)]
    t0 = time.perf_counter()
    for a in accs:
        used = ctl.step(slots, used, [min(x, u) for x, u in zip(a, used)])
    host_us = (time.perf_counter() - t0) / len(accs) * 1e6
    ctl.close()
    return {"host_us_per_step_64_slots": host_us, "alpha_measured": alpha,
            "gamma_page_costs": sb.spec_gamma_optimal(alpha, 2, 8, 2.0, 20.0),
            "draft_pass_ms": draft_ms, "verify_step_ms": step_ms,
            "gamma_measured_costs": sb.spec_gamma_optimal(alpha, 2, 8, draft_ms, step_ms)}


# ------------------------------------------------------------- CPU oracle
class OracleSample:
    """The oracle on this host, on a bounded sample of the verify step: one
    decoder layer of the model's shape over the M = B(gamma+1) new positions
    at the same cached length (cache contents from the same generator), an
    LM-head slice of head_rows rows, and the acceptance rule on one
    full-vocabulary step per sequence.  Every run() is a fresh step (new
    tokens, the cache reset to the context); its algorithmic bytes are the
    sample's own (that layer's weights and KV traffic, the head slice, the
    accept's logits and draft probabilities), so bytes / time is the oracle's
    rate on this workload, with no extrapolation.  The set-up (weights of the
    one layer and the head slice) is not timed."""

    def __init__(self, cfg: sb.ModelConfig, B: int, gamma: int, ctx: int, T: float, seed: int,
                 head_rows: int = 8192):
        from oracle import accept as OA
        from oracle import model as OM
        from oracle import weights as OW
        from oracle.bf16 import from_bits
        self.OA, self.OM = OA, OM
        self.cfg, self.B, self.gamma, self.ctx, self.T, self.seed = cfg, B, gamma, ctx, T, seed
        self.head_rows = min(head_rows, cfg.vocab)
        self.one = OM.Config(1, cfg.d_model, cfg.n_heads, cfg.n_kv_heads, cfg.d_ffn,
                             self.head_rows, cfg.rms_eps, cfg.rope_theta)
        self.W = OW.Weights(self.one, 1000 + seed)
        self.W.layer(0)
        self.W.head()
        self.kvs = OM.KVState(self.one, B, ctx + gamma + 1)
        K, V = wl.kv_prefix(seed, 1, B, cfg.n_kv_heads, ctx, cfg.head_dim)
        self.kvs.load_prefix([from_bits(K[0])], [from_bits(V[0])], [ctx] * B)
        self.it = 0
        c = cfg
        hd, d = c.head_dim, c.d_model
        qkv = (c.n_heads + 2 * c.n_kv_heads) * hd
        layer_w = (qkv * d + d * c.n_heads * hd + 3 * c.d_ffn * d) * 2
        kv_tok = c.n_kv_heads * hd * 2 * 2
        n = gamma + 1
        self.bytes = float(layer_w + B * ((ctx + n) * kv_tok + n * kv_tok)
                           + self.head_rows * d * 2 + B * (2 * n + gamma) * c.vocab * 4)
        self.desc = (f"one step of: 1 of {c.n_layers} decoder layers (M={B * n}, context {ctx}), "
                     f"LM head {self.head_rows} of {c.vocab} rows, accept on {B} full-vocabulary "
                     f"step(s); GB/s of that sample's own algorithmic bytes")

    def run(self) -> float:
        OA, OM = self.OA, self.OM
        self.it += 1
        s = self.seed + 7 * self.it
        B, g, V = self.B, self.gamma, self.cfg.vocab
        toks = wl.tokens(s, B, g + 1, self.head_rows)
        zq, zp = wl.accept_logits(s, B, g, V)
        ud = wl.uniforms(s, B, g, stream=8)
        u = wl.uniforms(s, B, g + 1)
        qx = [OA.draft_sample(zq[b, :g], ud[b], self.T if self.T > 0 else 1.0)[:2] for b in range(B)]
        self.kvs.lens[:] = self.ctx
        t0 = time.perf_counter()
        OM.forward(self.one, self.W, toks, self.kvs)
        for b in range(B):
            OA.accept(zp[b], qx[b][0], qx[b][1], u[b], self.T)
        return time.perf_counter() - t0


def oracle_rate(sample: OracleSample, steps: int, warmup: int = 1):
    """(GB/s, mean seconds per sample step, steps timed)."""
    for _ in range(warmup):
        sample.run()
    ts = [sample.run() for _ in range(steps)]
    return sample.bytes * len(ts) / sum(ts) / 1e9, sum(ts) / len(ts), len(ts)


def blas_threads():
    for k in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS", "MKL_NUM_THREADS"):
        if os.environ.get(k):
            return int(os.environ[k])
    return os.cpu_count()


# ----------------------------------------------------------- tree rounds
TREE_PARENTS = [-1, 0, 0, 1, 1, 2, 2]   # root + full binary tree of depth 2 (6 drafted nodes)


class TreeRound:
    """Draft-tree verification on the same model and cache: the root is the
    last emitted token, every node's children are two independent draws from
    a noisy copy of the target's distribution at that node (drafted level by
    level with untimed tree passes); the timed round is the tree forward,
    the tree accept walk and the KV commit."""

    def __init__(self, w: Workload):
        self.w = w
        B, V = w.B, w.cfg.vocab
        self.par = TREE_PARENTS
        self.n = len(self.par)
        dev = "cuda"
        self.tokens = torch.zeros(B, self.n, dtype=torch.int32, device=dev)
        self.parents = torch.tensor([self.par] * B, dtype=torch.int32, device=dev)
        anc, dep = [], []
        for k in range(1, self.n + 1):
            a, d = sb.spec_tree_masks(self.par[:k])
            anc.append(a)
            dep.append(d)
        self.masks = []   # per prefix size: (anc, depth) on the device
        for a, d in zip(anc, dep):
            at = torch.from_numpy(np.array([a] * B, dtype=np.uint64).view(np.int64)).to(dev)
            dt = torch.tensor([d] * B, dtype=torch.int32, device=dev)
            self.masks.append((at, dt))
        self.logits = torch.empty(B, self.n, V, device=dev)
        self.q = torch.zeros(B, self.n, V, device=dev)
        self.u = torch.zeros(B, self.n, device=dev)
        self.out = torch.empty(B, self.n, dtype=torch.int32, device=dev)
        self.path = torch.empty(B, self.n, dtype=torch.int32, device=dev)
        self.nacc = torch.empty(B, dtype=torch.int32, device=dev)
        self.tws = sb.workspace(sb.spec_tree_accept_workspace_bytes(B, V))
        self.fws = sb.workspace(sb.spec_workspace_bytes(w.cfg, B, self.n - 1, w.cap))
        self.qrows = torch.empty(2 * B, V, device=dev)
        self.xrows = torch.empty(2 * B, dtype=torch.int32, device=dev)
        self.emitted = 0

    def draft(self):
        w, B, V = self.w, self.w.B, self.w.cfg.vocab
        self.tokens[:, 0] = w.t_last
        # levels: nodes 0 | 1 2 | 3 4 5 6; node c's children are 2c + 1, 2c + 2
        for k, level in ((1, [0]), (3, [1, 2])):
            z = torch.empty(B, k, V, device="cuda")
            a, d = self.masks[k - 1]
            sb.spec_verify_forward_tree(w.model.handle, self.tokens[:, :k].contiguous(), a, d, B, k,
                                        w.kv, z, self.fws)
            w.kv.len.fill_(w.ctx)
            for c in level:
                zq = z[:, c] + w.sigma * torch.randn(B, V, device="cuda", generator=w.gen)
                zq2 = zq.repeat_interleave(2, dim=0).contiguous()
                ud = torch.rand(2 * B, device="cuda", generator=w.gen)
                sb.spec_draft_sample(zq2, 2 * B, V, w.T, w.top_p, ud, self.qrows, self.xrows, w.aws)
                self.q[:, c] = self.qrows.view(B, 2, V)[:, 0]
                self.tokens[:, 2 * c + 1:2 * c + 3] = self.xrows.view(B, 2)
        self.u.copy_(torch.rand(B, self.n, device="cuda", generator=w.gen))

    def step(self):
        w = self.w
        a, d = self.masks[-1]
        sb.spec_verify_forward_tree(w.model.handle, self.tokens, a, d, w.B, self.n, w.kv, self.logits,
                                    self.fws)
        sb.spec_tree_accept(self.logits, self.q, self.tokens, self.parents, self.u, w.B, self.n,
                            w.cfg.vocab, w.T, w.top_p, self.out, self.path, self.nacc, self.tws)
        sb.spec_kv_tree_commit(w.model.handle, w.kv, self.path, self.nacc, self.n, self.fws)

    def finish(self):
        w = self.w
        n = self.nacc.cpu().numpy()
        o = self.out.cpu().numpy()
        self.emitted += int((n + 1).sum())
        w.t_last = torch.from_numpy(o[np.arange(w.B), n].astype(np.int32)).cuda()
        w.kv.len.fill_(w.ctx)


def time_tree(w: Workload, K: int, warmup: int = 2):
    tr = TreeRound(w)
    times = []
    for i in range(warmup + K):
        tr.draft()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        a.record()
        tr.step()
        b.record()
        torch.cuda.synchronize()
        if i == warmup - 1:
            tr.emitted = 0
        if i >= warmup:
            times.append(a.elapsed_time(b))
        tr.finish()
    # the tree accept and the commit alone (last round's inputs; the commit on
    # a cache reset to the context + the round's slots each time)
    stream = torch.cuda.current_stream()
    ta, tc = [], []
    for _ in range(5):
        e0, e1, e2 = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        w.kv.len.fill_(w.ctx + tr.n)
        e0.record(stream)
        sb.spec_tree_accept(tr.logits, tr.q, tr.tokens, tr.parents, tr.u, w.B, tr.n, w.cfg.vocab, w.T,
                            w.top_p, tr.out, tr.path, tr.nacc, tr.tws)
        e1.record(stream)
        sb.spec_kv_tree_commit(w.model.handle, w.kv, tr.path, tr.nacc, tr.n, tr.fws)
        e2.record(stream)
        torch.cuda.synchronize()
        ta.append(e0.elapsed_time(e1))
        tc.append(e1.elapsed_time(e2))
    w.kv.len.fill_(w.ctx)
    for ws in (tr.tws, tr.fws):
        st, bits = sb.spec_device_status(ws)
        if st != sb.SPEC_OK:
            raise RuntimeError(f"tree device status {hex(bits)}")
    w.check_status()
    ms = sum(times) / len(times)
    c = w.cfg
    hd, d = c.head_dim, c.d_model
    kv_tok = c.n_layers * c.n_kv_heads * hd * 2 * 2
    fwd = w.gemm_bytes() + w.B * tr.n * d * 2 + w.B * ((w.ctx + tr.n) * kv_tok + tr.n * kv_tok) \
        + w.B * tr.n * c.vocab * 4
    return {"workload": f"draft tree: root + full binary tree of depth 2 ({tr.n - 1} drafted "
                        f"nodes), batch {w.B}, context {w.ctx}, same model, draft and T",
            "ms_per_round": ms, "emitted_per_round": tr.emitted / (K * w.B),
            "emitted_tokens_per_s": tr.emitted / (sum(times) / 1e3),
            "hbm_gbs": fwd / (ms / 1e3) / 1e9, "rounds": K,
            "tree_accept_us": statistics.median(ta) * 1e3, "commit_us": statistics.median(tc) * 1e3}


# ------------------------------------------------------------- paged KV
def time_paged(w: Workload, K: int):
    """The same step on a paged copy of the cache (64-slot pages through a
    page table, pages taken from the host pool's free list): forward +
    accept + device rollback timed; the pool's release of the pages past the
    new length, and its reservation for the next pass, happen between steps."""
    B, c = w.B, w.cfg
    max_pages = -(-w.cap // sb.PAGE_SLOTS)
    pk = sb.PagedKVCache(c, B, n_pages=B * max_pages + 4, max_pages=max_pages)
    for b in range(B):
        pk.reserve(b, w.ctx)
    t = pk.host_table()
    for b in range(B):
        for j in range(-(-w.ctx // sb.PAGE_SLOTS)):
            lo, hi = j * sb.PAGE_SLOTS, min(w.ctx, (j + 1) * sb.PAGE_SLOTS)
            pk.k[:, t[b, j], :, :hi - lo] = w.kv.k[:, b, :, lo:hi]
            pk.v[:, t[b, j], :, :hi - lo] = w.kv.v[:, b, :, lo:hi]
    pk.len.fill_(w.ctx)
    st = torch.cuda.current_stream()
    times = []
    free_before = pk.free_pages()
    for i in range(K + 2):
        w.draft()
        for b in range(B):
            pk.reserve(b, w.ctx + w.n)
        pk.sync()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        e = torch.cuda.Event(enable_timing=True)
        a.record(st)
        sb.spec_verify_forward_paged(w.model.handle, w.tokens, B, w.gamma, pk, w.logits, w.ws)
        sb.spec_accept(w.logits, w.q, w.x, w.u, B, w.gamma, c.vocab, w.T, w.top_p, w.out, w.nacc,
                       w.aws)
        sb.spec_paged_kv_truncate(pk, w.nacc, w.gamma, w.ws)
        e.record(st)
        torch.cuda.synchronize()
        if i >= 2:
            times.append(a.elapsed_time(e))
        lens = pk.len.cpu().numpy()
        for b in range(B):
            pk.release(b, int(lens[b]))
        w.finish()
        pk.len.fill_(w.ctx)
        for b in range(B):
            pk.release(b, w.ctx)
    w.check_status()
    ms = sum(times) / len(times)
    out = {"workload": f"the verify step on a paged cache ({sb.PAGE_SLOTS}-slot pages, "
                       f"{max_pages} pages per sequence), same model, context and draft",
           "ms_per_step": ms, "value": w.bytes_per_step() / (ms / 1e3) / 1e9, "unit": "GB/s",
           "steps": K, "pages_returned": pk.free_pages() == free_before}
    pk.close()
    return out


# ------------------------------------------------------- per-config lines
def _ev():
    return torch.cuda.Event(enable_timing=True)


class L2Flush:
    """Writes a 512 MB buffer (about four times the L2) before a timed
    iteration whose working set would otherwise stay in L2; untimed."""

    def __init__(self):
        self.buf = torch.empty(512 << 20, dtype=torch.uint8, device="cuda")
        self.i = 0

    def __call__(self):
        self.i += 1
        self.buf.fill_(self.i & 0xFF)
        torch.cuda.synchronize()


def _parity(name, cases, near, excused):
    return {"sample": name, "cases": cases, "in_margin": near, "excused": excused,
            "in_margin_frac": near / max(1, cases), "boundary_frac": excused / max(1, cases)}


def launch_floor_us(K: int = 200) -> float:
    """Median device time of this library's smallest launch (the rollback
    kernel on one sequence): the latency floor of a one-launch call."""
    cfg = sb.ModelConfig(1, 256, 4, 2, 256, 1000)
    kv = sb.KVCache(cfg, 1, 64)
    kv.len.fill_(10)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, 1, 4, 64))
    nacc = torch.zeros(1, dtype=torch.int32, device="cuda")
    ts = []
    for _ in range(K):
        a, b = _ev(), _ev()
        a.record()
        sb.spec_kv_truncate(kv, nacc, 0, ws)
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
    return statistics.median(ts) * 1e3


def config_accept_only(steps: int = 1000):
    """Accept-only workload: batch 1, gamma 4, V 4096, z_q ~ N(0, 2^2),
    z_p = z_q + N(0, 0.5^2), q = softmax(z_q) in fp64 on the host, drafts
    drawn from q, T = 1; `steps` independent steps, L2 flushed before each.
    Its bytes (147 KB) are far below anything HBM-bound: the bound is the
    launch latency of one kernel, reported as the floor."""
    from oracle import accept as OA
    B, g, V, T = 1, 4, 4096, 1.0
    seed = wl.BASE_SEED
    zq, zp = wl.accept_logits(seed, steps, g, V)
    ud = wl.uniforms(seed, steps, g, stream=8)
    u = wl.uniforms(seed, steps, g + 1)
    q = np.zeros((steps, g, V), np.float32)
    x = np.zeros((steps, g), np.int32)
    for i in range(steps):
        qs, ts, _ = OA.draft_sample(zq[i, :g], ud[i], T)
        q[i], x[i] = qs.astype(np.float32), ts
    dz, dq = torch.from_numpy(zp).cuda(), torch.from_numpy(q).cuda()
    dx, du = torch.from_numpy(x).cuda(), torch.from_numpy(u).cuda()
    out = torch.empty(steps, g + 1, dtype=torch.int32, device="cuda")
    nacc = torch.empty(steps, dtype=torch.int32, device="cuda")
    ws = sb.workspace(sb.spec_accept_workspace_bytes(B, g, V))
    flush = L2Flush()
    ts = []
    for i in range(steps):
        flush()
        a, b = _ev(), _ev()
        a.record()
        sb.spec_accept(dz[i:i + 1], dq[i:i + 1], dx[i:i + 1], du[i:i + 1], B, g, V, T, 1.0,
                       out[i:i + 1], nacc[i:i + 1], ws)
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) * 1e3)
    if sb.spec_device_status(ws)[0] != sb.SPEC_OK:
        raise RuntimeError("accept-only device status")
    o, na = out.cpu().numpy(), nacc.cpu().numpy()
    near = excused = 0
    t0 = time.perf_counter()
    for i in range(steps):
        r = OA.accept(zp[i], q[i], x[i], u[i], T)
        near += r.boundary
        if not (int(na[i]) == r.n_accepted and o[i].tolist() == r.tokens):
            excused += 1
            if not r.boundary:
                raise RuntimeError(f"accept-only step {i} differs from the oracle")
    oracle_us = (time.perf_counter() - t0) / steps * 1e6
    med = statistics.median(ts)
    floor = launch_floor_us()
    nbytes = (2 * (g + 1) + g) * V * 4
    return {"workload": f"spec_accept only: batch 1, gamma 4, V 4096, T 1, {steps} steps, "
                        f"L2 flushed before each", "us_per_call": med,
            "p90_us": float(np.percentile(ts, 90)), "bytes_per_call": nbytes,
            "roofline": {"bound": "latency", "achieved_us": med, "floor_us": floor,
                         "frac": floor / med,
                         "note": "one launch of the smallest kernel of this library"},
            "acceptance": float(na.mean()) / g,
            "parity": _parity("every step vs the oracle on identical inputs", steps, near, excused),
            "cpu_baseline": {"us_per_call": oracle_us, "kind": "oracle", "cores": 1,
                             "sample": f"the oracle's accept on the same {steps} steps"}}


def config_lm_head(hbm: float, steps: int = 40):
    """LM-head verify + accept: activations ~ N(0, 1) in bf16 for 5
    positions, LM head 4096 x 32000 ~ N(0, 0.02^2); draft probabilities from
    the same head on the activations + N(0, 0.3^2) (fp64, host), T = 1; the
    timed step is the M = 5 skinny GEMM then the fused accept, L2 flushed
    before each step."""
    from oracle import accept as OA
    from oracle import model as OM
    from oracle import weights as OW
    cfg = sb.ModelConfig(0, 4096, 32, 8, 128, 32000)
    seed = wl.BASE_SEED + 1
    m = sb.Model(cfg, seed)
    head = OW.tensor(seed, OW.HEAD, cfg.vocab, cfg.d_model)
    ws = sb.workspace(sb.spec_workspace_bytes(cfg, 5, 0, 1))
    aws = sb.workspace(sb.spec_accept_workspace_bytes(1, 4, cfg.vocab))
    z = torch.empty(1, 5, cfg.vocab, device="cuda")
    out = torch.empty(1, 5, dtype=torch.int32, device="cuda")
    nacc = torch.empty(1, dtype=torch.int32, device="cuda")
    flush = L2Flush()
    ts, t_or = [], []
    near = excused = 0
    err = 0.0
    accepted = 0
    for i in range(steps):
        hb = wl.hidden_bf16(seed + i, 5, cfg.d_model)
        h = wl.bf16_bits_to_f32(hb).astype(np.float64)
        t0 = time.perf_counter()
        ref = OM.lm_head(h, head)
        noisy = h[:4] + wl.gauss(seed + i, (4, cfg.d_model), 0.3)
        q, x, _ = OA.draft_sample(OM.lm_head(noisy, head), wl.uniforms(seed + i, 4, stream=8), 1.0)
        u = wl.uniforms(seed + i, 1, 5)
        r = OA.accept(ref.astype(np.float32), q.astype(np.float32), x, u[0], 1.0)
        t_or.append(time.perf_counter() - t0)
        dh = torch.from_numpy(hb.view(np.int16)).cuda()
        dq = torch.from_numpy(q.astype(np.float32)[None]).cuda()
        dx = torch.from_numpy(x.astype(np.int32)[None]).cuda()
        du = torch.from_numpy(u).cuda()
        flush()
        a, b = _ev(), _ev()
        a.record()
        sb.spec_lm_head(m.handle, dh, 5, z, ws)
        sb.spec_accept(z, dq, dx, du, 1, 4, cfg.vocab, 1.0, 1.0, out, nacc, aws)
        b.record()
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b))
        accepted += int(nacc[0])
        err = max(err, float((np.abs(z[0].double().cpu().numpy() - ref) / (1 + np.abs(ref))).max()))
        # parity sample: the device accept on the oracle's logits
        sb.spec_accept(torch.from_numpy(ref.astype(np.float32)[None]).cuda(), dq, dx, du, 1, 4,
                       cfg.vocab, 1.0, 1.0, out, nacc, aws)
        near += r.boundary
        if not (int(nacc[0]) == r.n_accepted and out[0].tolist() == r.tokens):
            excused += 1
            if not r.boundary:
                raise RuntimeError(f"LM-head step {i} accept differs from the oracle")
    for w_ in (ws, aws):
        if sb.spec_device_status(w_)[0] != sb.SPEC_OK:
            raise RuntimeError("LM-head workload device status")
    m.close()
    ms = statistics.median(ts)
    nbytes = cfg.vocab * cfg.d_model * 2 + 5 * cfg.d_model * 2 + 5 * cfg.vocab * 4 * 2 \
        + 4 * cfg.vocab * 4
    gbs = nbytes / (ms / 1e3) / 1e9
    return {"workload": "LM head 4096 x 32000 on 5 positions + fused accept, batch 1, gamma 4, "
                        f"T 1, {steps} steps, L2 flushed before each",
            "ms_per_step": ms, "value": gbs, "unit": "GB/s", "bytes_per_step": nbytes,
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": hbm, "unit": "GB/s",
                         "frac": gbs / hbm, "peak_source": "measured (burst copy)"},
            "logits_max_rel_err": err, "acceptance": accepted / (4 * steps),
            "parity": _parity("device accept on the oracle's logits, every step", steps, near,
                              excused),
            "cpu_baseline": {"ms_per_step": statistics.median(t_or) * 1e3, "kind": "oracle",
                             "cores": blas_threads(),
                             "value": nbytes / statistics.median(t_or) / 1e9, "unit": "GB/s",
                             "sample": "the oracle's LM head + accept on the same steps"}}


def run_workload(w: Workload, steps: int, warmup: int, hbm: float, inst: bool = True):
    """ms/step, GB/s, fractions, tokens/s and acceptance of a workload's
    verify step (forward + accept + rollback), plus the forward kernel's own
    launch time when inst."""
    time_steps(w, warmup)
    w.check_status()
    w.emitted = w.accepted = 0
    times = time_steps(w, steps)
    w.check_status()
    ms = sum(times) / len(times)
    nbytes = w.bytes_per_step()
    gbs = nbytes / (ms / 1e3) / 1e9
    fl = w.flops_per_step()
    tf = fl / (ms / 1e3) / 1e12
    res = {"batch": w.B, "gamma": w.gamma, "temperature": w.T, "top_p": w.top_p,
           "sigma": w.sigma, "context_mean": float(w.lens.mean()),
           "ms_per_step": ms, "value": gbs, "unit": "GB/s", "bytes_per_step": nbytes,
           "hbm_frac_of_measured": gbs / hbm, "hbm_frac_of_8tbs": gbs / 8000.0,
           "tflops": tf, "flops_per_step": fl,
           "emitted_tokens_per_s": w.emitted / (sum(times) / 1e3),
           "acceptance": w.accepted / max(1, steps * w.B * w.gamma),
           "accept_us": accept_time(w, 5) * 1e3}
    if inst:
        gm = gn = am = an = pm = pn = 0.0
        for ms_, n_, _ in instrumented(w, 2):
            gm += ms_[0]; gn += n_[0]; am += ms_[1]; an += n_[1]; pm += ms_[2]; pn += n_[2]
        if pn:
            kms = pm / pn
            res["forward_kernel"] = {"kernel": "forward_kernel", "launch_ms": kms,
                                     "achieved_gbs": w.forward_bytes() / (kms / 1e3) / 1e9,
                                     "frac": w.forward_bytes() / (kms / 1e3) / 1e9 / hbm}
        elif gn:
            res["forward_kernel"] = {"kernel": "gemm_tc_kernel + attention (per-step schedule)",
                                     "gemm_ms_per_step": gm / 2, "attention_ms_per_step": am / 2,
                                     "gemm_gbs": w.gemm_bytes() / (gm / 2 / 1e3) / 1e9}
    return res


def config_1b(hbm: float, steps: int, warmup: int):
    """The 1B-shaped decoder: batch 1, 512 prefix tokens uniform over the
    vocabulary prefilled through spec_verify_forward (untimed), gamma 4,
    T 1, noisy-target draft sigma 0.5; 2.1 GB of weights per step."""
    w = Workload(sb.LLAMA_1B, 1, 4, 512, 1.0, 1.0, 0.5, seed=5, kv_init="prefill")
    res = run_workload(w, steps, warmup, hbm)
    w.close()
    smp = OracleSample(sb.LLAMA_1B, 1, 4, 512, 1.0, 5)
    val, sec, k = oracle_rate(smp, 2)
    res.update({"workload": "1B-shaped synthetic Llama decoder, batch 1, 512 prefilled tokens, "
                            "gamma 4, T 1, noisy-target draft sigma 0.5",
                "roofline": {"bound": "hbm", "achieved": res["value"], "peak": hbm, "unit": "GB/s",
                             "frac": res["value"] / hbm, "peak_source": "measured (burst copy)"},
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": blas_threads(),
                                 "kind": "oracle", "sample": f"{k} x {smp.desc}"}})
    return res


def config_8b_variants(w: Workload, hbm: float, steps: int, warmup: int):
    """The 8B headline workload at the other draft lengths and at greedy
    decoding: same model and 2048-token context; gamma 2 and 8 at T 1, and
    gamma 2, 4 and 8 at T 0."""
    out = []
    for gamma, T in ((2, 1.0), (8, 1.0), (2, 0.0), (4, 0.0), (8, 0.0)):
        v = Workload(w.cfg, 1, gamma, w.ctx, T, 1.0, w.sigma, seed=3, model=w.model, kv=w.kv)
        r = run_workload(v, steps, warmup, hbm)
        r["workload"] = (f"8B-shaped decoder, batch 1, context {w.ctx}, gamma {gamma}, T {T}, "
                         f"noisy-target draft sigma {w.sigma}")
        out.append(r)
    w.kv.len.copy_(w.lens_dev)
    return out


def config_batched(model: sb.Model, hbm: float, tflops: float, steps: int, warmup: int):
    """The batched 8B workload: batch 16 and 64, per-sequence cached lengths
    uniform in [512, 4096] (cache contents N(0, 1) drawn on the device),
    gamma 4, T 0.8 and top-p 0.9 on p and q, drafts from noisy copies of
    the target with sigma 0.3 and 1.0; bytes and FLOPs from the drawn
    lengths, against the HBM and the bf16 tensor bounds."""
    out = []
    for B in (16, 64):
        lens = wl.context_lengths(wl.BASE_SEED + B, B, 512, 4096)
        w = Workload(sb.LLAMA_8B, B, 4, lens, 0.8, 0.9, 0.3, seed=40 + B, model=model,
                     kv_init="device", cap=4096 + 16)
        for sigma in (0.3, 1.0):
            w.sigma = sigma
            r = run_workload(w, steps, warmup, hbm, inst=(sigma == 0.3))
            t_hbm = r["bytes_per_step"] / (hbm * 1e9) * 1e3
            t_tc = r["flops_per_step"] / (tflops * 1e12) * 1e3
            r["workload"] = (f"8B-shaped decoder, batch {B}, contexts U[512, 4096] (mean "
                             f"{lens.mean():.0f}), gamma 4, T 0.8, top-p 0.9, draft sigma {sigma}")
            r["roofline"] = {"bound": "hbm" if t_hbm >= t_tc else "tensor",
                             "hbm_ms": t_hbm, "tensor_ms": t_tc,
                             "frac": max(t_hbm, t_tc) / r["ms_per_step"],
                             "tensor_frac": r["tflops"] / tflops,
                             "hbm_frac": r["hbm_frac_of_measured"],
                             "peaks": {"hbm_gbs": hbm, "bf16_tflops": tflops,
                                       "source": "measured (burst)"}}
            out.append(r)
        del w
        torch.cuda.empty_cache()
    return out


def headline_parity(T: float, top_p: float, steps: int = 100):
    """Parity sample at the headline's accept shape (batch 1, gamma 4,
    V 128256): the device accept against the oracle on identical seeded
    inputs (accept-only recipe), counted under the boundary rule."""
    from oracle import accept as OA
    g, V = 4, 128256
    ws = sb.workspace(sb.spec_accept_workspace_bytes(1, g, V))
    out = torch.empty(1, g + 1, dtype=torch.int32, device="cuda")
    nacc = torch.empty(1, dtype=torch.int32, device="cuda")
    near = excused = 0
    for i in range(steps):
        seed = wl.BASE_SEED + 500 + i
        zq, zp = wl.accept_logits(seed, 1, g, V)
        q, x, _ = OA.draft_sample(zq[0, :g], wl.uniforms(seed, g, stream=8), T if T > 0 else 1.0,
                                  top_p)
        u = wl.uniforms(seed, 1, g + 1)
        sb.spec_accept(torch.from_numpy(zp).cuda(), torch.from_numpy(q.astype(np.float32)[None]).cuda(),
                       torch.from_numpy(x.astype(np.int32)[None]).cuda(), torch.from_numpy(u).cuda(),
                       1, g, V, T, top_p, out, nacc, ws)
        r = OA.accept(zp[0], q.astype(np.float32), x, u[0], T, top_p)
        near += r.boundary
        if not (int(nacc[0]) == r.n_accepted and out[0].tolist() == r.tokens):
            excused += 1
            if not r.boundary:
                raise RuntimeError(f"headline parity step {i} differs from the oracle")
    return _parity(f"{steps} accept steps at batch 1, gamma 4, V 128256, T {T}, top-p {top_p} "
                   "(accept-only recipe), identical inputs", steps, near, excused)


# ------------------------------------------------------------------ main
def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--gamma", type=int, default=4)
    ap.add_argument("--batch", type=int, default=1)
    ap.add_argument("--context", type=int, default=2048)
    ap.add_argument("--temperature", type=float, default=1.0)
    ap.add_argument("--top-p", type=float, default=1.0)
    ap.add_argument("--sigma", type=float, default=0.5)
    ap.add_argument("--shape", default="8b", choices=["8b", "1b"])
    ap.add_argument("--layers", type=int, default=0,
                    help="override the decoder depth (profiling a smaller model)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true",
                    help="skip the per-config sub-lines (accept-only, LM head, 1B, 8B variants, "
                         "batched)")
    return ap.parse_args()


def job_seconds(t_local: float, world: int, device) -> float:
    """The job's time for the timed region: the maximum over the ranks (each
    rank's replica runs the same steps; the slowest one ends the job)."""
    if world == 1:
        return t_local
    import torch.distributed as dist
    tt = torch.tensor([t_local], dtype=torch.float64, device=device)
    dist.all_reduce(tt, op=dist.ReduceOp.MAX)
    return float(tt)


def job_value(step_bytes: float, steps: int, world: int, seconds: float) -> float:
    """Whole-job algorithmic GB/s: the bytes all replicas moved over the job's time."""
    return step_bytes * steps * world / seconds / 1e9


def main():
    args = parse()
    if args.warmup < 3:
        args.warmup = 3
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    cfg = sb.LLAMA_8B if args.shape == "8b" else sb.LLAMA_1B
    if args.layers:
        import dataclasses
        cfg = dataclasses.replace(cfg, n_layers=args.layers)
    workload = (f"{args.shape.upper()}-shaped synthetic Llama decoder verify pass + accept + "
                f"rollback, batch {args.batch}, gamma {args.gamma}, context {args.context}, "
                f"T={args.temperature}, top_p={args.top_p}, noisy-target draft sigma {args.sigma}")
    config = {"workload": workload, "batch": args.batch, "gamma": args.gamma,
              "context": args.context, "temperature": args.temperature, "top_p": args.top_p,
              "l2": "inputs larger than L2 (weights stream from HBM every step)",
              "parallelism": f"replicas x{world}"}
    if args.impl == "reference":
        if rank != 0:
            return
        # the oracle as it stands on this host's cores: every step is one
        # timed bounded sample of the workload (OracleSample), W untimed
        # then K timed, so the line's steps are the steps that ran
        smp = OracleSample(cfg, args.batch, args.gamma, args.context, args.temperature, 3)
        val, sec, k = oracle_rate(smp, args.steps, args.warmup)
        line = {"metric": METRIC, "value": val, "unit": "GB/s", "impl": "reference",
                "n_gpus": args.gpus, "steps": k, "warmup": args.warmup,
                "ms_per_step": sec * 1e3, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "step_is": smp.desc, "bytes_per_step": smp.bytes,
                "cpu_baseline": {"value": val, "unit": "GB/s", "cores": blas_threads(),
                                 "kind": "oracle", "sample": smp.desc},
                "e2e": {"value": val, "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return
    torch.cuda.set_device(local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    __import__("__graft_entry__").build()
    w = Workload(cfg, args.batch, args.gamma, args.context, args.temperature, args.top_p,
                 args.sigma, seed=3 + rank, steps_cap=args.steps)
    time_steps(w, args.warmup)
    w.check_status()
    w.emitted = w.accepted = 0
    if world > 1:
        torch.distributed.barrier()
    with ClockSampler(local) as clk:
        times = time_steps(w, args.steps)
    w.check_status()
    emitted, accepted = w.emitted, w.accepted
    t_total = job_seconds(sum(times) / 1e3, world, "cuda")
    step_bytes = w.bytes_per_step()
    value = job_value(step_bytes, args.steps, world, t_total)
    try:
        gt = time_graph(w, max(3, args.steps // 2))
        w.check_status()
        gms = sum(gt) / len(gt)
        graph = {"ms_per_step": gms, "value": step_bytes * world / (gms / 1e3) / 1e9, "unit": "GB/s",
                 "steps": len(gt)}
    except Exception as exc:  # capture not supported by this driver / torch
        graph = {"unavailable": str(exc).splitlines()[0][:200]}
    e2e_times, h2d, d2h = time_e2e(w, max(3, args.steps // 2))
    e2e_val = step_bytes * len(e2e_times) * world / (sum(e2e_times) / 1e3) / 1e9
    gm = gn = gb = am = an = pm = pn = 0.0
    k_inst = 3
    for ms, n, by in instrumented(w, k_inst):
        gm += ms[0]; gn += n[0]; gb += by[0]; am += ms[1]; an += n[1]; pm += ms[2]; pn += n[2]
    acc_ms = accept_time(w, 10)
    try:
        m_us, ma_us = mask_time(w, 10)
        constrained = {"workload": f"one allowed-token set per target row ({w.B * w.n} rows x "
                                   f"{w.cfg.vocab}, 5% of tokens allowed)",
                       "mask_us": m_us, "masked_accept_us": ma_us,
                       "mask_frac_of_step": m_us / (t_total / args.steps * 1e6)}
    except Exception as exc:
        constrained = {"unavailable": str(exc).splitlines()[0][:200]}
    try:
        gctl = gamma_ctl_probe(w, accepted / max(1, args.steps * args.batch * args.gamma),
                               t_total / args.steps * 1e3)
    except Exception as exc:
        gctl = {"unavailable": str(exc).splitlines()[0][:200]}
    try:
        paged = time_paged(w, max(5, args.steps // 2))
    except Exception as exc:
        paged = {"unavailable": str(exc).splitlines()[0][:200]}
    try:
        tree = time_tree(w, max(5, args.steps // 2)) if w.n <= 8 else None
    except Exception as exc:
        tree = {"unavailable": str(exc).splitlines()[0][:200]}
    hbm, _, src = peaks()
    # launches of this library's kernels per step: the forward's (one
    # persistent kernel, or embedding + per-step GEMM / attention kernels),
    # then accept and the rollback
    launches = int(round((gn + an + pn) / k_inst)) + (1 if gn else 0) + 2
    if pn:
        kernel, k_ms, k_n, k_bytes = "forward_kernel", pm, pn, w.forward_bytes() * pn
    else:
        kernel, k_ms, k_n, k_bytes = "gemm_tc_kernel", gm, gn, gb
    achieved = k_bytes / (k_ms / 1e3) / 1e9 if k_ms else None
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": t_total / args.steps * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic", "config": config,
        "emitted_tokens_per_s": emitted * world / t_total,
        "acceptance": accepted / max(1, args.steps * args.batch * args.gamma),
        "hbm_frac_of_8tbs": value / world / 8000.0,
        "hbm_frac_of_measured": value / world / hbm,
        "bytes_per_step": step_bytes,
        "accept_us": acc_ms * 1e3, "accept_frac_of_step": acc_ms / (t_total / args.steps * 1e3),
        "e2e": {"value": e2e_val, "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h},
        "graph": graph,
        "gpu_launches": launches * args.steps,
        "roofline": {"bound": "hbm", "achieved": achieved, "peak": hbm, "unit": "GB/s",
                     "frac": (achieved / hbm) if achieved else None,
                     "traffic": kernel_traffic(kernel),
                     "algorithmic_bytes_per_launch": k_bytes / k_n if k_n else None,
                     "kernel": kernel, "peak_source": src,
                     "launch_ms": k_ms / k_n if k_n else None},
        "clocks": clk.summary(),
    }
    line["constrained"] = constrained
    line["gamma_ctl"] = gctl
    line["paged"] = paged
    if tree is not None:
        line["tree"] = tree
    if world == 1 and not args.no_configs and args.shape == "8b" and not args.layers:
        _, tflops, _ = peaks()
        configs = {}
        steps_c = max(5, args.steps // 2)
        for name, fn in (("accept_only_v4096", lambda: config_accept_only()),
                         ("lm_head_accept", lambda: config_lm_head(hbm)),
                         ("decoder_1b", lambda: config_1b(hbm, steps_c, args.warmup)),
                         ("decoder_8b_variants", lambda: config_8b_variants(w, hbm, steps_c,
                                                                            args.warmup)),
                         ("batched_8b", lambda: config_batched(w.model, hbm, tflops or 1892.2,
                                                               steps_c, args.warmup))):
            try:
                configs[name] = fn()
            except Exception as exc:
                configs[name] = {"unavailable": str(exc).splitlines()[0][:200]}
        line["configs"] = configs
        try:
            line["parity"] = headline_parity(args.temperature, args.top_p)
        except Exception as exc:
            line["parity"] = {"unavailable": str(exc).splitlines()[0][:200]}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        smp = OracleSample(cfg, args.batch, args.gamma, args.context, args.temperature, 3)
        val, sec, k = oracle_rate(smp, 3)
        line["cpu_baseline"] = {"value": val, "unit": "GB/s", "cores": blas_threads(),
                                "kind": "oracle", "sample": f"{k} x {smp.desc}",
                                "ms_per_sample_step": sec * 1e3}
    if rank == 0:
        print(json.dumps(line))
    w.model.close()
    if world > 1:
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
