// Persistent decode forward: the whole verification pass of a decode-shaped
// batch (M = B*(gamma+1) <= 128 token rows, <= 64 query rows per KV head) in
// one cooperative kernel.
//
// Why: the pass is a stream of 15 GB of weights through HBM ([lattice] /
// [pigeon] *The idea*: one weight read scores every drafted position), cut
// into ~160 dependent steps (4 projections + attention per layer).  As
// separate kernels every boundary drains the weight stream (tail of one
// kernel, launch and pipeline fill of the next).  Here every CTA stays
// resident; the steps become phases separated by grid-wide barriers, and the
// weight producer runs ahead of them: up to all but two ring stages of the
// next phase's weight tiles stream into shared memory while the dependency
// resolves; the activation loads (which need the previous phase's output)
// wait for the barrier.
//
// Phases: EMBED, then per layer QKV -> ATT -> CMB -> O -> GU -> DOWN, then
// HEAD.  Warp roles (224 threads):
//   warp 0 lane 0  weight producer (TMA, runs ahead across phases)
//   warp 1         TMEM owner; lane 0 issues the GEMMs' tcgen05.mma
//   warps 2-5      GEMM epilogues (TMEM -> fused epilogue), embedding,
//                  attention partials (ATT: S^T and O^T as tcgen05 MMAs with
//                  TMA-loaded key blocks for head dim 128, warp-level MMAs
//                  for 64; the first key block's cached rows come early) and
//                  their merge (CMB); they arrive on the grid barrier for
//                  every phase
//   warp 6 lane 0  activation producer (TMA after each phase's barrier)
// Grid barrier: one monotonic counter; phase k is complete when it holds
// (k+1) * gridDim.x arrivals.  All waits are bounded (~2 s); a CTA that times
// out sets the status bit, drains its own copies, frees TMEM and returns.
// The file also holds the attention phase and its merge as launches of their
// own (attn_step_kernel, cmb_step_kernel) for decode passes above 128 token
// rows.
#include "attn_common.cuh"
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int kMkThreads = 224;
static_assert(sizeof(MkParams) <= 32764, "kernel parameter space");
constexpr int kAttBlockKeys = 32;   // keys per attention warp block
constexpr int kAttUnitKeys = 64;    // keys per attention work unit (2 blocks)
constexpr int kArriveBar = 2;       // named barrier of the epilogue warps for arrivals

enum PhaseKind { PH_EMBED, PH_QKV, PH_ATT, PH_CMB, PH_O, PH_GU, PH_D, PH_HEAD };
constexpr int kPhPerLayer = 6;

SPEC_DEVINL int ph_kind(int ph, int L) {
  if (ph == 0) return PH_EMBED;
  if (ph == 1 + kPhPerLayer * L) return PH_HEAD;
  return PH_QKV + (ph - 1) % kPhPerLayer;
}
SPEC_DEVINL bool is_gemm(int k) {
  return k == PH_QKV || k == PH_O || k == PH_GU || k == PH_D || k == PH_HEAD;
}

struct GPh {
  int wmap, xmap, N, K, epi, l;
};

SPEC_DEVINL GPh gph(const MkParams& P, int ph) {
  const int k = ph_kind(ph, P.L);
  const int l = k == PH_HEAD ? P.L : (ph - 1) / kPhPerLayer;
  GPh g;
  g.l = l;
  switch (k) {
    case PH_QKV: g = {4 * l + 0, 0, P.qkv_rows, P.d, EPI_QKV, l}; break;
    case PH_O: g = {4 * l + 1, 2, P.d, P.H * P.hd, EPI_RESID, l}; break;
    case PH_GU: g = {4 * l + 2, 0, 2 * P.ffn, P.d, EPI_SWIGLU, l}; break;
    case PH_D: g = {4 * l + 3, 4, P.d, P.ffn, EPI_RESID, l}; break;
    default: g = {4 * P.L, 0, P.V, P.d, EPI_STORE, l}; break;
  }
  return g;
}

// Work split of one GEMM phase.  The phase uses only the first G CTAs of the
// grid: at most one per work unit, so every CTA of the split owns units (the
// fixup counts contributors by CTA index), and at most 63 contributors per
// tile (the fixup's slot table).  CTAs past the split idle in that phase.
struct PhaseSplit {
  Partition part;
  uint32_t u0, u1;
};

SPEC_DEVINL PhaseSplit phase_split(const GPh& g, uint32_t me, uint32_t GR) {
  const uint32_t kc = static_cast<uint32_t>(g.K) / 64;
  const uint32_t tiles = static_cast<uint32_t>(g.N + 127) / 128;
  const uint32_t U = tiles * kc;
  const uint32_t G = min(min(GR, U), 63u * tiles);
  PhaseSplit s{Partition{U, G, kc}, 0u, 0u};
  if (me < G) {
    s.u0 = s.part.start(me);
    s.u1 = s.part.start(me + 1);
  }
  return s;
}

// Position in the sequence of weight tiles one CTA streams: GEMM phase, work
// unit, and the unit's (tile, K chunk).
struct WCursor {
  int ph = -1;
  uint32_t u = 0, u1 = 0, kc = 1, tile = 0, kci = 0;
  int wmap = 0;
  SPEC_DEVINL void step() {
    ++u;
    if (++kci == kc) {
      kci = 0;
      ++tile;
    }
  }
};

// Move `c` onto a unit it still has to stream; false past the last phase.
SPEC_DEVINL bool wcur_seek(const MkParams& P, WCursor& c, int nph, uint32_t me, uint32_t GR) {
  while (c.u >= c.u1) {
    if (++c.ph >= nph) return false;
    if (!is_gemm(ph_kind(c.ph, P.L))) continue;
    const GPh g = gph(P, c.ph);
    const PhaseSplit ps = phase_split(g, me, GR);
    c.kc = static_cast<uint32_t>(g.K) / 64;
    c.u = ps.u0;
    c.u1 = ps.u1;
    c.tile = c.u / c.kc;
    c.kci = c.u - c.tile * c.kc;
    c.wmap = g.wmap;
  }
  return true;
}

template <typename T>
SPEC_DEVINL const T* layer_ptr(const T* base0, long long stride, int l) {
  return reinterpret_cast<const T*>(reinterpret_cast<const char*>(base0) + stride * l);
}

// Epilogue parameters of one GEMM phase.
SPEC_DEVINL GemmParams phase_params(const MkParams& P, const GPh& g) {
  GemmParams p{};
  p.N = g.N;
  p.K = g.K;
  p.M = P.M;
  p.tok0 = 0;
  p.ntok = P.ntok;
  p.split = 1;
  p.ksub = 1;
  p.kc = g.K / 64;
  p.n_tiles = (g.N + 127) / 128;
  p.units = static_cast<long long>(p.n_tiles) * p.kc;
  p.epi = g.epi;
  p.ssq_tiles = P.d / 128;
  p.ssq_ld = P.ssq_ld;
  p.inv_d = P.inv_d;
  p.eps = P.eps;
  p.d = P.d;
  p.partials = P.partials;
  p.counters = P.counters;
  p.status = P.status;
  if (g.epi == EPI_QKV) {
    p.ssq_in = P.ssq;
    p.q = P.q;
    p.q_lo = P.q_lo;
    p.kcache = P.kc + P.layer_kv * g.l;
    p.vcache = P.vc + P.layer_kv * g.l;
    p.pos_base = P.pos_base;
    p.seq_ok = P.seq_ok;
    p.rope = P.rope;
    p.depth = P.depth;
    p.kv_table = P.kv_table;
    p.kv_max_pages = P.kv_max_pages;
    p.kv_n_pages = P.kv_n_pages;
    p.n_per_seq = P.n;
    p.H = P.H;
    p.Hkv = P.Hkv;
    p.hd = P.hd;
    p.cap = P.cap;
  } else if (g.epi == EPI_RESID) {
    p.h = P.h;
    p.hb = P.hb;
    p.hb_lo = P.hb_lo;
    p.ssq_out = P.ssq;
    const bool o_proj = g.wmap % 4 == 1;
    p.g_next = o_proj ? layer_ptr(P.g_mlp0, P.layer_stride, g.l)
                      : (g.l + 1 < P.L ? layer_ptr(P.g_attn0, P.layer_stride, g.l + 1) : P.gfinal);
  } else if (g.epi == EPI_SWIGLU) {
    p.ssq_in = P.ssq;
    p.act = P.act;
    p.act_lo = P.act_lo;
    p.ffn = P.ffn;
  } else {
    p.ssq_in = P.ssq;
    p.out = P.logits;
    p.ldo = P.V;
  }
  return p;
}

SPEC_DEVINL void fence_proxy_async() { asm volatile("fence.proxy.async.global;" ::: "memory"); }

// Wait (one thread) until `target` arrivals; bounded.
SPEC_DEVINL bool grid_wait(const unsigned* bar, unsigned target, volatile int* abort,
                           int32_t* status) {
  return wait_count(bar, target, abort, status);
}

struct MkSmem {
  uint8_t* ring;
  uint8_t* att;  // attention staging; also the epilogue exchange buffer
  uint64_t* full;
  uint64_t* empty;
  uint64_t* accfull;
  uint64_t* accempty;
  uint64_t* attbar;  // tensor-core attention MMAs done
  uint64_t* kvbar;   // [4] the attention's TMA loads: K of buffers 0, 1, then V of buffers 0, 1
  uint64_t* qbar;    // the attention's TMA load of q
  uint32_t* tmem_slot;
  int* abort;
  int* flag;
  unsigned* aseq;   // weight stages issued (read by the activation producer)
  int* open;        // last GEMM phase whose grid barrier the activation producer passed
  float* rs;
  float* red;
  int* slots;
  float* sq;        // [128] embedding partial sums
  int* qpre;        // [3][128] QKV epilogue: KV slot, rotary position, fit flag per column
  int* au;          // [8] this CTA's first attention unit (AttUnit's fields, then a valid flag),
                    // found during the QKV phase
  int* aplan;       // [kAttPlanInts] the attention's units (att_plan)
};

__host__ __device__ inline size_t mk_att_bytes(int hd) { return static_cast<size_t>(384) * hd; }
constexpr size_t kMkBarBytes = 512;
// The attention plan in shared memory: chunks per sequence [128], the units
// before each sequence [129], the position base of each sequence [128], the
// chunk length in keys of each sequence [128].
constexpr int kAttPlanInts = 516;
constexpr int kPlanNu = 0, kPlanPre = 128, kPlanLb = 257, kPlanCk = 385;
constexpr size_t kMkTail = kMkBarBytes + 256 * 4 + 64 * 4 + 64 * 4 + 128 * 4 + 384 * 4 + 8 * 4 + kAttPlanInts * 4 + 64;

SPEC_DEVINL MkSmem mk_carve(uint8_t* raw, size_t ring_bytes, int hd) {
  uintptr_t base = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023);
  MkSmem s;
  s.ring = reinterpret_cast<uint8_t*>(base);
  s.att = s.ring + ring_bytes;
  uint8_t* t = s.att + mk_att_bytes(hd);
  s.full = reinterpret_cast<uint64_t*>(t);
  s.empty = s.full + kMaxStages;
  s.accfull = s.empty + kMaxStages;
  s.accempty = s.accfull + kMkMaxAcc;
  s.attbar = s.accempty + kMkMaxAcc;
  s.kvbar = s.attbar + 1;
  s.qbar = s.kvbar + 4;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.qbar + 1);
  s.abort = reinterpret_cast<int*>(s.tmem_slot + 1);
  s.flag = s.abort + 1;
  s.aseq = reinterpret_cast<unsigned*>(s.flag + 1);
  s.open = reinterpret_cast<int*>(s.aseq + 1);
  s.rs = reinterpret_cast<float*>(t + kMkBarBytes);
  s.red = s.rs + 256;
  s.slots = reinterpret_cast<int*>(s.red + 64);
  s.sq = reinterpret_cast<float*>(s.slots + 64);
  s.qpre = reinterpret_cast<int*>(s.sq + 128);
  s.au = s.qpre + 384;
  s.aplan = s.au + 8;
  return s;
}

// Ring stages the weight producer leaves free until a GEMM phase's grid
// barrier has passed: it streams at most S - kPreFree tiles of the phase
// ahead.  A full ring of early tiles (the refill of every CTA at once) slows
// the stream-K exchange and barrier round trips that end the phase before;
// with 8 stages, two free measured best (3.54 ms a pass against 3.57 with
// none free and 3.81 with all eight free on one GB300; on another, three
// free ran 0.03 ms slower than two and one free the same as two).
constexpr int kPreFree = 2;

// The weight producer waits (bounded) until the activation producer has
// passed the grid barrier of phase ph.
SPEC_DEVINL bool open_wait(const MkSmem& sm, int ph) {
  const unsigned long long t0 = globaltimer();
  while (*reinterpret_cast<volatile int*>(sm.open) < ph) {
    if (*sm.abort) return false;
    if (globaltimer() - t0 > kWaitLimitNs) {
      *sm.abort = 1;
      return false;
    }
    __nanosleep(32);
  }
  return true;
}

// Stream-K exchange of the persistent kernel.  A tile cut over several CTAs
// is finished by the CTA holding its first unit (whose share of the tile is
// the last segment of its range); the other contributors store their fp32
// partial sums as 64-bit words (value, tag) with tag = (launch epoch << 9) |
// phase, and the finisher polls those words until every tag is the current
// one.  No fence, counter or second pass sits between a contributor's last
// MMA and the finisher's read; the epoch (a workspace word advanced once per
// launch) keeps words of an earlier launch, e.g. an earlier replay of a
// captured graph, from being taken as current.
SPEC_DEVINL unsigned long long tag_word(uint32_t tag, float v) {
  return (static_cast<unsigned long long>(tag) << 32) | __float_as_uint(v);
}

SPEC_DEVINL unsigned long long* part_word(unsigned long long* part, uint32_t c, int slot, int ntok,
                                          int col, int r) {
  return part + ((static_cast<long long>(c) * 2 + slot) * ntok + col) * kTileN + r;
}

// acc[j] (the finisher's own accumulators on entry; the finisher is the
// tile's first contributor) += the other contributors' column c0 + j
// (j < JN), added in CTA order.  CB contributors' words are in flight
// together.  False when the wait gave up (abort set).
template <int JN, int CB>
SPEC_DEVINL bool fixup_tagged(unsigned long long* part, int ntok, int c0, int r, uint32_t c_first,
                              int nc, const int* slots, float (&acc)[16], uint32_t tag,
                              volatile int* abort, int32_t* status) {
  for (int i0 = 1; i0 < nc; i0 += CB) {
    unsigned long long w[CB][JN];
    const unsigned long long* src[CB];
#pragma unroll
    for (int k = 0; k < CB; ++k) {
      const int i = i0 + k;
      const bool remote = i < nc;
      src[k] = remote ? part_word(part, c_first + static_cast<uint32_t>(i), slots[i], ntok, c0, r)
                      : nullptr;
#pragma unroll
      for (int j = 0; j < JN; ++j)
        w[k][j] = remote ? ld_relaxed_u64(src[k] + j * kTileN) : tag_word(tag, 0.f);
    }
    unsigned long long t0 = 0;
    for (;;) {
      bool ready = true;
#pragma unroll
      for (int k = 0; k < CB; ++k)
#pragma unroll
        for (int j = 0; j < JN; ++j)
          if (static_cast<uint32_t>(w[k][j] >> 32) != tag) {
            w[k][j] = ld_relaxed_u64(src[k] + j * kTileN);
            ready = false;
          }
      if (ready) break;
      if (*abort) return false;
      const unsigned long long now = globaltimer();
      if (t0 == 0) {
        t0 = now;
      } else if (now - t0 > kWaitLimitNs) {
        *abort = 1;
        set_status(status, SPEC_DEV_TIMEOUT);
        return false;
      }
    }
#pragma unroll
    for (int k = 0; k < CB; ++k)
#pragma unroll
      for (int j = 0; j < JN; ++j) acc[j] += __uint_as_float(static_cast<uint32_t>(w[k][j]));
  }
  return true;
}

// The epilogue threads' writes of a phase are published by one release: the
// CTA barrier orders every thread's writes before the arriving thread's
// release reduction (cumulative: it publishes what that thread has
// observed through the barrier).  Each thread orders its own generic-proxy writes before
// the next phase's TMA reads.
SPEC_DEVINL void phase_arrive(const MkParams& P) {
  fence_proxy_async();
  named_bar(kArriveBar, kEpiThreads);
  if (threadIdx.x == kEpiFirstThread) red_release_add(P.bar, 1u);
}

// All epilogue threads wait for phase `ph - 1` to be complete: one thread
// acquires the barrier count, the CTA barrier orders the others after it.
SPEC_DEVINL bool epi_wait(const MkParams& P, const MkSmem& sm, int ph) {
  if (threadIdx.x == kEpiFirstThread) {
    grid_wait(P.bar, static_cast<unsigned>(ph) * gridDim.x, sm.abort, P.status);
    __threadfence();
  }
  named_bar(kArriveBar, kEpiThreads);
  return *sm.abort == 0;
}

// ------------------------------------------------------------------ embed
SPEC_DEVINL void embed_phase(const MkParams& P, const MkSmem& sm) {
  const int e = threadIdx.x - kEpiFirstThread;
  if (blockIdx.x == 0) {
    for (int b = e; b < P.B; b += kEpiThreads) {
      const int L = P.len[b];
      const int32_t bad = seq_fit(L, P.n, P.cap, P.kv_table, P.kv_max_pages, P.kv_n_pages, b);
      P.pos_base[b] = L < 0 ? 0 : L;
      P.seq_ok[b] = bad ? 0 : 1;
      if (!bad)
        P.len[b] = L + P.n;
      else
        set_status(P.status, bad);
    }
  }
  const int fpt = P.d / 128;  // features per thread (a tile of 128 = 128/fpt threads)
  for (int m = blockIdx.x; m < P.M; m += gridDim.x) {
    int tok = P.tokens[m];
    if (tok < 0 || tok >= P.V) {
      if (e == 0) set_status(P.status, SPEC_DEV_BAD_TOKEN);
      tok = 0;
    }
    const uint16_t* row = P.embed + static_cast<long long>(tok) * P.d;
    float sq = 0.f;
    if (fpt % 8 == 0) {
      // batches of up to 32 features: every load issued before any store
      // (the stores could alias the loads, which would serialise them)
      for (int i0 = 0; i0 < fpt; i0 += 32) {
        const int nck = min(32, fpt - i0) / 8;
        uint4 raw[4];
        float4 gg[8];
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c < nck) {
            const int f = e * fpt + i0 + c * 8;
            raw[c] = __ldg(reinterpret_cast<const uint4*>(row + f));
            gg[2 * c] = __ldg(reinterpret_cast<const float4*>(P.g_attn0 + f));
            gg[2 * c + 1] = __ldg(reinterpret_cast<const float4*>(P.g_attn0 + f + 4));
          }
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          if (c < nck) {
            const int f = e * fpt + i0 + c * 8;
            const long long idx = static_cast<long long>(m) * P.d + f;
            const uint32_t w[4] = {raw[c].x, raw[c].y, raw[c].z, raw[c].w};
            const float g[8] = {gg[2 * c].x, gg[2 * c].y, gg[2 * c].z, gg[2 * c].w,
                                gg[2 * c + 1].x, gg[2 * c + 1].y, gg[2 * c + 1].z, gg[2 * c + 1].w};
            float x[8];
            uint32_t hi2[4], lo2[4];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              x[2 * k] = bf16lo(w[k]);
              x[2 * k + 1] = bf16hi(w[k]);
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
              const float y0 = x[2 * k] * g[2 * k], y1 = x[2 * k + 1] * g[2 * k + 1];
              const uint16_t b0 = f32_to_bf16(y0), b1 = f32_to_bf16(y1);
              hi2[k] = static_cast<uint32_t>(b0) | (static_cast<uint32_t>(b1) << 16);
              const uint16_t l0 = f32_to_bf16(y0 - bf16_to_f32(b0)), l1 = f32_to_bf16(y1 - bf16_to_f32(b1));
              lo2[k] = static_cast<uint32_t>(l0) | (static_cast<uint32_t>(l1) << 16);
            }
#pragma unroll
            for (int k = 0; k < 8; ++k) sq += x[k] * x[k];
            *reinterpret_cast<float4*>(P.h + idx) = make_float4(x[0], x[1], x[2], x[3]);
            *reinterpret_cast<float4*>(P.h + idx + 4) = make_float4(x[4], x[5], x[6], x[7]);
            *reinterpret_cast<uint4*>(P.hb + idx) = make_uint4(hi2[0], hi2[1], hi2[2], hi2[3]);
            *reinterpret_cast<uint4*>(P.hb_lo + idx) = make_uint4(lo2[0], lo2[1], lo2[2], lo2[3]);
          }
        }
      }
    } else {
      for (int i = 0; i < fpt; ++i) {
        const int f = e * fpt + i;
        const float x = bf16_to_f32(row[f]);
        const long long idx = static_cast<long long>(m) * P.d + f;
        P.h[idx] = x;
        const float y = x * P.g_attn0[f];
        const uint16_t hi = f32_to_bf16(y);
        P.hb[idx] = hi;
        P.hb_lo[idx] = f32_to_bf16(y - bf16_to_f32(hi));
        sq += x * x;
      }
    }
    sm.sq[e] = sq;
    named_bar(kArriveBar, kEpiThreads);
    if (e < fpt) {  // fpt tiles of 128 features, 128/fpt threads each, in order
      const int tpt = kEpiThreads / fpt;
      float s = 0.f;
      for (int k = 0; k < tpt; ++k) s += sm.sq[e * tpt + k];
      P.ssq[static_cast<long long>(e) * P.ssq_ld + m] = s;
    }
    named_bar(kArriveBar, kEpiThreads);
  }
}

// ------------------------------------------------------------- attention
// Every sequence's keys are cut into chunks of the same length (a multiple of
// the block, 64 or 128 keys), chosen for about four units per CTA and at most
// P.att_nch chunks per sequence (the partials' slots); a unit is one chunk of
// one KV head, and the units of a batch are numbered sequence by sequence, so
// the CTAs share the keys evenly whatever the sequences' lengths (att_plan).
// A unit of the warp-level path walks its chunk in blocks of 64 keys: warp
// (slot s, query tile qt) takes keys [32 s, 32 s + 32) of every block for the
// 16 query rows of tile qt and keeps its own online softmax state; the two
// slots merge in shared memory into the unit's partial (max, sum, O).
SPEC_DEVINL int att_chunk_keys(int Tk, int nch, int unit_keys) {
  const int per = (Tk + nch - 1) / nch;
  return ((per + unit_keys - 1) / unit_keys) * unit_keys;
}
// Keys per attention block of the phase: 128 on the tensor cores, else 64.
SPEC_DEVINL int att_unit_keys(const MkParams& P) { return P.att_tc ? 128 : kAttUnitKeys; }

// Where a 64-key block of keys and values sits in shared memory: eight pieces
// of 16 rows (piece q = slot * 4 + (value ? 2 : 0) + half, slot = key / 32,
// half = key / 16 % 2), `pps` pieces per region and regions `stride` bytes
// apart.  The attention stage holds one block contiguously; while the
// attention phase runs, the ring stages' activation areas (idle between this
// CTA's last QKV MMA and the O phase's activation loads) hold a second one.
struct KVLayout {
  uint32_t base, stride;
  int pps;
  template <int HD>
  SPEC_DEVINL uint32_t piece(int q) const {
    return base + static_cast<uint32_t>(q / pps) * stride + static_cast<uint32_t>(q % pps) * 16u * HD * 2u;
  }
};

// Issue the cp.async copies of the 64-key block at kb (keys and values) into
// `lay`: `what` = 0 every row (zero fill past kend), 1 the rows this pass
// does not write (cached keys below Lb; zero fill past kend), 2 the rows this
// pass writes (keys Lb .. kend-1).
template <int HD, bool kPaged>
SPEC_DEVINL void att_load_block(const KVLayout& lay, const uint16_t* kc, const uint16_t* vc,
                                const KVMap& map, int b, int kvh, int kb, int kend, int Lb, int what,
                                int e) {
  constexpr int kCPR = HD / 8;
  for (int idx = e; idx < kAttUnitKeys * kCPR; idx += kEpiThreads) {
    const int i = idx / kCPR, c = idx % kCPR;  // key kb + i
    const int key = kb + i;
    const bool valid = key < kend;
    const bool fresh = valid && key >= Lb;
    if ((what == 1 && fresh) || (what == 2 && !fresh)) continue;
    const long long g = map.row<kPaged ? 2 : 1>(b, kvh, valid ? key : kb) + c * 8;
    const int qk = (i >> 5) * 4 + ((i >> 4) & 1);
    const uint32_t off = swz<HD>(i & 15, c);
    cp_async16(lay.piece<HD>(qk) + off, kc + g, valid ? 16 : 0);
    cp_async16(lay.piece<HD>(qk + 2) + off, vc + g, valid ? 16 : 0);
  }
}

// Attention unit of this CTA: (sequence, KV head, key chunk), or false.
struct AttUnit {
  int b, kvh, ch, Lb, kbeg, kend, nu;
};
// The plan of this pass's attention units, by the epilogue threads of every
// CTA alike (it depends on the sequences' position bases only, fixed from the
// embedding phase on): a chunk length ck for the batch (about four units a
// CTA), then per sequence its chunks c = ceil(Tk / ck), the units before it,
// its position base and its own chunk length, Tk / c rounded up to whole
// blocks.  Chunks of one length within a sequence keep the units that a CTA
// takes in turn (unit, unit + grid, ...) near one length: with one length for
// the whole batch every sequence ends in a short chunk, and where the units
// per sequence are even the CTAs of one parity took every long one.  grid:
// the CTAs of the attention phase (the merge plans with the attention's).
SPEC_DEVINL void att_plan(const MkParams& P, const MkSmem& sm, int grid) {
  const int e = threadIdx.x - kEpiFirstThread;
  int* const pl = sm.aplan;
  if (e < 32) {
    int tot = 0, mx = 0;
    for (int b = e; b < P.B; b += 32) {
      const int Lb = __ldcg(P.pos_base + b);
      const int Tk = min(Lb + P.n, P.cap);
      pl[kPlanLb + b] = Lb;
      pl[kPlanNu + b] = Tk;
      tot += Tk;
      mx = max(mx, Tk);
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      tot += __shfl_xor_sync(0xffffffffu, tot, o);
      mx = max(mx, __shfl_xor_sync(0xffffffffu, mx, o));
    }
    const int uk = att_unit_keys(P);
    const long long per = (static_cast<long long>(tot) * P.Hkv + 4ll * grid - 1) / (4ll * grid);
    int ck = static_cast<int>((per + uk - 1) / uk) * uk;
    ck = max(ck, att_chunk_keys(mx, P.att_nch, uk));  // at most att_nch chunks a sequence
    __syncwarp();
    int carry = 0;
    for (int b0 = 0; b0 < P.B; b0 += 32) {
      const int b = b0 + e;
      const int Tk = b < P.B ? pl[kPlanNu + b] : 0;
      const int c = (Tk + ck - 1) / ck;
      // c chunks of ckb <= ck keys: (c - 1) * ckb < Tk <= c * ckb
      const int ckb = c > 0 ? ((Tk + c - 1) / c + uk - 1) / uk * uk : uk;
      int x = c * P.Hkv;  // inclusive scan of the units over the 32 sequences
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (e >= o) x += y;
      }
      if (b < P.B) {
        pl[kPlanNu + b] = c;
        pl[kPlanPre + b] = carry + x - c * P.Hkv;
        pl[kPlanCk + b] = ckb;
      }
      carry += __shfl_sync(0xffffffffu, x, 31);
    }
    if (e == 0) pl[kPlanPre + P.B] = carry;
  }
  named_bar(kArriveBar, kEpiThreads);
}

SPEC_DEVINL int att_units(const MkSmem& sm, const MkParams& P) { return sm.aplan[kPlanPre + P.B]; }

SPEC_DEVINL bool att_unit(const MkParams& P, const MkSmem& sm, int unit, AttUnit& u) {
  const int* pl = sm.aplan;
  if (unit >= pl[kPlanPre + P.B]) return false;
  int lo = 0, hi = P.B - 1;  // the last sequence whose units start at or before this one
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pl[kPlanPre + mid] <= unit)
      lo = mid;
    else
      hi = mid - 1;
  }
  const int r = unit - pl[kPlanPre + lo], nu = pl[kPlanNu + lo], ck = pl[kPlanCk + lo];
  u.b = lo;
  u.kvh = r / nu;
  u.ch = r - u.kvh * nu;
  u.Lb = pl[kPlanLb + lo];
  const int Tk = min(u.Lb + P.n, P.cap);
  u.kbeg = u.ch * ck;
  u.kend = min(u.kbeg + ck, Tk);
  u.nu = nu;
  return u.kbeg < u.kend;
}

SPEC_DEVINL KVLayout att_stage_layout(const MkSmem& sm, int hd) {
  // [q hi 32 rows | q lo 32 rows | block]
  return KVLayout{smem_u32(sm.att) + 64u * hd * 2u, 0u, 8};
}

// Load the cached keys / values of the first 64-key block of this CTA's first
// attention unit of layer l (they do not depend on the pass), early: the
// attention stage is not used by the GEMM phases before the attention phase
// beyond the epilogue exchange buffer and the QKV bookkeeping, which sit in
// the q area.
template <int HD, bool kPaged>
SPEC_DEVINL void att_prefetch(const MkParams& P, const MkSmem& sm, int l) {
  const int e = threadIdx.x - kEpiFirstThread;
  AttUnit u;
  if (!att_unit(P, sm, blockIdx.x, u)) return;
  const KVMap map{P.kv_table, P.kv_max_pages, P.kv_n_pages, P.Hkv, P.cap, HD};
  att_load_block<HD, kPaged>(att_stage_layout(sm, HD), P.kc + P.layer_kv * l, P.vc + P.layer_kv * l, map, u.b,
                     u.kvh, u.kbeg, u.kend, u.Lb, 1, e);
}

// One 64-key block of a unit for this warp's 32 keys (slot) and 16 query rows
// (qt): scores with q as bf16 hi/lo, the online softmax, P (hi/lo) times V.
template <int HD>
SPEC_DEVINL void att_block(const MkParams& P, const KVLayout& lay, uint32_t aQ, uint32_t aQlo, int kb,
                           int kend, int Lb, int b, int R, int G, int rbase, int slot, int qt, int lane,
                           float (&mrow)[2], float (&lrow)[2], float (&oacc)[HD / 8][4]) {
  const int g8 = lane >> 2, t4 = lane & 3;
  const int k0 = kb + slot * kAttBlockKeys;
  if (k0 >= kend) return;
  const uint32_t kp[2] = {lay.piece<HD>(slot * 4), lay.piece<HD>(slot * 4 + 1)};
  const uint32_t vp[2] = {lay.piece<HD>(slot * 4 + 2), lay.piece<HD>(slot * 4 + 3)};
  float sacc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < HD / 16; ++kk) {
    uint32_t a0, a1, a2, a3, q0, q1, q2, q3;
    const int qrow = qt * 16 + (lane & 15);
    ldsm_x4(aQ + swz<HD>(qrow, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
    ldsm_x4(aQlo + swz<HD>(qrow, kk * 2 + (lane >> 4)), q0, q1, q2, q3);
#pragma unroll
    for (int np = 0; np < 2; ++np) {
      const int key = (lane & 7) + ((lane >> 4) << 3);
      uint32_t b0, b1, b2, b3;
      ldsm_x4(kp[np] + swz<HD>(key, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
      mma_bf16(sacc[np * 2], a0, a1, a2, a3, b0, b1);
      mma_bf16(sacc[np * 2 + 1], a0, a1, a2, a3, b2, b3);
      mma_bf16(sacc[np * 2], q0, q1, q2, q3, b0, b1);
      mma_bf16(sacc[np * 2 + 1], q0, q1, q2, q3, b2, b3);
    }
  }
#pragma unroll
  for (int hr = 0; hr < 2; ++hr) {
    const int r = rbase + qt * 16 + g8 + hr * 8;  // the query row of the unit
    const bool rv = r < R;
    const int jn = rv ? r / G : 0;
    const uint64_t am = (P.anc && rv) ? __ldg(P.anc + static_cast<long long>(b) * P.n + jn) : 0ull;
    float mx = -INFINITY;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const int kabs = k0 + nt * 8 + t4 * 2 + x;
        const bool ok = rv && kabs < kend && key_visible(kabs, Lb, jn, P.anc, am);
        const float v = ok ? sacc[nt][hr * 2 + x] * P.scale_log2 : -INFINITY;
        sacc[nt][hr * 2 + x] = v;
        mx = fmaxf(mx, v);
      }
    }
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
    const float mn = fmaxf(mrow[hr], mx);
    const float alpha = mrow[hr] == -INFINITY ? 0.f : exp2f(mrow[hr] - mn);
    float sum = 0.f;
#pragma unroll
    for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const float pe = mn == -INFINITY ? 0.f : exp2f(sacc[nt][hr * 2 + x] - mn);
        sacc[nt][hr * 2 + x] = pe;
        sum += pe;
      }
    }
    sum += __shfl_xor_sync(0xffffffffu, sum, 1);
    sum += __shfl_xor_sync(0xffffffffu, sum, 2);
    mrow[hr] = mn;
    lrow[hr] = lrow[hr] * alpha + sum;
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd) {
      oacc[nd][hr * 2] *= alpha;
      oacc[nd][hr * 2 + 1] *= alpha;
    }
  }
#pragma unroll
  for (int k2 = 0; k2 < 2; ++k2) {
    const uint32_t a0 = pack_bf16x2(sacc[2 * k2][0], sacc[2 * k2][1]);
    const uint32_t a1 = pack_bf16x2(sacc[2 * k2][2], sacc[2 * k2][3]);
    const uint32_t a2 = pack_bf16x2(sacc[2 * k2 + 1][0], sacc[2 * k2 + 1][1]);
    const uint32_t a3 = pack_bf16x2(sacc[2 * k2 + 1][2], sacc[2 * k2 + 1][3]);
    const uint32_t p0 = pack_bf16x2(sacc[2 * k2][0] - bf16lo(a0), sacc[2 * k2][1] - bf16hi(a0));
    const uint32_t p1 = pack_bf16x2(sacc[2 * k2][2] - bf16lo(a1), sacc[2 * k2][3] - bf16hi(a1));
    const uint32_t p2 = pack_bf16x2(sacc[2 * k2 + 1][0] - bf16lo(a2), sacc[2 * k2 + 1][1] - bf16hi(a2));
    const uint32_t p3 = pack_bf16x2(sacc[2 * k2 + 1][2] - bf16lo(a3), sacc[2 * k2 + 1][3] - bf16hi(a3));
#pragma unroll
    for (int dn = 0; dn < HD / 16; ++dn) {
      uint32_t b0, b1, b2, b3;
      ldsm_x4_t(vp[k2] + swz<HD>(lane & 15, dn * 2 + (lane >> 4)), b0, b1, b2, b3);
      mma_bf16(oacc[2 * dn], a0, a1, a2, a3, b0, b1);
      mma_bf16(oacc[2 * dn + 1], a0, a1, a2, a3, b2, b3);
      mma_bf16(oacc[2 * dn], p0, p1, p2, p3, b0, b1);
      mma_bf16(oacc[2 * dn + 1], p0, p1, p2, p3, b2, b3);
    }
  }
}

// The attention phase: every unit (sequence b, KV head, key chunk) runs its
// chunk for the n x G query rows of the KV head's group; its partial (max,
// sum, O) goes to the chunk partials, merged by the next phase.  Block 0's
// cached rows were loaded early; block 1 goes to the ring stages' activation
// areas at once, so both blocks' copies are in flight with q's.
// Merge the chunk partials of every query row by log-sum-exp into the
// attention output (bf16 hi/lo).  One warp per (sequence, KV head, row,
// 64-dimension group): each lane owns two adjacent dimensions (float2
// loads), so every partial load of a lane is in flight at once and a decode
// batch needs at most one item per warp (8 KV heads x 20 rows x 2 groups at
// batch 1, against 608 warps).
template <int HD>
SPEC_DEVINL void cmb_phase(const MkParams& P, const MkSmem& sm) {
  const int e = threadIdx.x - kEpiFirstThread;
  const int w = e >> 5, lane = e & 31;
  const int G = P.H / P.Hkv;
  const int R = P.n * G;
  const int qdim = P.H * HD;
  const int nch = P.att_nch;
  constexpr int kDG = HD / 64;
  const int items = P.B * P.Hkv * R * kDG;
  const float2* mlp = reinterpret_cast<const float2*>(P.att_ml);
  for (int it = blockIdx.x * 4 + w; it < items; it += gridDim.x * 4) {
    const int dg = it % kDG;
    const int r = (it / kDG) % R;
    const int kvh = (it / (kDG * R)) % P.Hkv;
    const int b = it / (kDG * R * P.Hkv);
    const int nu = sm.aplan[kPlanNu + b];
    const long long ubase = (static_cast<long long>(b) * P.Hkv + kvh) * nch;
    const float2* ob = reinterpret_cast<const float2*>(P.att_o + (ubase * kMkAttRows + r) * HD + dg * 64) + lane;
    float2 acc = make_float2(0.f, 0.f);
    float lsum = 0.f, m = -INFINITY;
    for (int u0 = 0; u0 < nu; u0 += 32) {
      // lane k holds unit u0 + k's (max, sum); the o loads of the 32 units
      // below do not depend on them
      const int cnt = min(32, nu - u0);
      const float2 mv = lane < cnt ? __ldcg(&mlp[(ubase + u0 + lane) * kMkAttRows + r]) : make_float2(-INFINITY, 0.f);
      float2 ov[32];
#pragma unroll
      for (int k = 0; k < 32; ++k)
        ov[k] = k < cnt ? __ldcg(ob + static_cast<long long>(u0 + k) * kMkAttRows * HD / 2) : make_float2(0.f, 0.f);
      const float mb = warp_max(mv.x);
      const float mn = fmaxf(m, mb);
      const float scale = m == -INFINITY ? 0.f : exp2f(m - mn);
      const float wgt = mv.x == -INFINITY ? 0.f : exp2f(mv.x - mn);
      float ax = 0.f, ay = 0.f;
#pragma unroll
      for (int k = 0; k < 32; ++k) {
        const float wk = __shfl_sync(0xffffffffu, wgt, k);
        ax += wk * ov[k].x;
        ay += wk * ov[k].y;
      }
      acc.x = acc.x * scale + ax;
      acc.y = acc.y * scale + ay;
      lsum = lsum * scale + warp_sum(wgt * mv.y);
      m = mn;
    }
    const int j = r / G, g = r % G;
    const long long off =
        (static_cast<long long>(b) * P.n + j) * qdim + (kvh * G + g) * HD + dg * 64 + 2 * lane;
    const float o0 = acc.x / lsum, o1 = acc.y / lsum;
    const uint16_t h0 = f32_to_bf16(o0), h1 = f32_to_bf16(o1);
    *reinterpret_cast<uint32_t*>(P.o + off) = static_cast<uint32_t>(h0) | (static_cast<uint32_t>(h1) << 16);
    const uint16_t l0 = f32_to_bf16(o0 - bf16_to_f32(h0)), l1 = f32_to_bf16(o1 - bf16_to_f32(h1));
    *reinterpret_cast<uint32_t*>(P.o_lo + off) = static_cast<uint32_t>(l0) | (static_cast<uint32_t>(l1) << 16);
  }
}

template <int HD, bool kPaged>
SPEC_DEVINL void att_phase(const MkParams& P, const MkSmem& sm, int l, uint32_t sbytes) {
  const int e = threadIdx.x - kEpiFirstThread;
  const int w = e >> 5, lane = e & 31;
  const int slot = w >> 1, qt = w & 1;
  const int G = P.H / P.Hkv;
  const int R = P.n * G;
  const int qdim = P.H * HD;
  constexpr int kRowB = HD * 2;
  constexpr int kCPR = HD / 8;
  const uint32_t aQ = smem_u32(sm.att), aQlo = aQ + 32 * kRowB;
  const KVLayout stage_lay = att_stage_layout(sm, HD);
  // the second block in the ring stages' activation areas, when they hold it
  const int act_pps = (2 * P.ntok * 128) / (16 * kRowB);
  const bool two = act_pps > 0 && P.stages * act_pps >= 8;
  const KVLayout act_lay{smem_u32(sm.ring) + kATileBytes, sbytes, act_pps > 0 ? act_pps : 1};
  float* merge = reinterpret_cast<float*>(sm.att);  // [2 tiles][16][HD], reuses the q area
  const uint16_t* kc = P.kc + P.layer_kv * l;
  const uint16_t* vc = P.vc + P.layer_kv * l;
  const KVMap map{P.kv_table, P.kv_max_pages, P.kv_n_pages, P.Hkv, P.cap, HD};
  const int nch = P.att_nch;
  const int units = att_units(sm, P);
  const int g8 = lane >> 2, t4 = lane & 3;
  for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
    AttUnit u;
    if (!att_unit(P, sm, unit, u)) continue;  // uniform across the CTA
    // query rows in passes of 32 (two tiles of 16); the unit's key blocks
    // are loaded again for each pass
    for (int rbase = 0; rbase < R; rbase += 32) {
    const bool first = unit == static_cast<int>(blockIdx.x) && rbase == 0;
    // block 0: the cached rows were prefetched for the first unit; block 1
    // into the activation areas at once
    att_load_block<HD, kPaged>(stage_lay, kc, vc, map, u.b, u.kvh, u.kbeg, u.kend, u.Lb, first ? 2 : 0, e);
    const bool staged1 = two && u.kbeg + kAttUnitKeys < u.kend;
    if (staged1)
      att_load_block<HD, kPaged>(act_lay, kc, vc, map, u.b, u.kvh, u.kbeg + kAttUnitKeys, u.kend, u.Lb, 0, e);
    // q (hi, lo) rows rbase .. rbase + 31 with async copies (zero rows past R)
    for (int idx = e; idx < 32 * kCPR; idx += kEpiThreads) {
      const int r = idx / kCPR, c = idx % kCPR;
      const int rr = rbase + r;
      const bool valid = rr < R;
      const int j = valid ? rr / G : 0, g = valid ? rr % G : 0;
      const long long off = (static_cast<long long>(u.b) * P.n + j) * qdim + (u.kvh * G + g) * HD + c * 8;
      cp_async16(aQ + swz<HD>(r, c), P.q + off, valid ? 16 : 0);
      cp_async16(aQlo + swz<HD>(r, c), P.q_lo + off, valid ? 16 : 0);
    }
    const bool active = rbase + qt * 16 < R;
    float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
    float oacc[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    cp_async_wait_all();
    named_bar(kArriveBar, kEpiThreads);
    for (int kb = u.kbeg, bi = 0; kb < u.kend; kb += kAttUnitKeys, ++bi) {
      const bool in_act = staged1 && bi == 1;
      if (bi > 0 && !in_act) {
        named_bar(kArriveBar, kEpiThreads);  // the stage's previous block consumed
        att_load_block<HD, kPaged>(stage_lay, kc, vc, map, u.b, u.kvh, kb, u.kend, u.Lb, 0, e);
        cp_async_wait_all();
        named_bar(kArriveBar, kEpiThreads);
      }
      if (active)
        att_block<HD>(P, in_act ? act_lay : stage_lay, aQ, aQlo, kb, u.kend, u.Lb, u.b, R, G, rbase, slot,
                      qt, lane, mrow, lrow, oacc);
    }
    // ---- merge the two slots: slot 1 through shared memory
    named_bar(kArriveBar, kEpiThreads);  // the q area becomes the merge buffer
    float* mb = merge + qt * 16 * HD;
    float* mm = sm.red + qt * 32;  // [16] max, [16] sum
    if (slot == 1 && active) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int rr = g8 + hr * 8;
#pragma unroll
        for (int nd = 0; nd < HD / 8; ++nd) {
          mb[rr * HD + nd * 8 + t4 * 2] = oacc[nd][hr * 2];
          mb[rr * HD + nd * 8 + t4 * 2 + 1] = oacc[nd][hr * 2 + 1];
        }
        if (t4 == 0) {
          mm[rr] = mrow[hr];
          mm[16 + rr] = lrow[hr];
        }
      }
    }
    named_bar(kArriveBar, kEpiThreads);
    if (slot == 0 && active) {
      const long long ubase = (static_cast<long long>(u.b) * P.Hkv + u.kvh) * nch + u.ch;
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int rr = g8 + hr * 8;
        const int r = rbase + qt * 16 + rr;
        const float m1 = mm[rr], l1 = mm[16 + rr];
        const float mn = fmaxf(mrow[hr], m1);
        const float s0 = mrow[hr] == -INFINITY ? 0.f : exp2f(mrow[hr] - mn);
        const float s1 = m1 == -INFINITY ? 0.f : exp2f(m1 - mn);
        if (r < R) {
          float* dst = P.att_o + (ubase * kMkAttRows + r) * HD;
#pragma unroll
          for (int nd = 0; nd < HD / 8; ++nd) {
            const int c = nd * 8 + t4 * 2;
            float2 v;
            v.x = oacc[nd][hr * 2] * s0 + mb[rr * HD + c] * s1;
            v.y = oacc[nd][hr * 2 + 1] * s0 + mb[rr * HD + c + 1] * s1;
            __stcg(reinterpret_cast<float2*>(dst + c), v);
          }
          if (t4 == 0) {
            float2 ml;
            ml.x = mn;
            ml.y = lrow[hr] * s0 + l1 * s1;
            __stcg(reinterpret_cast<float2*>(P.att_ml + (ubase * kMkAttRows + r) * 2), ml);
          }
        }
      }
    }
    named_bar(kArriveBar, kEpiThreads);  // shared memory free for the next pass
    }
  }
  // the activation areas go back to the TMA loads of the O phase
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------- attention on tcgen05
// The attention phase on the tensor cores (head dim 128).  Per 128-key block
// of a unit (sequence b, KV head, key chunk) and per pass of 32 query rows:
//   S^T[key][r] = K[key] . q[r]     one UMMA chain, M = 128 keys, N = 64 (the
//                                   32 rows' q as bf16 hi rows, then lo rows)
//   P[r][key]   = 2^(s - m_r)       written as bf16 hi / lo columns of the
//                                   next B operand, MN-major: one 128-byte
//                                   row of 64 values per key
//   O^T[d][r]   = sum_key V[key][d] P[r][key]
//                                   M = 128 dims: A = V^T, read MN-major
//                                   from the V tile as stored ([key][dim])
// with an online softmax over the unit's blocks.  Each epilogue thread owns
// TMEM lane t (t = its warp quarter * 32 + lane): key t of S^T, then
// dimension t of O^T; the per-row max and sum over the 128 keys are warp
// transpose-reductions (31 shuffles for 32 rows) and a 4-warp merge in
// shared memory; each thread stores its key's 64 P values as eight 16-byte
// words.  The first epilogue thread issues the MMAs (the GEMM issuer
// is idle between GEMM phases) and commits them to the attention barrier.
// Shared memory: q [64][128] and K [128][128] in the attention stage, P over
// K's first half once the scores are in TMEM; V in F ring stages that the
// weight producer leaves free until the O phase's grid barrier has passed (it
// issues at most S - F of that phase's tiles before it, and nothing of a
// later phase).  With stages of 32 KB or more, F = 3: V, and a second K and V
// buffer, so that a block's K and V copies fly while the block before it is
// computed; below that F = 2 (V's two halves) and one buffer.  The cached
// rows of a CTA's first block come early: K's during the QKV phase (the
// attention stage's K area is not used by the GEMM phases), V's once the
// CTA's last QKV accumulator has been read (its F stages are then free).
constexpr int kTcKeys = 128;
constexpr int kTcRows = 32;

// Ring stages of sbytes bytes kept free for the attention phase.
__host__ __device__ inline int tc_free_stages(uint32_t sbytes) { return sbytes >= 2u * 16384u ? 3 : 2; }

// Byte offset of 16-byte chunk c (of 8 in a 128-byte row) of row i in a
// K-major tile with 128-byte swizzling: 8-row groups of 1024 bytes.
SPEC_DEVINL uint32_t sw128_off(int i, int c) {
  return static_cast<uint32_t>((i >> 3) * 1024 + (i & 7) * 128 + ((c ^ (i & 7)) << 4));
}

// Reduce 32 values per lane over the warp's lanes with op; afterwards lane l
// holds the result for value l (recursive halving: 31 shuffles).
template <class Op>
SPEC_DEVINL float warp_transpose_reduce(float (&v)[32], Op op) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 16, n = 32; o >= 1; o >>= 1, n >>= 1) {
    const bool upper = (lane & o) != 0;
#pragma unroll
    for (int i = 0; i < n / 2; ++i) {
      const float send = upper ? v[i] : v[i + n / 2];
      const float keep = upper ? v[i + n / 2] : v[i];
      v[i] = op(keep, __shfl_xor_sync(0xffffffffu, send, o));
    }
  }
  return v[0];
}

SPEC_DEVINL void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,"
      "%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory descriptor with explicit leading / stride byte offsets
// (128-byte swizzle).  K-major tiles use (16, 1024); the MN-major V^T view
// uses (distance between its two 64-dimension sub-tiles, 1024).
SPEC_DEVINL uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Where the attention phase keeps its operands (shared addresses).
struct TcLayout {
  uint32_t q;             // [64 rows][128] as 2 sub-tiles [64][64] (8 KB apart)
  uint32_t k[2];          // [128 keys][128] as 2 sub-tiles [128][64] (16 KB apart); P
                          // [128 keys][64 rows] (one 128-byte swizzled row per key) over the first
  uint32_t v0[2], v1[2];  // the V tile's two [128 keys][64 dims] sub-tiles (v0 < v1)
  bool db;                // two buffers (else [1] = [0])
};

// n_issued: weight tiles this CTA streamed before the O phase of this layer
// (the O phase's first tile goes to ring stage n_issued % S).
SPEC_DEVINL TcLayout tc_layout(const MkSmem& sm, uint32_t sbytes, int S, uint32_t n_issued) {
  const int F = tc_free_stages(sbytes);
  const int f0 = static_cast<int>((n_issued + static_cast<uint32_t>(S - F)) % static_cast<uint32_t>(S));
  TcLayout t;
  t.q = smem_u32(sm.att);
  t.k[0] = t.q + 16384;
  const uint32_t ring = smem_u32(sm.ring);
  const auto stage = [&](int i) { return ring + static_cast<uint32_t>((f0 + i) % S) * sbytes; };
  if (F == 3) {  // V, then the second K, then the second V: one stage each
    t.db = true;
    t.v0[0] = stage(0);
    t.k[1] = stage(1);
    t.v0[1] = stage(2);
    t.v1[0] = t.v0[0] + 16384u;
    t.v1[1] = t.v0[1] + 16384u;
  } else {  // V's halves in two stages, the lower address first
    t.db = false;
    t.v0[0] = min(stage(0), stage(1));
    t.v1[0] = max(stage(0), stage(1));
    t.k[1] = t.k[0];
    t.v0[1] = t.v0[0];
    t.v1[1] = t.v1[0];
  }
  return t;
}

// cp.async of rows [i0, i1) of the 128 keys x 128 dims of one cache's block
// kb into [key][dim] sub-tiles (sub0, sub0 + stride), rows past kend zero
// filled.  Thread e moves 16-byte chunk e % 16 of rows e / 16 + 8k: its
// destinations are 1024 bytes apart.
template <bool kPaged>
SPEC_DEVINL void tc_load_range(uint32_t sub0, uint32_t stride, const uint16_t* cache, const KVMap& map, int b,
                               int kvh, int kb, int kend, int i0, int i1, int e) {
  const int c = e & 15, ir = e >> 4;
  const uint32_t dst0 = sub0 + static_cast<uint32_t>(c >> 3) * stride + sw128_off(ir, c & 7);
  for (int i = ir + (i0 > ir ? ((i0 - ir + 7) & ~7) : 0); i < i1; i += 8) {
    const int key = kb + i;
    const bool valid = key < kend;
    const long long g = map.row<kPaged ? 2 : 1>(b, kvh, valid ? key : kb) + c * 8;
    cp_async16(dst0 + static_cast<uint32_t>(i >> 3) * 1024u, cache + g, valid ? 16 : 0);
  }
}

// The block's rows by `what` (as in att_load_block): 0 every row (zero fill
// past kend); 1 the rows this pass does not write (cached keys, and the zero
// fill); 2 the rows it writes (keys Lb .. kend - 1).
template <bool kPaged>
SPEC_DEVINL void tc_load_rows(uint32_t sub0, uint32_t stride, const uint16_t* cache, const KVMap& map,
                              int b, int kvh, int kb, int kend, int Lb, int what, int e) {
  const int nc = min(max(Lb - kb, 0), kTcKeys), nv = min(max(kend - kb, 0), kTcKeys);
  if (what == 0) {
    tc_load_range<kPaged>(sub0, stride, cache, map, b, kvh, kb, kend, 0, kTcKeys, e);
  } else if (what == 1) {
    tc_load_range<kPaged>(sub0, stride, cache, map, b, kvh, kb, kend, 0, nc, e);
    tc_load_range<kPaged>(sub0, stride, cache, map, b, kvh, kb, kend, nv, kTcKeys, e);
  } else {
    tc_load_range<kPaged>(sub0, stride, cache, map, b, kvh, kb, kend, nc, nv, e);
  }
}

// TMA loads of block kb of unit u's K (which 0) or V (1) cache of layer l
// into the sub-tiles s0 (dimensions 0..63) and s1 (64..127), completing on
// bar: one box of 128 rows per sub-tile, or one per 64-slot page.  Rows past
// the chunk's end hold whatever the cache holds there (tc_zero_rows clears
// V's).  One thread.
template <bool kPaged>
SPEC_DEVINL void tc_tma_kv(const MkParams& P, const AttUnit& u, int l, int kb, uint32_t s0, uint32_t s1, int which,
                           uint64_t* bar) {
  const CUtensorMap* m = &P.kvmap[which];
  const uint64_t pol = l2_policy_evict_first();
  mbar_arrive_expect_tx(bar, 2u * kTcKeys * 128u);
  if constexpr (!kPaged) {
    // (below 2^31: the launcher enables these loads only then)
    const int row = static_cast<int>(((static_cast<long long>(l) * P.B + u.b) * P.Hkv + u.kvh) * P.cap + kb);
    tma_load_2d_s(s0, m, bar, 0, row, pol);
    tma_load_2d_s(s1, m, bar, 64, row, pol);
  } else {
#pragma unroll
    for (int pg = 0; pg < 2; ++pg) {
      const int idx = min(kb / kPageSlots + pg, P.kv_max_pages - 1);
      int page = __ldg(P.kv_table + static_cast<long long>(u.b) * P.kv_max_pages + idx);
      page = page < 0 ? 0 : (page >= P.kv_n_pages ? P.kv_n_pages - 1 : page);
      const int row =
          static_cast<int>(((static_cast<long long>(l) * P.kv_n_pages + page) * P.Hkv + u.kvh) * kPageSlots);
      tma_load_2d_s(s0 + pg * kPageSlots * 128u, m, bar, 0, row, pol);
      tma_load_2d_s(s1 + pg * kPageSlots * 128u, m, bar, 64, row, pol);
    }
  }
}

// TMA loads of the 32 query rows rbase .. rbase + 31 of unit u (token-major,
// G heads a token; rows past the sequence are other tokens or zero): hi to
// tile rows 0..31, lo to 32..63.  One thread.
SPEC_DEVINL void tc_tma_q(const MkParams& P, const AttUnit& u, int rbase, uint32_t q, uint64_t* bar) {
  const int G = P.H / P.Hkv;
  const uint64_t pol = l2_policy_evict_first();
  mbar_arrive_expect_tx(bar, 4u * kTcRows * 128u);
  const int z = u.b * P.n + rbase / G, y = u.kvh * G;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    tma_load_3d_s(q + h * 8192u, &P.qmap[0], bar, 64 * h, y, z, pol);
    tma_load_3d_s(q + h * 8192u + 4096u, &P.qmap[1], bar, 64 * h, y, z, pol);
  }
}

// Zero rows nv .. 127 of a [128 keys][128 dims] tile (sub-tiles s0, s1).
SPEC_DEVINL void tc_zero_rows(uint32_t s0, uint32_t s1, int nv, int e) {
  for (int i = nv * 16 + e; i < kTcKeys * 16; i += kEpiThreads) {
    const int row = i >> 4, c = i & 15;
    const uint32_t a = (c < 8 ? s0 : s1) + static_cast<uint32_t>(row) * 128u + static_cast<uint32_t>(c & 7) * 16u;
    asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(a), "r"(0) : "memory");
  }
}

// The cached keys of this CTA's first attention block of layer l, early
// (during the QKV phase; the attention stage's K area is not used by the
// GEMM phases).
template <bool kPaged>
SPEC_DEVINL void tc_prefetch(const MkParams& P, const MkSmem& sm, int l, uint32_t& ld_pend) {
  const int e = threadIdx.x - kEpiFirstThread;
  AttUnit u;
  const bool ok = att_unit(P, sm, blockIdx.x, u);
  if (e == 0) {  // kept for the attention phase (its sequence's length is an L2 round trip)
    const int f[8] = {u.b, u.kvh, u.ch, u.Lb, u.kbeg, u.kend, u.nu, ok ? 1 : 0};
    for (int i = 0; i < 8; ++i) sm.au[i] = f[i];
  }
  if (!ok) return;
  if (P.att_tma) {  // the whole block (its fresh rows are reloaded after the barrier)
    if (e == 0) tc_tma_kv<kPaged>(P, u, l, u.kbeg, smem_u32(sm.att) + 16384, smem_u32(sm.att) + 32768, 0, &sm.kvbar[0]);
    ld_pend |= 1u;
    return;
  }
  const KVMap map{P.kv_table, P.kv_max_pages, P.kv_n_pages, P.Hkv, P.cap, 128};
  tc_load_rows<kPaged>(smem_u32(sm.att) + 16384, 16384, P.kc + P.layer_kv * l, map, u.b, u.kvh, u.kbeg,
                       u.kend, u.Lb, 1, e);
}

// The cached rows of the same block's V, once this CTA has read its last QKV
// accumulator: every MMA of the phase has then completed, and the weight
// producer writes none of the three stages that the attention phase uses.
template <bool kPaged>
SPEC_DEVINL void tc_prefetch_v(const MkParams& P, const MkSmem& sm, int l, uint32_t sbytes, uint32_t n_issued,
                               uint32_t& ld_pend) {
  const int e = threadIdx.x - kEpiFirstThread;
  AttUnit u;
  if (!att_unit(P, sm, blockIdx.x, u)) return;
  const TcLayout L = tc_layout(sm, sbytes, P.stages, n_issued);
  if (P.att_tma) {
    if (e == 0) tc_tma_kv<kPaged>(P, u, l, u.kbeg, L.v0[0], L.v1[0], 1, &sm.kvbar[2]);
    ld_pend |= 4u;
    return;
  }
  const KVMap map{P.kv_table, P.kv_max_pages, P.kv_n_pages, P.Hkv, P.cap, 128};
  tc_load_rows<kPaged>(L.v0[0], L.v1[0] - L.v0[0], P.vc + P.layer_kv * l, map, u.b, u.kvh, u.kbeg, u.kend, u.Lb, 1,
                       e);
}

SPEC_DEVINL void tc_wait(uint64_t* bar, uint32_t& parity, volatile int* abort) {
  mbar_wait(bar, parity, abort);
  parity ^= 1u;
  tc_fence_after();
}

template <bool kPaged>
// ld_par: bit i the parity of the next completion of kvbar[i] (i < 4) or
// qbar (4); ld_pend: the same bits for TMA loads issued and not yet waited.
SPEC_DEVINL void att_phase_tc(const MkParams& P, const MkSmem& sm, int l, uint32_t sbytes,
                              uint32_t n_issued, uint32_t tmem_att, uint32_t& att_par, uint32_t& ld_par,
                              uint32_t& ld_pend) {
  constexpr int HD = 128;
  const int e = threadIdx.x - kEpiFirstThread;
  const int quarter = (threadIdx.x >> 5) & 3, lane = threadIdx.x & 31;
  const int t = quarter * 32 + lane;  // this thread's TMEM lane: a key of S^T, a dim of O^T
  const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
  const int G = P.H / P.Hkv;
  const int R = P.n * G;
  const int qdim = P.H * HD;
  const TcLayout L = tc_layout(sm, sbytes, P.stages, n_issued);
  const uint16_t* kc = P.kc + P.layer_kv * l;
  const uint16_t* vc = P.vc + P.layer_kv * l;
  const KVMap map{P.kv_table, P.kv_max_pages, P.kv_n_pages, P.Hkv, P.cap, HD};
  const int nch = P.att_nch;
  const int units = att_units(sm, P);
  float* rowm = sm.rs;         // [32] running max of each row (log2 units)
  float* rowl = sm.rs + 32;    // [32] running sum
  float* alpha = sm.rs + 64;   // [32] rescale of this block
  float* red = sm.rs + 128;    // [4][32] per-warp partials
  unsigned long long* am = reinterpret_cast<unsigned long long*>(sm.qpre);  // [32] tree masks
  const uint32_t id_s = idesc_bf16(kTcKeys, 2 * kTcRows);
  // A (V^T) and B (P) both MN-major
  const uint32_t id_o = idesc_bf16(HD, 2 * kTcRows) | (1u << 15) | (1u << 16);
  // q, K and V by TMA, issued by the first epilogue thread and waited by all
  const bool tma = P.att_tma != 0;
  if (tma && e == 0) fence_proxy_async();  // this step's q and K/V rows (other CTAs' stores), then TMA reads
  const auto ld_wait = [&](int i) {
    if (mbar_wait(i < 4 ? &sm.kvbar[i] : sm.qbar, (ld_par >> i) & 1u, sm.abort)) {
      ld_par ^= 1u << i;
      ld_pend &= ~(1u << i);
    }
  };
  for (int unit = blockIdx.x; unit < units; unit += gridDim.x) {
    AttUnit u;
    if (unit == static_cast<int>(blockIdx.x)) {  // found during the QKV phase
      if (!sm.au[7]) continue;
      u = AttUnit{sm.au[0], sm.au[1], sm.au[2], sm.au[3], sm.au[4], sm.au[5], sm.au[6]};
    } else if (!att_unit(P, sm, unit, u)) {
      continue;  // uniform across the CTA
    }
    for (int rbase = 0; rbase < R; rbase += kTcRows) {
      const bool first_unit = unit == static_cast<int>(blockIdx.x) && rbase == 0;
      // q rows rbase .. rbase + 31 (zero past R): hi in tile rows 0..31, lo in
      // 32..63.  Thread e moves 16-byte chunk e % 16 of rows e / 16 + 8k of
      // both halves.
      if (tma) {
        if (e == 0) tc_tma_q(P, u, rbase, L.q, sm.qbar);
        ld_pend |= 16u;
      } else {
        const int c = e & 15;
#pragma unroll
        for (int k = 0; k < kTcRows / 8; ++k) {
          const int r = (e >> 4) + 8 * k, rr = rbase + r;
          const bool valid = rr < R;
          long long off = 0;
          if (valid) {
            const int j = rr / G, g = rr - j * G;
            off = (static_cast<long long>(u.b) * P.n + j) * qdim + (u.kvh * G + g) * HD + c * 8;
          }
          const uint32_t d = L.q + static_cast<uint32_t>(c >> 3) * 8192 + sw128_off(r, c & 7);
          cp_async16(d, P.q + off, valid ? 16 : 0);
          cp_async16(d + 4096u, P.q_lo + off, valid ? 16 : 0);  // row r + 32
        }
      }
      if (e < kTcRows) {
        const int rr = rbase + e;
        rowm[e] = -INFINITY;
        rowl[e] = 0.f;
        am[e] = (P.anc && rr < R) ? __ldg(P.anc + static_cast<long long>(u.b) * P.n + rr / G) : 0ull;
      }
      float acc[kTcRows];
#pragma unroll
      for (int r = 0; r < kTcRows; ++r) acc[r] = 0.f;
      // K and V of block kb into buffer bf, as one group of copies (the first
      // block of the CTA's first unit: its cached rows came early)
      const auto issue = [&](int kb, int bf) {
        const bool early = first_unit && kb == u.kbeg;
        if (tma) {
          if (!early) {
            if (e == 0) {
              tc_tma_kv<kPaged>(P, u, l, kb, L.k[bf], L.k[bf] + 16384, 0, &sm.kvbar[bf]);
              tc_tma_kv<kPaged>(P, u, l, kb, L.v0[bf], L.v1[bf], 1, &sm.kvbar[2 + bf]);
            }
            ld_pend |= (1u << bf) | (4u << bf);
          }
          return;
        }
        const int what = early ? 2 : 0;
        tc_load_rows<kPaged>(L.k[bf], 16384, kc, map, u.b, u.kvh, kb, u.kend, u.Lb, what, e);
        tc_load_rows<kPaged>(L.v0[bf], L.v1[bf] - L.v0[bf], vc, map, u.b, u.kvh, kb, u.kend, u.Lb, what, e);
        cp_async_commit();
      };
      if (L.db) issue(u.kbeg, 0);
      for (int kb = u.kbeg, bf = 0; kb < u.kend; kb += kTcKeys, bf ^= L.db ? 1 : 0) {
        if (!L.db) issue(kb, 0);
        if (tma) {
          ld_wait(bf);
          ld_wait(2 + bf);
          if (kb == u.kbeg) ld_wait(4);
          if (first_unit && kb == u.kbeg) {  // the early block: this step's rows now
            tc_load_rows<kPaged>(L.k[bf], 16384, kc, map, u.b, u.kvh, kb, u.kend, u.Lb, 2, e);
            tc_load_rows<kPaged>(L.v0[bf], L.v1[bf] - L.v0[bf], vc, map, u.b, u.kvh, kb, u.kend, u.Lb, 2, e);
            cp_async_wait_all();
          }
          // V rows past the chunk's end (the cache holds anything there; their
          // P is 0, and 0 times a NaN would not be)
          if (u.kend - kb < kTcKeys) tc_zero_rows(L.v0[bf], L.v1[bf], u.kend - kb, e);
        } else {
          cp_async_wait_group<0>();
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        named_bar(kArriveBar, kEpiThreads);
        if (e == 0) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < HD / 16; ++kk)
            umma_bf16(tmem_att, sdesc_sw128(L.k[bf] + (kk >> 2) * 16384 + (kk & 3) * 32, 16, 1024),
                      sdesc_sw128(L.q + (kk >> 2) * 8192 + (kk & 3) * 32, 16, 1024), id_s, kk > 0 ? 1u : 0u);
          umma_commit(sm.attbar);
        }
        // the next block's K and V fly while this one is computed (their
        // buffer's last readers, the MMAs of block kb - 128, are done)
        if (L.db && kb + kTcKeys < u.kend) issue(kb + kTcKeys, bf ^ 1);
        tc_wait(sm.attbar, att_par, sm.abort);
        // ---- scores of key kb + t for the 32 rows (hi + lo halves)
        float sv[kTcRows], hv2[kTcRows];
        tmem_ld32(tmem_att + lane_addr, sv);
        tmem_ld32(tmem_att + lane_addr + kTcRows, hv2);
        // bit r: row rbase + r may see key kb + t (a cached key, or a key of
        // this step that the row's token attends to)
        const int key = kb + t;
        uint32_t vis = 0u;
        if (key < u.kend) {
          const int nr = min(R - rbase, kTcRows);
          vis = nr >= 32 ? 0xFFFFFFFFu : (1u << nr) - 1u;
          if (key >= u.Lb) {
            const int s = key - u.Lb;  // the key's token index within the step
            if (P.anc) {
              uint32_t m = 0u;
              if (s < 64)
                for (int r = 0; r < nr; ++r) m |= static_cast<uint32_t>((am[r] >> s) & 1ull) << r;
              vis &= m;
            } else {
              // chain: row rr (token rr / G) sees token s iff rr >= s * G
              const int first = s * G - rbase;
              vis &= first <= 0 ? 0xFFFFFFFFu : (first >= 32 ? 0u : 0xFFFFFFFFu << first);
            }
          }
        }
#pragma unroll
        for (int r = 0; r < kTcRows; ++r)
          sv[r] = ((vis >> r) & 1u) ? (sv[r] + hv2[r]) * P.scale_log2 : -INFINITY;
        // ---- row maxima over the 128 keys
        float tv[kTcRows];
#pragma unroll
        for (int r = 0; r < kTcRows; ++r) tv[r] = sv[r];
        red[quarter * kTcRows + lane] = warp_transpose_reduce(tv, [](float a, float b) { return fmaxf(a, b); });
        named_bar(kArriveBar, kEpiThreads);
        if (e < kTcRows) {
          const float mb = fmaxf(fmaxf(red[e], red[kTcRows + e]), fmaxf(red[2 * kTcRows + e], red[3 * kTcRows + e]));
          const float mo = rowm[e];
          const float mn = fmaxf(mo, mb);
          alpha[e] = mo == -INFINITY ? 0.f : exp2f(mo - mn);
          rowm[e] = mn;
        }
        named_bar(kArriveBar, kEpiThreads);
#pragma unroll
        for (int r = 0; r < kTcRows; ++r) {
          const float m = rowm[r];
          sv[r] = sv[r] == -INFINITY ? 0.f : exp2f(sv[r] - m);
          tv[r] = sv[r];
        }
        red[quarter * kTcRows + lane] = warp_transpose_reduce(tv, [](float a, float b) { return a + b; });
        // ---- P row of key t: rows 0..31 as bf16 hi, then their lo parts
        {
          uint32_t w[kTcRows];
#pragma unroll
          for (int i = 0; i < kTcRows / 2; ++i) {
            w[i] = pack_bf16x2(sv[2 * i], sv[2 * i + 1]);
            w[kTcRows / 2 + i] = pack_bf16x2(sv[2 * i] - bf16lo(w[i]), sv[2 * i + 1] - bf16hi(w[i]));
          }
          const uint32_t prow = L.k[bf] + static_cast<uint32_t>(t) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c)
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(prow + ((c ^ (t & 7)) << 4)),
                         "r"(w[4 * c]), "r"(w[4 * c + 1]), "r"(w[4 * c + 2]), "r"(w[4 * c + 3])
                         : "memory");
        }
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        named_bar(kArriveBar, kEpiThreads);
        if (e < kTcRows)
          rowl[e] = rowl[e] * alpha[e] + ((red[e] + red[kTcRows + e]) + (red[2 * kTcRows + e] + red[3 * kTcRows + e]));
        if (e == 0) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kTcKeys / 16; ++kk)
            umma_bf16(tmem_att + 2 * kTcRows, sdesc_sw128(L.v0[bf] + kk * 2048, L.v1[bf] - L.v0[bf], 1024),
                      sdesc_sw128(L.k[bf] + kk * 2048, 8192, 1024), id_o, kk > 0 ? 1u : 0u);
          umma_commit(sm.attbar);
        }
        tc_wait(sm.attbar, att_par, sm.abort);
        // ---- O^T: dimension t of the 32 rows
        float ov[kTcRows], ol[kTcRows];
        tmem_ld32(tmem_att + lane_addr + 2 * kTcRows, ov);
        tmem_ld32(tmem_att + lane_addr + 3 * kTcRows, ol);
#pragma unroll
        for (int r = 0; r < kTcRows; ++r) acc[r] = acc[r] * alpha[r] + (ov[r] + ol[r]);
        tc_fence_before();
        named_bar(kArriveBar, kEpiThreads);  // operands and TMEM free for the next block
        if (*sm.abort) break;
      }
      // ---- this unit's partial for rows rbase .. rbase + 31
      const long long ubase = (static_cast<long long>(u.b) * P.Hkv + u.kvh) * nch + u.ch;
#pragma unroll
      for (int r = 0; r < kTcRows; ++r)
        if (rbase + r < R) __stcg(P.att_o + (ubase * kMkAttRows + rbase + r) * HD + t, acc[r]);
      if (e < kTcRows && rbase + e < R)
        __stcg(reinterpret_cast<float2*>(P.att_ml + (ubase * kMkAttRows + rbase + e) * 2),
               make_float2(rowm[e], rowl[e]));
      named_bar(kArriveBar, kEpiThreads);  // the row statistics free for the next pass
      if (*sm.abort) {
        cp_async_wait_all();  // a block's copies may still be in flight
        return;
      }
    }
  }
  // the ring stages go back to the TMA loads of the O phase
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// -------------------------------------------------------------- the kernel
template <int HD, bool kPaged>
__global__ void __launch_bounds__(kMkThreads, 1) forward_kernel(const __grid_constant__ MkParams P) {
  extern __shared__ uint8_t smem_raw[];
  const int nb = 2 * P.ntok;  // B rows per stage: hi rows then lo rows
  const int ncols = 2 * P.ntok;
  const uint32_t sbytes = static_cast<uint32_t>(stage_bytes(nb, 1));
  const int S = P.stages;
  const MkSmem sm = mk_carve(smem_raw, static_cast<size_t>(sbytes) * S, HD);
  const int warp = threadIdx.x >> 5;
  const uint32_t me = blockIdx.x, GR = gridDim.x;
  const int nph = 2 + kPhPerLayer * P.L;
  // GEMM accumulators in [0, nacc ncols); the attention's S^T and O^T after them
  const int nacc = P.nacc;
  const uint32_t tcols =
      tmem_cols_pow2(static_cast<uint32_t>(nacc * ncols) + (P.att_tc ? 4u * kTcRows : 0u));

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int a = 0; a < kMkMaxAcc; ++a) {
      mbar_init(&sm.accfull[a], 1);
      mbar_init(&sm.accempty[a], 4);
    }
    mbar_init(sm.attbar, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&sm.kvbar[i], 1);
    mbar_init(sm.qbar, 1);
    *sm.abort = 0;
    *sm.aseq = 0;
    *sm.open = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot, tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;

  if (warp == 0) {
    if (elect_lane0()) {
      // ------------------------------------------------- weight producer
      // Streams every GEMM phase's weight tiles of this CTA into the ring,
      // running ahead across phases: the ring's free stages limit it, and
      // before a phase's grid barrier has passed it issues at most all but
      // kPreFree stages' worth of that phase's tiles.
      const uint64_t pol_w = l2_policy_evict_first();
      uint32_t issued[kMaxStages];
      for (int s = 0; s < S; ++s) issued[s] = 0;
      uint32_t n = 0;
      int stage = 0;
      uint32_t phase = 0;
      WCursor cur;
      const int pre = S > kPreFree ? S - kPreFree : 1;
      int cur_ph = -1;
      int in_ph = 0;
      while (wcur_seek(P, cur, nph, me, GR)) {
        if (cur.ph != cur_ph) {
          cur_ph = cur.ph;
          in_ph = 0;
          // the tensor-core attention borrows ring stages until the O phase
          // has opened: nothing of the phase after it goes out before that
          if (P.att_tc && ph_kind(cur.ph, P.L) == PH_GU && !open_wait(sm, cur.ph - 1)) break;
        }
        // at most `pre` tiles of a phase before its grid barrier has passed
        // (of the O phase, tc_free_stages fewer when the attention borrows them)
        const int lim = (P.att_tc && ph_kind(cur.ph, P.L) == PH_O) ? S - tc_free_stages(sbytes) : pre;
        if (in_ph == lim && !open_wait(sm, cur.ph)) break;
        ++in_ph;
        if (n >= static_cast<uint32_t>(S) && !mbar_wait(&sm.empty[stage], phase ^ 1u, sm.abort)) break;
        uint8_t* st = sm.ring + static_cast<size_t>(stage) * sbytes;
        mbar_arrive_expect_tx(&sm.full[stage], sbytes);
        tma_load_2d(st, &P.wmap[cur.wmap], &sm.full[stage], static_cast<int>(cur.kci * kTileK),
                    static_cast<int>(cur.tile * kTileN), pol_w);
        ++issued[stage];
        ++n;
        atomicExch(sm.aseq, n);
        cur.step();
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (*sm.abort) {
        volatile int never = 0;
        for (int s = 0; s < S; ++s)
          if (issued[s]) mbar_wait(&sm.full[s], (issued[s] - 1) & 1u, &never);
      }
    }
  } else if (warp == 6) {
    if (elect_lane0()) {
      // --------------------------------------------- activation producer
      const uint64_t pol_x = l2_policy_evict_last();
      uint32_t n = 0;
      int stage = 0;
      bool ok = true;
      for (int ph = 0; ph < nph && ok; ++ph) {
        if (!is_gemm(ph_kind(ph, P.L))) continue;
        const GPh g = gph(P, ph);
        const uint32_t kc = g.K / 64;
        const PhaseSplit ps = phase_split(g, me, GR);
        const uint32_t u0 = ps.u0, u1 = ps.u1;
        if (u1 == u0) continue;
        if (!grid_wait(P.bar, static_cast<unsigned>(ph) * GR, sm.abort, P.status)) break;
        fence_proxy_async();  // the previous phase's generic-proxy writes, then TMA reads
        *reinterpret_cast<volatile int*>(sm.open) = ph;
        uint32_t kci = u0 % kc;
        for (uint32_t u = u0; u < u1; ++u) {
          // the weight producer has claimed this stage (expect_tx registered)
          const unsigned long long t0 = globaltimer();
          while (*reinterpret_cast<volatile unsigned*>(sm.aseq) <= n) {
            if (*sm.abort || globaltimer() - t0 > kWaitLimitNs) {
              *sm.abort = 1;
              ok = false;
              break;
            }
          }
          if (!ok) break;
          uint8_t* b = sm.ring + static_cast<size_t>(stage) * sbytes + kATileBytes;
          const int x = static_cast<int>(kci * kTileK);
          tma_load_2d(b, &P.xmap[g.xmap], &sm.full[stage], x, 0, pol_x);
          tma_load_2d(b + P.ntok * 128, &P.xmap[g.xmap + 1], &sm.full[stage], x, 0, pol_x);
          ++n;
          if (++kci == kc) kci = 0;
          if (++stage == S) stage = 0;
        }
      }
    }
  } else if (warp == 1) {
    if (elect_lane0()) {
      // ----------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_bf16(kTileN, ncols);
      int stage = 0;
      uint32_t phase = 0;
      int a = 0;          // accumulator buffer of the next segment
      uint32_t apar = 0;  // its use parity
      bool ok = true;
      for (int ph = 0; ph < nph && ok; ++ph) {
        if (!is_gemm(ph_kind(ph, P.L))) continue;
        const GPh g = gph(P, ph);
        const uint32_t kc = g.K / 64;
        const PhaseSplit ps = phase_split(g, me, GR);
        const uint32_t u0 = ps.u0, u1 = ps.u1;
        uint32_t u = u0;
        while (u < u1 && ok) {
          const uint32_t t = u / kc;
          const uint32_t seg_end = min(u1, (t + 1) * kc);
          if (!mbar_wait(&sm.accempty[a], apar ^ 1u, sm.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t dcol = tmem_base + static_cast<uint32_t>(a * ncols);
          for (uint32_t v = u; v < seg_end; ++v) {
            if (!mbar_wait(&sm.full[stage], phase, sm.abort)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint32_t abase = smem_u32(sm.ring + static_cast<size_t>(stage) * sbytes);
            const uint32_t bbase = abase + kATileBytes;
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk)
              umma_bf16(dcol, sdesc_k128(abase + kk * 32), sdesc_k128(bbase + kk * 32), idesc,
                        (v > u || kk > 0) ? 1u : 0u);
            umma_commit(&sm.empty[stage]);
            if (++stage == S) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (!ok) break;
          umma_commit(&sm.accfull[a]);
          u = seg_end;
          if (++a == nacc) {
            a = 0;
            apar ^= 1u;
          }
        }
      }
    }
  } else if (warp >= 2 && warp <= 5) {
    // ------------------------------------ epilogue / embedding / attention
    const int e = threadIdx.x - kEpiFirstThread;
    const int quarter = warp & 3;
    const int r = quarter * 32 + (threadIdx.x & 31);
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    Smem gs;  // the GEMM epilogue's view of shared memory
    gs.rs = sm.rs;
    gs.xbuf = reinterpret_cast<float*>(sm.att);
    gs.red = sm.red;
    gs.slots = sm.slots;
    gs.flag = sm.flag;
    int a = 0;          // accumulator buffer of the next segment
    uint32_t apar = 0;  // its use parity
    uint32_t n_issued = 0;  // weight tiles of the GEMM phases so far (this CTA)
    uint32_t att_par = 0;   // parity of the attention barrier
    uint32_t ld_par = 0, ld_pend = 0;  // the attention's TMA loads (att_phase_tc)
    const uint32_t tmem_att = tmem_base + static_cast<uint32_t>(nacc * ncols);
    unsigned long long* const part64 = reinterpret_cast<unsigned long long*>(P.partials);
    // read before this CTA arrives on the embedding phase; advanced after it
    const uint32_t epoch = *reinterpret_cast<volatile unsigned*>(P.epoch) & 0x7FFFFFu;
    for (int ph = 0; ph < nph; ++ph) {
      const int kind = ph_kind(ph, P.L);
      const uint32_t tag = (epoch << 9) | static_cast<uint32_t>(ph);
      int v_layer = -1;  // QKV phase of this layer done here: its first V block next
      if (kind == PH_EMBED) {
        embed_phase(P, sm);
      } else if (kind == PH_ATT) {
        if (!epi_wait(P, sm, ph)) break;
        if constexpr (HD == 128) {
          if (P.att_tc) {
            att_phase_tc<kPaged>(P, sm, (ph - 1) / kPhPerLayer, sbytes, n_issued, tmem_att, att_par, ld_par,
                                 ld_pend);
            if (*sm.abort) break;
          } else {
            att_phase<HD, kPaged>(P, sm, (ph - 1) / kPhPerLayer, sbytes);
          }
        } else {
          att_phase<HD, kPaged>(P, sm, (ph - 1) / kPhPerLayer, sbytes);
        }
      } else if (kind == PH_CMB) {
        if (!epi_wait(P, sm, ph)) break;
        cmb_phase<HD>(P, sm);
      } else {
        if (!epi_wait(P, sm, ph)) break;
        // every CTA read the epoch before arriving on the embedding phase
        if (ph == 1 && blockIdx.x == 0 && e == 0) *P.epoch = epoch + 1;
        const GPh g = gph(P, ph);
        const GemmParams p = phase_params(P, g);
        const uint32_t kc = g.K / 64;
        const PhaseSplit ps = phase_split(g, me, GR);
        const Partition& part = ps.part;
        const uint32_t u0 = ps.u0, u1 = ps.u1;
        n_issued += u1 - u0;
        if (p.ssq_in) {
          for (int c = e; c < p.ntok; c += kEpiThreads) {
            float s = 0.f;
            if (c < p.M)
              for (int t = 0; t < p.ssq_tiles; ++t) s += __ldcg(p.ssq_in + static_cast<long long>(t) * p.ssq_ld + c);
            sm.rs[c] = rsqrtf(s * p.inv_d + p.eps);
          }
        }
        // QKV: per token column KV slot, rotary position and fit flag
        int* const qpre = sm.qpre;
        if (p.epi == EPI_QKV) {
          att_plan(P, sm, gridDim.x);
          // this layer's first key block, early
          if constexpr (HD == 128) {
            if (P.att_tc)
              tc_prefetch<kPaged>(P, sm, g.l, ld_pend);
            else
              att_prefetch<HD, kPaged>(P, sm, g.l);
          } else {
            att_prefetch<HD, kPaged>(P, sm, g.l);
          }
          for (int c = e; c < p.ntok; c += kEpiThreads) {
            const int m = min(c, p.M - 1);
            const int b = m / p.n_per_seq, node = m - b * p.n_per_seq;
            const int base = __ldcg(p.pos_base + b);
            qpre[c] = base + node;
            qpre[128 + c] = base + (p.depth ? __ldg(p.depth + m) : node);
            qpre[256 + c] = __ldcg(p.seq_ok + b);
          }
        }
        named_bar(kEpiBar, kEpiThreads);
        uint32_t u = u0;
        while (u < u1) {
          const uint32_t t = u / kc;
          const uint32_t seg_end = min(u1, (t + 1) * kc);
          // the residual stream of this tile's rows, loaded while the MMAs run
          float hv[16];
          const bool pre_h = p.epi == EPI_RESID && p.ntok <= 16;
          const int f = static_cast<int>(t) * kTileN + r;
          if (pre_h) {
#pragma unroll
            for (int j = 0; j < 16; ++j)
              hv[j] = (j < p.M && f < p.N) ? __ldcg(p.h + static_cast<long long>(j) * p.d + f) : 0.f;
          }
          // the epilogue's other inputs, also loaded while the MMAs run
          EpiPre pre;
          pre.rolled = true;
          if (p.epi == EPI_RESID) {
            pre.have_gn = true;
            pre.gn = f < p.N ? __ldg(p.g_next + f) : 0.f;
          } else if (p.epi == EPI_QKV) {
            const int dim = f % p.hd, half = p.hd >> 1;
            pre.have_fr = true;
            pre.fr = __ldg(p.rope + (dim < half ? dim : dim - half));
            pre.qkv = qpre;
          }
          const uint32_t tacc = tmem_base + lane_addr + static_cast<uint32_t>(a * ncols);
          const uint32_t c_first = part.cta_of(t * kc);
          const uint32_t c_last = part.cta_of((t + 1) * kc - 1);
          const int nc = static_cast<int>(c_last - c_first + 1);
          const bool finisher = nc == 1 || me == c_first;
          mbar_wait(&sm.accfull[a], apar, sm.abort);
          named_bar(kEpiBar, kEpiThreads);
          if (*sm.abort) break;
          tc_fence_after();
          if (!finisher) {
            const int slot = part.slot(me, t);
            for (int c0 = 0; c0 < p.M; c0 += 16) {
              float v[16];
              load_acc(tacc, c0, p.ntok, 1, v);
              // the columns the finisher reads: 8 when at most 8 are valid, else 16
              const int jn = p.M - c0 <= 8 ? 8 : 16;
              unsigned long long* dst = part_word(part64, me, slot, p.ntok, c0, r);
#pragma unroll
              for (int j = 0; j < 16; ++j)
                if (j < jn) st_relaxed_u64(dst + j * kTileN, tag_word(tag, v[j]));
            }
          } else {
            if (nc > 1) {
              if (e < nc) sm.slots[e] = part.slot(c_first + e, t);
              named_bar(kEpiBar, kEpiThreads);
            }
            for (int c0 = 0; c0 < p.ntok; c0 += 16) {
              float acc[16];
              // wide batches: this chunk's residual values requested before
              // the contributors' words, so the two round trips overlap
              if (p.epi == EPI_RESID && !pre_h) {
#pragma unroll
                for (int j = 0; j < 16; ++j)
                  hv[j] = (c0 + j < p.M && f < p.N) ? __ldcg(p.h + static_cast<long long>(c0 + j) * p.d + f)
                                                    : 0.f;
              }
              load_acc(tacc, c0, p.ntok, 1, acc);
              if (nc > 1) {
                const bool ok = p.M - c0 <= 8 ? fixup_tagged<8, 5>(part64, p.ntok, c0, r, c_first, nc,
                                                                    sm.slots, acc, tag, sm.abort, P.status)
                                              : fixup_tagged<16, 2>(part64, p.ntok, c0, r, c_first, nc,
                                                                    sm.slots, acc, tag, sm.abort, P.status);
                if (!ok) break;
              }
              epilogue_chunk_h<kPaged ? 2 : 1>(p, gs, t, r, c0, acc, hv, p.epi == EPI_RESID, pre);
            }
          }
          tc_fence_before();
          __syncwarp();
          if ((threadIdx.x & 31) == 0) mbar_arrive(&sm.accempty[a]);
          u = seg_end;
          if (++a == nacc) {
            a = 0;
            apar ^= 1u;
          }
        }
        if (*sm.abort) break;
        if (p.epi == EPI_QKV) v_layer = g.l;
      }
      phase_arrive(P);
      if constexpr (HD == 128) {
        if (P.att_tc && v_layer >= 0) tc_prefetch_v<kPaged>(P, sm, v_layer, sbytes, n_issued, ld_pend);
      }
    }
    // after a timeout the attention's TMA loads still in flight land first
    // (bounded waits)
    if (*sm.abort && ld_pend) {
      volatile int never = 0;
      for (int i = 0; i < 5; ++i)
        if ((ld_pend >> i) & 1u) mbar_wait(i < 4 ? &sm.kvbar[i] : sm.qbar, (ld_par >> i) & 1u, &never);
    }
  }

  if (*sm.abort && threadIdx.x == 0) set_status(P.status, SPEC_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tcols);
  }
}

// The tensor-core attention (head dim 128) of one layer as launches of its
// own, for passes the persistent kernel does not take (more than 128 token
// rows): one CTA per SM runs the persistent kernel's attention phase over the
// batch's units (attn_step_kernel), then cmb_step_kernel merges the chunk
// partials.  Three ring-sized stages of kStepStageBytes hold V and the second
// K and V buffer.
constexpr uint32_t kStepStageBytes = 36864;
constexpr int kStepStages = kStepAttStages;

template <bool kPaged>
__global__ void __launch_bounds__(kMkThreads, 1) attn_step_kernel(const __grid_constant__ MkParams P, int l) {
  extern __shared__ uint8_t smem_raw[];
  const MkSmem sm = mk_carve(smem_raw, static_cast<size_t>(kStepStageBytes) * kStepStages, 128);
  const int warp = threadIdx.x >> 5;
  const int e = threadIdx.x - kEpiFirstThread;
  if (threadIdx.x == 0) {
    mbar_init(sm.attbar, 1);
    for (int i = 0; i < 4; ++i) mbar_init(&sm.kvbar[i], 1);
    mbar_init(sm.qbar, 1);
    *sm.abort = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot, 4u * kTcRows);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (e >= 0 && e < kEpiThreads) {
    att_plan(P, sm, gridDim.x);
    uint32_t att_par = 0, ld_par = 0, ld_pend = 0;
    tc_prefetch<kPaged>(P, sm, l, ld_pend);
    tc_prefetch_v<kPaged>(P, sm, l, kStepStageBytes, 0, ld_pend);
    att_phase_tc<kPaged>(P, sm, l, kStepStageBytes, 0, *sm.tmem_slot, att_par, ld_par, ld_pend);
    if (*sm.abort && ld_pend) {  // loads still in flight land first (bounded)
      volatile int never = 0;
      for (int i = 0; i < 5; ++i)
        if ((ld_pend >> i) & 1u) mbar_wait(i < 4 ? &sm.kvbar[i] : sm.qbar, (ld_par >> i) & 1u, &never);
    }
  }
  if (*sm.abort && threadIdx.x == 0) set_status(P.status, SPEC_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(*sm.tmem_slot, 4u * kTcRows);
  }
}

// The merge of attn_step_kernel's chunk partials: the persistent kernel's CMB
// phase (one warp per (sequence, KV head, row, 64 dimensions) item, a
// latency-bound chain of L2 loads) in CTAs that hold only the plan, so that
// several of them share an SM instead of the attention launch's one.
constexpr int kCmbCtasPerSm = 3;

__global__ void __launch_bounds__(kGemmThreads, kCmbCtasPerSm)
    cmb_step_kernel(const __grid_constant__ MkParams P, int att_grid) {
  extern __shared__ uint8_t smem_raw[];
  const MkSmem sm = mk_carve(smem_raw, 0, 0);
  const int e = threadIdx.x - kEpiFirstThread;
  if (e < 0) return;  // warps 0 and 1: the four warps after them take the items
  att_plan(P, sm, att_grid);
  cmb_phase<128>(P, sm);
}

}  // namespace

size_t forward_smem_bytes(int ntok, int stages, int hd) {
  return 1024 + stage_bytes(2 * ntok, 1) * stages + mk_att_bytes(hd) + kMkTail;
}

int forward_max_stages(int ntok, int hd, size_t budget) {
  const size_t fixed = 1024 + mk_att_bytes(hd) + kMkTail;
  if (budget <= fixed) return 0;
  int s = static_cast<int>((budget - fixed) / stage_bytes(2 * ntok, 1));
  return s > kMaxStages ? kMaxStages : s;
}

// Does the persistent forward run its attention on the tensor cores?  Head
// dim 128, the S^T and O^T columns beside the GEMM accumulators within TMEM,
// and a ring deep enough to lend tc_free_stages and keep one.
bool forward_att_tc(int ntok, int stages, int hd) {
  const int F = tc_free_stages(static_cast<uint32_t>(stage_bytes(2 * ntok, 1)));
  return hd == 128 && 4 * ntok + 4 * kTcRows <= 512 && stages >= F + 1;
}

// TMEM accumulator buffers of the persistent forward: as many as fit its 512
// columns (up to kMkMaxAcc) beside the attention's, so that a segment's MMAs
// need not wait for the epilogue of the segment two before it (the previous
// phase's finisher, whose epilogue ends the phase).
int forward_acc_buffers(int ntok, bool att_tc) {
  const int ncols = 2 * ntok, extra = att_tc ? 4 * kTcRows : 0;
  for (int nb = kMkMaxAcc; nb > 2; --nb)
    if (nb * ncols + extra <= 512) return nb;
  return 2;
}

// CTAs per SM the persistent forward can keep resident (0: not launchable).
int forward_ctas_per_sm(int ntok, int stages, int hd) {
  const size_t smem = forward_smem_bytes(ntok, stages, hd);
  const void* fns[2] = {hd == 128 ? reinterpret_cast<const void*>(forward_kernel<128, false>)
                                  : reinterpret_cast<const void*>(forward_kernel<64, false>),
                        hd == 128 ? reinterpret_cast<const void*>(forward_kernel<128, true>)
                                  : reinterpret_cast<const void*>(forward_kernel<64, true>)};
  const void* fn = fns[0];
  for (const void* f : fns)  // both cache layouts take the same shared memory
    if (cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) !=
        cudaSuccess)
      return 0;
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, fn, kMkThreads, smem) != cudaSuccess) return 0;
  // every resident CTA holds its accumulators in TMEM (512 columns per SM)
  const bool tc = forward_att_tc(ntok, stages, hd);
  uint32_t need = static_cast<uint32_t>(forward_acc_buffers(ntok, tc) * 2 * ntok) + (tc ? 4u * kTcRows : 0u),
           cols = 32;
  while (cols < need) cols <<= 1;
  const int by_tmem = static_cast<int>(512 / cols);
  return n < by_tmem ? n : by_tmem;
}

cudaError_t launch_forward(const MkParams& P, int grid, int hd, cudaStream_t stream) {
  const size_t smem = forward_smem_bytes(P.ntok, P.stages, hd);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kMkThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const bool paged = P.kv_table != nullptr;
  if (hd == 128)
    return paged ? cudaLaunchKernelEx(&cfg, forward_kernel<128, true>, P)
                 : cudaLaunchKernelEx(&cfg, forward_kernel<128, false>, P);
  return paged ? cudaLaunchKernelEx(&cfg, forward_kernel<64, true>, P)
               : cudaLaunchKernelEx(&cfg, forward_kernel<64, false>, P);
}


// One layer's tensor-core attention for the per-step schedule (P as for the
// persistent kernel's attention: stages = kStepStages; grid = the SM count):
// the attention launch, then the merge launch.
cudaError_t launch_attention_tc(const MkParams& P, int l, int grid, cudaStream_t stream) {
  const size_t smem = 1024 + static_cast<size_t>(kStepStageBytes) * kStepStages + mk_att_bytes(128) + kMkTail;
  const void* fn = P.kv_table ? reinterpret_cast<const void*>(attn_step_kernel<true>)
                              : reinterpret_cast<const void*>(attn_step_kernel<false>);
  static PerDevice<cudaError_t> configured;
  cudaError_t e = cudaErrorInvalidDevice;
  if (!configured.get(
          [&] {
            for (const void* f : {reinterpret_cast<const void*>(attn_step_kernel<true>),
                                  reinterpret_cast<const void*>(attn_step_kernel<false>)}) {
              const cudaError_t r =
                  cudaFuncSetAttribute(f, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
              if (r != cudaSuccess) return r;
            }
            return cudaSuccess;
          },
          &e))
    return cudaErrorInvalidDevice;
  if (e != cudaSuccess) return e;
  void* args[] = {const_cast<MkParams*>(&P), &l};
  e = cudaLaunchKernel(fn, dim3(grid), dim3(kMkThreads), args, smem, stream);
  if (e != cudaSuccess) return e;
  // (the plan's chunk length depends on the attention's grid: the merge plans
  // with it, then takes its items over kCmbCtasPerSm times as many CTAs)
  void* cargs[] = {const_cast<MkParams*>(&P), &grid};
  return cudaLaunchKernel(reinterpret_cast<const void*>(cmb_step_kernel), dim3(grid * kCmbCtasPerSm),
                          dim3(kGemmThreads), cargs, 1024 + kMkTail, stream);
}
}  // namespace spec
