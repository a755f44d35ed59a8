// Device pieces of the weight-streaming GEMM shared by the per-projection
// kernel (gemm.cu) and the persistent decode forward (forward.cu): the
// stream-K partition, stage geometry, accumulator loads and the fused
// epilogues.
#pragma once

#include "common.cuh"
#include "internal.h"

namespace spec {
namespace {

constexpr int kGemmThreads = 192;  // 6 warps: producer, MMA, 4 epilogue
constexpr int kTileN = 128;             // weight rows per tile (UMMA M)
constexpr int kTileK = 64;              // K elements per stage (one 128-byte swizzle row)
constexpr int kATileBytes = kTileN * 128;
constexpr int kMaxStages = 16;
constexpr int kEpiThreads = 128;
constexpr int kEpiBar = 1;
constexpr int kEpiFirstThread = 64;  // epilogue warps are 2..5

// Contiguous equal split of the U = n_tiles * kc work units over G CTAs
// (32-bit: the host guarantees U * G < 2^32).
struct Partition {
  uint32_t U;
  uint32_t G;
  uint32_t kc;
  __device__ uint32_t start(uint32_t c) const { return (c * U) / G; }
  __device__ uint32_t cta_of(uint32_t u) const { return ((u + 1) * G - 1) / U; }
  __device__ uint32_t tile_of(uint32_t u) const { return u / kc; }
  // Does CTA c cover units of more than one tile?
  __device__ bool multi(uint32_t c) const {
    const uint32_t s = start(c), e = start(c + 1);
    return e > s && tile_of(s) != tile_of(e - 1);
  }
  // Partial-slot CTA c uses for its contribution to tile t.
  __device__ int slot(uint32_t c, uint32_t t) const {
    return (c == cta_of(t * kc) && multi(c)) ? 1 : 0;
  }
};

struct Smem {
  uint8_t* stage_base;
  uint64_t* full;
  uint64_t* empty;
  uint64_t* accfull;
  uint64_t* accempty;
  uint32_t* tmem_slot;
  int* abort;
  int* flag;
  int* slots;    // [kMaxContrib] partial-slot index of each contributor of a tile
  float* rs;     // [256]
  float* xbuf;   // [16][128]
  float* red;    // [4][16]
};

// One stage = ksub K-sub-tiles of 64: [A_0 .. A_{ksub-1}][B_0 .. B_{ksub-1}], each
// B sub-tile holding `rows_b` token rows (hi rows, then lo rows).
__host__ __device__ inline size_t stage_bytes(int rows_b, int ksub = 1) {
  return (static_cast<size_t>(kATileBytes) + static_cast<size_t>(rows_b) * 128) * ksub;
}

constexpr size_t kTailBytes = 1024 /*barriers*/ + 256 * 4 /*rs*/ + 16 * 128 * 4 /*xbuf*/ +
                              4 * 16 * 4 /*red*/ + 64 * 4 /*slots*/ + 64;

__device__ Smem carve(uint8_t* raw, int rows_b, int stages, int ksub) {
  uintptr_t base = (reinterpret_cast<uintptr_t>(raw) + 1023) & ~static_cast<uintptr_t>(1023);
  Smem s;
  s.stage_base = reinterpret_cast<uint8_t*>(base);
  uint8_t* t = s.stage_base + stage_bytes(rows_b, ksub) * stages;
  s.full = reinterpret_cast<uint64_t*>(t);
  s.empty = s.full + kMaxStages;
  s.accfull = s.empty + kMaxStages;
  s.accempty = s.accfull + 2;
  s.tmem_slot = reinterpret_cast<uint32_t*>(s.accempty + 2);
  s.abort = reinterpret_cast<int*>(s.tmem_slot + 1);
  s.flag = s.abort + 1;
  s.rs = reinterpret_cast<float*>(t + 1024);
  s.xbuf = s.rs + 256;
  s.red = s.xbuf + 16 * 128;
  s.slots = reinterpret_cast<int*>(s.red + 4 * 16);
  return s;
}

__device__ __forceinline__ uint32_t tmem_cols_pow2(uint32_t need) {
  uint32_t c = 32;
  while (c < need) c <<= 1;
  return c;
}

__device__ __forceinline__ uint32_t tmem_cols_for(int ntok) {
  uint32_t need = 2u * static_cast<uint32_t>(ntok);
  uint32_t c = 32;
  while (c < need) c <<= 1;
  return c;
}

__device__ __forceinline__ float ldcg(const float* p) { return __ldcg(p); }
__device__ __forceinline__ int ldcg_i(const int* p) { return __ldcg(p); }

// Accumulator columns [c0, c0+16) of this thread's row.  With the stacked
// split (split == 1) the lo half of the activations sits in columns ntok..,
// added here.
__device__ __forceinline__ void load_acc(uint32_t tacc, int c0, int ntok, int split,
                                         float (&v)[16]) {
  tmem_ld16(tacc + static_cast<uint32_t>(c0), v);
  if (split == 1) {
    float lo[16];
    tmem_ld16(tacc + static_cast<uint32_t>(ntok + c0), lo);
#pragma unroll
    for (int j = 0; j < 16; ++j) v[j] += lo[j];
  }
}

// Stream-K fixup: the sum of the nc contributions (CTAs c_first .. c_first +
// nc - 1, this CTA's own in `own`) to the 16 token columns c0.. of row r of a
// tile, added in CTA order (deterministic).  The loads of kBatch contributors
// are in flight together.
template <int kBatch>
__device__ __forceinline__ void fixup_sum(const float* partials, int ntok, int c0, int r,
                                          uint32_t c_first, int nc, uint32_t me, const int* slots,
                                          const float (&own)[16], float (&acc)[16]) {
#pragma unroll
  for (int j = 0; j < 16; ++j) acc[j] = 0.f;
  for (int i0 = 0; i0 < nc; i0 += kBatch) {
    float v[kBatch][16];
#pragma unroll
    for (int k = 0; k < kBatch; ++k) {
      const int i = i0 + k;
      const uint32_t c = c_first + static_cast<uint32_t>(i);
      if (i < nc && c != me) {
        const float* src = partials + (static_cast<long long>(c) * 2 + slots[i]) * ntok * kTileN +
                           c0 * kTileN + r;
#pragma unroll
        for (int j = 0; j < 16; ++j) v[k][j] = ldcg(src + j * kTileN);
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) v[k][j] = i < nc ? own[j] : 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kBatch; ++k)
#pragma unroll
      for (int j = 0; j < 16; ++j) acc[j] += v[k][j];
  }
}

// --------------------------------------------------------------- epilogues
// Values an epilogue needs besides the accumulators, loaded ahead of it (while
// the MMAs run) by callers that can; left unset, the epilogue loads them.
struct EpiPre {
  bool have_gn = false;
  float gn = 0.f;           // EPI_RESID: the next norm's gain of this row's feature
  bool have_fr = false;
  float2 fr{};              // EPI_QKV: RoPE frequency of this row's dimension
  const int* qkv = nullptr; // EPI_QKV: shared [3][128] per token column: KV slot, rotary
                            // position, fit flag (persistent kernel, tok0 = 0)
  // The persistent kernel: the epilogues loop over the valid token columns
  // only (an unrolled 16-column body ran its invalid columns predicated),
  // their operands staged in the exchange buffer ([2][16][128] floats).
  bool rolled = false;
};

// sin and cos of the rotary angle of position pos for a dimension whose
// frequency is fr.x + fr.y turns per position (hi + lo): pos * fr.x = t + terr
// exactly (an fma gives the product's rounding error), whole turns are
// removed exactly (t - rint(t) is representable), and the hardware sine and
// cosine run on the reduced angle, |angle| <= pi (+ a few ulps), where their
// absolute error is about 2^-21.4.  The angle so keeps ~1e-6 absolute accuracy
// at any cached position; an unreduced fp32 angle of thousands of radians
// would lose ~|angle| * 2^-22 to its own rounding.
SPEC_DEVINL void rope_sincos(int pos, float2 fr, float* sn, float* cs) {
  const float fp = static_cast<float>(pos);
  const float t = fp * fr.x;
  const float terr = fmaf(fp, fr.x, -t) + fp * fr.y;
  const float frac = (t - rintf(t)) + terr;
  __sincosf(6.28318530717958648f * frac, sn, cs);
}

// Apply the epilogue to 16 token columns [c0, c0+16) of this thread's row.
// With have_h the residual-stream values of these columns were loaded
// beforehand (hv); otherwise the residual epilogue loads them.
// kKV: the KV cache layout of the QKV epilogue's appends (KVMap::row).
template <int kKV = 0>
__device__ void epilogue_chunk_h(const GemmParams& p, const Smem& sm, uint32_t tile, int r, int c0,
                                 const float (&acc)[16], const float (&hv_in)[16], bool have_h,
                                 const EpiPre& pre) {
  const int f = static_cast<int>(tile) * kTileN + r;  // weight row = output feature
  const int e = threadIdx.x - kEpiFirstThread;
  float v[16];
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    const int m = p.tok0 + c0 + j;
    v[j] = acc[j] * (p.ssq_in ? sm.rs[c0 + j] : 1.0f);
    (void)m;
  }
  if (p.epi == EPI_STORE) {
    if (f < p.N) {
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        const int m = p.tok0 + c0 + j;
        if (m < p.M) p.out[static_cast<long long>(m) * p.ldo + f] = v[j];
      }
    }
    return;
  }
  if (p.epi == EPI_RESID && pre.rolled) {
    // this thread's values and residual rows go to its own slots of the
    // exchange buffer; the loop over the valid columns reads them back
    float* xv = sm.xbuf;
    float* xh = sm.xbuf + 16 * kTileN;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      xv[j * kTileN + r] = v[j];
      xh[j * kTileN + r] = hv_in[j];
    }
    const bool fok = f < p.N;
    const int jn = min(16, p.M - p.tok0 - c0);
#pragma unroll 1
    for (int j = 0; j < jn; ++j) {
      const float hn = xh[j * kTileN + r] + xv[j * kTileN + r];
      if (fok) {
        const long long idx = static_cast<long long>(p.tok0 + c0 + j) * p.d + f;
        p.h[idx] = hn;
        const float x = hn * pre.gn;
        const uint16_t hi = f32_to_bf16(x);
        p.hb[idx] = hi;
        if (p.hb_lo) p.hb_lo[idx] = f32_to_bf16(x - bf16_to_f32(hi));
      }
      xv[j * kTileN + r] = fok ? hn * hn : 0.f;  // this column's square, row r
    }
    named_bar(kEpiBar, kEpiThreads);
    // Σh² of each valid column over the tile's 128 rows: 8 threads per
    // column, 16 rows each, then a fixed 3-step butterfly (a fixed order)
    {
      const int j = e >> 3, part = e & 7;
      float s = 0.f;
      if (j < jn) {
        const float* col = xv + j * kTileN + part * 16;
#pragma unroll
        for (int i = 0; i < 16; ++i) s += col[i];
      }
      s += __shfl_xor_sync(0xffffffffu, s, 4);
      s += __shfl_xor_sync(0xffffffffu, s, 2);
      s += __shfl_xor_sync(0xffffffffu, s, 1);
      if (j < jn && part == 0) p.ssq_out[static_cast<long long>(tile) * p.ssq_ld + p.tok0 + c0 + j] = s;
    }
    named_bar(kEpiBar, kEpiThreads);
    return;
  }
  if (p.epi == EPI_RESID) {
    // all 16 residual loads in flight before the first store (the residual
    // stream is rewritten by other CTAs between passes over it: L2 loads)
    const bool fok = f < p.N;
    const float gn = pre.have_gn ? pre.gn : (fok ? p.g_next[f] : 0.f);
    float hv[16], sq[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int m = p.tok0 + c0 + j;
      hv[j] = have_h ? hv_in[j] : ((m < p.M && fok) ? ldcg(p.h + static_cast<long long>(m) * p.d + f) : 0.f);
    }
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int m = p.tok0 + c0 + j;
      sq[j] = 0.f;
      if (m < p.M && fok) {
        const long long idx = static_cast<long long>(m) * p.d + f;
        const float hn = hv[j] + v[j];
        p.h[idx] = hn;
        const float x = hn * gn;
        const uint16_t hi = f32_to_bf16(x);
        p.hb[idx] = hi;
        if (p.hb_lo) p.hb_lo[idx] = f32_to_bf16(x - bf16_to_f32(hi));
        sq[j] = hn * hn;
      }
    }
    const int warp = (threadIdx.x >> 5) & 3;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      if (p.tok0 + c0 + j >= p.M) break;  // uniform: no valid column left
      const float s = warp_sum(sq[j]);
      if ((threadIdx.x & 31) == 0) sm.red[warp * 16 + j] = s;
    }
    named_bar(kEpiBar, kEpiThreads);
    if (e < 16) {
      const int m = p.tok0 + c0 + e;
      // quarters in row order 0..3 (warp w%4 holds rows 32*(w%4)..)
      const float s = ((sm.red[0 * 16 + e] + sm.red[1 * 16 + e]) + sm.red[2 * 16 + e]) +
                      sm.red[3 * 16 + e];
      if (m < p.M) p.ssq_out[static_cast<long long>(tile) * p.ssq_ld + m] = s;
    }
    named_bar(kEpiBar, kEpiThreads);
    return;
  }
  if (p.epi == EPI_QKV) {
    // exchange the 16 columns of every row through shared memory for RoPE
#pragma unroll
    for (int j = 0; j < 16; ++j) sm.xbuf[j * kTileN + r] = v[j];
    named_bar(kEpiBar, kEpiThreads);
    const int hd = p.hd, half = hd >> 1;
    const int qdim = p.H * hd, kdim = p.Hkv * hd;
    const int dim = f % hd;
    const bool rot = f < qdim + kdim;
    const int pr = dim < half ? r + half : r - half;
    const float2 fr = pre.have_fr ? pre.fr : p.rope[dim < half ? dim : dim - half];
    if (pre.qkv) {
      // the persistent forward: KV slot, rotary position and fit flag per
      // column are in shared memory, and so are the values (the exchange
      // buffer), so the loop runs over the valid columns only
      const int jn = min(16, p.M - p.tok0 - c0);
#pragma unroll 1
      for (int j = 0; j < jn; ++j) {
        if (f >= p.N) break;
        const int m = p.tok0 + c0 + j;
        float out = sm.xbuf[j * kTileN + r];
        if (rot) {
          float sn, cs;
          rope_sincos(pre.qkv[128 + c0 + j], fr, &sn, &cs);
          const float partner = sm.xbuf[j * kTileN + pr];
          out = dim < half ? out * cs - partner * sn : out * cs + partner * sn;
        }
        const int slot = pre.qkv[c0 + j];
        if (f < qdim) {
          const long long qi = static_cast<long long>(m) * qdim + f;
          const uint16_t hi = f32_to_bf16(out);
          p.q[qi] = hi;
          if (p.q_lo) p.q_lo[qi] = f32_to_bf16(out - bf16_to_f32(hi));
        } else if (pre.qkv[256 + c0 + j] && slot < p.cap) {
          const int kf = f < qdim + kdim ? f - qdim : f - qdim - kdim;
          const KVMap map{p.kv_table, p.kv_max_pages, p.kv_n_pages, p.Hkv, p.cap, hd};
          const long long idx = map.row<kKV>(m / p.n_per_seq, kf / hd, slot) + (kf % hd);
          (f < qdim + kdim ? p.kcache : p.vcache)[idx] = f32_to_bf16(out);
        }
      }
      named_bar(kEpiBar, kEpiThreads);
      return;
    }
    // slot = len + node index; rotary position = len + node depth (the node
    // index itself for a chain)
    int slotv[16], posv[16], okv[16];
#pragma unroll
    for (int j = 0; j < 16; ++j) {  // sequence bookkeeping, loads in flight together
      const int m = min(p.tok0 + c0 + j, p.M - 1);
      const int b = m / p.n_per_seq;
      const int base = ldcg_i(p.pos_base + b), node = m - b * p.n_per_seq;
      slotv[j] = base + node;
      posv[j] = base + (p.depth ? __ldg(p.depth + m) : node);
      okv[j] = ldcg_i(p.seq_ok + b);
    }
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
      const int m = p.tok0 + c0 + j;
      if (m >= p.M || f >= p.N) continue;
      const int b = m / p.n_per_seq;
      float out = v[j];
      const int pos = posv[j];
      if (rot) {
        float sn, cs;
        rope_sincos(pos, fr, &sn, &cs);
        const float partner = sm.xbuf[j * kTileN + pr];
        out = dim < half ? v[j] * cs - partner * sn : v[j] * cs + partner * sn;
      }
      if (f < qdim) {
        const long long qi = static_cast<long long>(m) * qdim + f;
        const uint16_t hi = f32_to_bf16(out);
        p.q[qi] = hi;
        if (p.q_lo) p.q_lo[qi] = f32_to_bf16(out - bf16_to_f32(hi));
      } else if (okv[j] && slotv[j] < p.cap) {
        const int kf = f < qdim + kdim ? f - qdim : f - qdim - kdim;
        const int kvh = kf / hd;
        const KVMap map{p.kv_table, p.kv_max_pages, p.kv_n_pages, p.Hkv, p.cap, hd};
        const long long idx = map.row<kKV>(b, kvh, slotv[j]) + (kf % hd);
        if (f < qdim + kdim)
          p.kcache[idx] = f32_to_bf16(out);
        else
          p.vcache[idx] = f32_to_bf16(out);
      }
    }
    named_bar(kEpiBar, kEpiThreads);
    return;
  }
  // EPI_SWIGLU
  if (pre.rolled) {
    // rows 0..63 of the tile are gates, 64..127 the matching ups; every
    // thread takes feature r % 64 for every other valid column
#pragma unroll
    for (int j = 0; j < 16; ++j) sm.xbuf[j * kTileN + r] = v[j];
    named_bar(kEpiBar, kEpiThreads);
    const int fo = static_cast<int>(tile) * 64 + (r & 63);
    const int jn = min(16, p.M - p.tok0 - c0);
    if (fo < p.ffn) {
#pragma unroll 1
      for (int j = r >> 6; j < jn; j += 2) {
        const float g = sm.xbuf[j * kTileN + (r & 63)], u = sm.xbuf[j * kTileN + (r & 63) + 64];
        const float a = g / (1.0f + __expf(-g)) * u;
        const uint16_t hi = f32_to_bf16(a);
        const long long idx = static_cast<long long>(p.tok0 + c0 + j) * p.ffn + fo;
        p.act[idx] = hi;
        if (p.act_lo) p.act_lo[idx] = f32_to_bf16(a - bf16_to_f32(hi));
      }
    }
    named_bar(kEpiBar, kEpiThreads);
    return;
  }
  if (r >= 64) {
#pragma unroll
    for (int j = 0; j < 16; ++j) sm.xbuf[j * kTileN + r] = v[j];
  }
  named_bar(kEpiBar, kEpiThreads);
  if (r < 64) {
    const int fo = static_cast<int>(tile) * 64 + r;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const int m = p.tok0 + c0 + j;
      if (m < p.M && fo < p.ffn) {
        const float g = v[j], u = sm.xbuf[j * kTileN + r + 64];
        const float sg = g / (1.0f + __expf(-g));
        const float a = sg * u;
        const uint16_t hi = f32_to_bf16(a);
        const long long idx = static_cast<long long>(m) * p.ffn + fo;
        p.act[idx] = hi;
        if (p.act_lo) p.act_lo[idx] = f32_to_bf16(a - bf16_to_f32(hi));
      }
    }
  }
  named_bar(kEpiBar, kEpiThreads);
}

__device__ __forceinline__ void epilogue_chunk(const GemmParams& p, const Smem& sm, uint32_t tile, int r,
                                               int c0, const float (&acc)[16]) {
  const float none[16] = {};
  epilogue_chunk_h(p, sm, tile, r, c0, acc, none, false, EpiPre{});
}

}  // namespace
}  // namespace spec
