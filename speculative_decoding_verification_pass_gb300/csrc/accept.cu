// The acceptance step of speculative decoding, one CTA per sequence, and the
// KV rollback.
//
// Rule (pigeon guide, *How it works* steps 3-5; lattice notes, the rule and
// its worked example; "Build a Speculative Decoding Engine ...", *The
// Accept/Reject Mechanism*): for i = 0..gamma-1 accept x_{i+1} iff
// u_i < min(1, p_i(x)/q_i(x)); at the first rejection draw the replacement
// from norm(max(0, p_i - q_i)) over the whole vocabulary and stop; if every
// draft survives draw a bonus token from p_gamma.  p is softmax(z/T) of the
// target logits, after top-p when enabled (applied identically to p and q:
// pigeon guide, *When it breaks*).  T = 0 is the greedy rule: accept while
// the draft equals the argmax.
//
// Draft sampling (sample_kernel), per CTA (1024 threads):
//  * row statistics in one pass: per-thread online (max, sum of exp2) merged
//    by a fixed-order block reduction; rows are visited lazily, so only the
//    rows up to the first rejection (plus the bonus row) are read;
//  * top-p threshold: a radix select over the fp32 bit patterns of the
//    unnormalised probabilities, weighted by their mass in 2^-40 fixed point
//    (integer shared-memory histograms: exact, order-independent);
//  * the draw: weights in 2^-52 fixed point, exact block prefix scan over
//    tiles of 4096 ids in id order, the smallest id whose cumulative weight
//    exceeds u * total (exact integer arithmetic, so the selected id is
//    consistent with its own cumulative sums and deterministic).
#include <algorithm>
#include <climits>

#include "common.cuh"
#include "internal.h"

namespace spec {

namespace {

constexpr int kT = 1024;
constexpr int kWarps = kT / 32;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kFix52 = 4503599627370496.0f;  // 2^52
constexpr float kFix40 = 1099511627776.0f;     // 2^40
constexpr double kResidualFallback = 1e-8;

struct Red {
  float f[kWarps];
  float g[kWarps];
  int i[kWarps];
  unsigned long long u[kWarps];
  unsigned long long hist[256];
  float bf[4];
  int bi[4];
  unsigned long long bu[4];
};

SPEC_DEVINL unsigned long long warp_sum_u64(unsigned long long v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// Block sum of a uint64 (fixed order, exact).
__device__ unsigned long long block_sum_u64(unsigned long long v, Red& r) {
  v = warp_sum_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) r.u[w] = v;
  __syncthreads();
  if (w == 0) {
    unsigned long long t = l < kWarps ? r.u[l] : 0ull;
    t = warp_sum_u64(t);
    if (l == 0) r.bu[0] = t;
  }
  __syncthreads();
  return r.bu[0];
}

__device__ float block_sum_f(float v, Red& r) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) r.f[w] = v;
  __syncthreads();
  if (w == 0) {
    float t = l < kWarps ? r.f[l] : 0.f;
    t = warp_sum(t);
    if (l == 0) r.bf[0] = t;
  }
  __syncthreads();
  return r.bf[0];
}

__device__ int block_max_i(int v, Red& r) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) r.i[w] = v;
  __syncthreads();
  if (w == 0) {
    int t = l < kWarps ? r.i[l] : INT_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (l == 0) r.bi[0] = t;
  }
  __syncthreads();
  return r.bi[0];
}

// (max, sum exp2((z - max) * c)) merge.
SPEC_DEVINL void ms_merge(float& m, float& s, float m2, float s2, float c) {
  if (m2 == -INFINITY) return;
  if (m == -INFINITY) {
    m = m2;
    s = s2;
    return;
  }
  const float mn = fmaxf(m, m2);
  s = s * exp2f((m - mn) * c) + s2 * exp2f((m2 - mn) * c);
  m = mn;
}

// f(x, a[x], b[x]) for every id x of a row (b may be nullptr: f gets 0).
// When both rows allow it, each thread takes groups of 4 consecutive ids
// with 16-byte loads, several groups in flight; else one id at a time.
template <class F>
SPEC_DEVINL void visit_row(const float* a, const float* b, int V, F&& f) {
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(a) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(b) & 15) == 0;
  if (vec) {
    const float4* a4 = reinterpret_cast<const float4*>(a);
    const float4* b4 = reinterpret_cast<const float4*>(b);
    const int V4 = V >> 2;
#pragma unroll 4
    for (int i = threadIdx.x; i < V4; i += kT) {
      const float4 va = __ldcg(a4 + i);
      const float4 vb = b ? __ldcg(b4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      f(4 * i, va.x, vb.x);
      f(4 * i + 1, va.y, vb.y);
      f(4 * i + 2, va.z, vb.z);
      f(4 * i + 3, va.w, vb.w);
    }
  } else {
#pragma unroll 4
    for (int x = threadIdx.x; x < V; x += kT) f(x, __ldcg(a + x), b ? __ldcg(b + x) : 0.f);
  }
}

// Row statistics of softmax(z / T): block max and sum of exp2((z-max)*c).
__device__ void row_stats(const float* z, int V, float c, Red& r, float& m_out, float& s_out) {
  float m = -INFINITY, s = 0.f;
  visit_row(z, nullptr, V, [&](int, float v, float) {
    if (v > m) {
      s = (m == -INFINITY ? 0.f : s * exp2f((m - v) * c)) + 1.0f;
      m = v;
    } else if (v != -INFINITY) {  // masked-out logits (-inf) weigh nothing
      s += exp2f((v - m) * c);
    }
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float m2 = __shfl_xor_sync(0xffffffffu, m, o);
    const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
    ms_merge(m, s, m2, s2, c);
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    r.f[w] = m;
    r.g[w] = s;
  }
  __syncthreads();
  if (w == 0) {
    float mm = l < kWarps ? r.f[l] : -INFINITY;
    float ss = l < kWarps ? r.g[l] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float m2 = __shfl_xor_sync(0xffffffffu, mm, o);
      const float s2 = __shfl_xor_sync(0xffffffffu, ss, o);
      ms_merge(mm, ss, m2, s2, c);
    }
    if (l == 0) {
      r.bf[0] = mm;
      r.bf[1] = ss;
    }
  }
  __syncthreads();
  m_out = r.bf[0];
  s_out = r.bf[1];
}

// Argmax with the lowest id on ties.
__device__ int row_argmax(const float* z, int V, Red& r) {
  float best = -INFINITY;
  int bi = 0x7fffffff;
  visit_row(z, nullptr, V, [&](int x, float v, float) {
    if (v > best || (v == best && x < bi)) {
      best = v;
      bi = x;
    }
  });
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
    const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
    if (v2 > best || (v2 == best && i2 < bi)) {
      best = v2;
      bi = i2;
    }
  }
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  __syncthreads();
  if (l == 0) {
    r.f[w] = best;
    r.i[w] = bi;
  }
  __syncthreads();
  if (w == 0) {
    best = l < kWarps ? r.f[l] : -INFINITY;
    bi = l < kWarps ? r.i[l] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      const float v2 = __shfl_xor_sync(0xffffffffu, best, o);
      const int i2 = __shfl_xor_sync(0xffffffffu, bi, o);
      if (v2 > best || (v2 == best && i2 < bi)) {
        best = v2;
        bi = i2;
      }
    }
    if (l == 0) r.bi[0] = bi == 0x7fffffff ? 0 : bi;
  }
  __syncthreads();
  return r.bi[0];
}

// The distribution one logits row stands for: e(x) = exp2((z - m) * c),
// kept iff e(x) >= tau (tau = 0: no nucleus), p(x) = e(x) / Z.
struct RowDist {
  const float* z;
  float m, c, tau, Z;
  SPEC_DEVINL float e_of(float zv) const { return exp2f((zv - m) * c); }
  SPEC_DEVINL float p_of(float zv) const {
    const float v = e_of(zv);
    return v >= tau ? v / Z : 0.f;
  }
  SPEC_DEVINL float p(int x) const { return p_of(__ldcg(z + x)); }
};

// Nucleus histogram bins of 2^-40 fixed-point masses (fx <= 2^40), kept as
// three 14-bit limbs in 32-bit counters: 32-bit shared-memory atomics are
// native, 64-bit ones several times slower.  A bin set is [3][256] counters
// shared by a pair of warps; the limb sums stay below 2^32 while a bin set
// takes at most 2^18 ids per pass, and reassemble exactly.
constexpr int kLimbBits = 14;
constexpr unsigned kLimbMask = (1u << kLimbBits) - 1u;
constexpr int kMaxIdsPerBins = 1 << 18;  // a bin set serves 1/8 (grid) or 1/16 of a row
static_assert(kNucleusMaxVocab / 8 <= kMaxIdsPerBins, "nucleus bin limbs would overflow");
SPEC_DEVINL void bins_add(unsigned* bins, int bkt, unsigned long long fx) {
  atomicAdd(bins + bkt, static_cast<unsigned>(fx) & kLimbMask);
  atomicAdd(bins + 256 + bkt, static_cast<unsigned>(fx >> kLimbBits) & kLimbMask);
  atomicAdd(bins + 512 + bkt, static_cast<unsigned>(fx >> (2 * kLimbBits)));
}
SPEC_DEVINL unsigned long long bins_get(const unsigned* bins, int bkt) {
  return static_cast<unsigned long long>(bins[bkt]) +
         (static_cast<unsigned long long>(bins[256 + bkt]) << kLimbBits) +
         (static_cast<unsigned long long>(bins[512 + bkt]) << (2 * kLimbBits));
}

// Histograms of the nucleus radix select (dynamic shared memory of the
// per-sequence kernels): one bin set per pair of warps, summed afterwards.
constexpr int kBinSets = kWarps / 2;
constexpr size_t kHistBytes = static_cast<size_t>(kBinSets) * 3 * 256 * sizeof(unsigned);

// Softmax statistics and (top_p < 1) the nucleus threshold of one row.
__device__ RowDist make_dist(const float* z, int V, float T, float top_p, Red& r,
                             unsigned* whist) {
  RowDist d;
  d.z = z;
  d.c = kLog2e / T;
  float s;
  row_stats(z, V, d.c, r, d.m, s);
  d.tau = 0.f;
  d.Z = s;
  if (!(top_p < 1.0f)) return d;
  // mass-weighted radix select over the bit patterns of e(x) (all >= 0):
  // tau = the largest value v with sum_{e >= v} e >= top_p * sum e.
  unsigned long long tot = 0;
  visit_row(z, nullptr, V, [&](int, float zv, float) {
    tot += static_cast<unsigned long long>(d.e_of(zv) * kFix40);
  });
  tot = block_sum_u64(tot, r);
  const double target = static_cast<double>(top_p) * static_cast<double>(tot);
  uint32_t prefix = 0;
  unsigned long long above = 0;  // mass strictly above the current prefix range
  for (int level = 0; level < 4; ++level) {
    const int shift = 24 - 8 * level;
    const uint32_t hi_mask = level == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    unsigned* wh = whist + (threadIdx.x >> 6) * 3 * 256;
    for (int i = threadIdx.x; i < kBinSets * 3 * 256; i += kT) whist[i] = 0u;
    __syncthreads();
    visit_row(z, nullptr, V, [&](int, float zv, float) {
      const float v = d.e_of(zv);
      const uint32_t bits = __float_as_uint(v);
      if ((bits & hi_mask) == prefix)
        bins_add(wh, static_cast<int>((bits >> shift) & 0xFFu), static_cast<unsigned long long>(v * kFix40));
    });
    __syncthreads();
    for (int i = threadIdx.x; i < 256; i += kT) {
      unsigned long long t = 0;
      for (int w = 0; w < kBinSets; ++w) t += bins_get(whist + w * 3 * 256, i);
      r.hist[i] = t;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int chosen = -1;
      unsigned long long acc = above;
      int lowest_nonempty = -1;
      for (int bkt = 255; bkt >= 0; --bkt) {
        const unsigned long long h = r.hist[bkt];
        if (h) lowest_nonempty = bkt;
        if (static_cast<double>(acc + h) >= target && h) {
          chosen = bkt;
          break;
        }
        acc += h;
      }
      if (chosen < 0) chosen = lowest_nonempty < 0 ? 0 : lowest_nonempty;
      r.bu[1] = acc;
      r.bi[1] = chosen;
    }
    __syncthreads();
    above = r.bu[1];
    prefix |= static_cast<uint32_t>(r.bi[1]) << shift;
    __syncthreads();
  }
  d.tau = __uint_as_float(prefix);
  float z_kept = 0.f;
  visit_row(z, nullptr, V, [&](int, float zv, float) {
    const float v = d.e_of(zv);
    z_kept += v >= d.tau ? v : 0.f;
  });
  d.Z = block_sum_f(z_kept, r);
  return d;
}

// Weight of id x for the final draw: the residual max(0, p - q) or p itself.
// (The weight types expose the rows they read -- src() and q -- and the
// weight of one id from those rows' values, so passes can load them in
// vector groups.)
struct DrawWeights {
  RowDist p;
  const float* q;  // nullptr: draw from p
  SPEC_DEVINL const float* src() const { return p.z; }
  SPEC_DEVINL float w_of(float zv, float qv) const {
    const float pv = p.p_of(zv);
    return q ? fmaxf(pv - qv, 0.f) : pv;
  }
  SPEC_DEVINL unsigned long long fx_of(float zv, float qv) const {
    return static_cast<unsigned long long>(w_of(zv, qv) * kFix52);
  }
  SPEC_DEVINL unsigned long long fx(int x) const {
    return fx_of(__ldcg(p.z + x), q ? __ldcg(q + x) : 0.f);
  }
};

SPEC_DEVINL unsigned long long warp_incl_scan_u64(unsigned long long v) {
  const int l = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (l >= o) v += n;
  }
  return v;
}

// Arguments of draw(): the total is the sum of the first level's chunk
// totals; the last positive id is found only if the threshold is not crossed
// (u * total rounded up to the total); a residual whose total is numerically
// zero returns kDrawFallback instead of drawing.
constexpr unsigned long long kTotalFromChunks = ~0ull;
constexpr int kLastPosLazy = -2;
constexpr int kDrawFallback = -3;

template <class DW>
__device__ int last_positive(const DW& dw, int V, Red& r);

// Inverse-CDF draw: the smallest id t with sum_{x<=t} fx(x) > floor(u * total).
// `total` is the exact fixed-point sum (or kTotalFromChunks); `last_pos` the
// last id with fx > 0 (or kLastPosLazy).
// Two levels: every warp sums a contiguous chunk of ids exactly (independent
// loads in flight), an exclusive scan of the chunk totals finds the chunk
// where the cumulative weight crosses the threshold, and that chunk alone is
// scanned id by id in tiles of 4 ids per thread.  The integer sums are exact,
// so the id is the one a single scan in id order finds.  With fallback set
// and dw.q given, a total at or below the residual fallback returns
// kDrawFallback (the caller draws from p instead).
template <class DW>
__device__ int draw(const DW& dw, int V, float u, unsigned long long total, int last_pos, Red& r,
                    bool fallback = false) {
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  const int chunk = ((V + kWarps - 1) / kWarps + 127) & ~127;
  const float* src = dw.src();
  const bool vec = (V & 3) == 0 && (reinterpret_cast<uintptr_t>(src) & 15) == 0 &&
                   (reinterpret_cast<uintptr_t>(dw.q) & 15) == 0;
  {
    const int c0 = w * chunk, c1 = min(V, c0 + chunk);
    unsigned long long s = 0;
    if (vec) {  // c0 and c1 are multiples of 4
      const float4* a4 = reinterpret_cast<const float4*>(src);
      const float4* b4 = reinterpret_cast<const float4*>(dw.q);
#pragma unroll 4
      for (int i = c0 / 4 + l; i < c1 / 4; i += 32) {
        const float4 va = __ldcg(a4 + i);
        const float4 vb = dw.q ? __ldcg(b4 + i) : make_float4(0.f, 0.f, 0.f, 0.f);
        s += dw.fx_of(va.x, vb.x) + dw.fx_of(va.y, vb.y) + dw.fx_of(va.z, vb.z) + dw.fx_of(va.w, vb.w);
      }
    } else {
#pragma unroll 4
      for (int x = c0 + l; x < c1; x += 32) s += dw.fx(x);
    }
    s = warp_sum_u64(s);
    __syncthreads();  // the reduction area may still be read by a previous step
    if (l == 0) r.u[w] = s;
    __syncthreads();
    if (w == 0) {
      const unsigned long long t = l < kWarps ? r.u[l] : 0ull;
      const unsigned long long ti = warp_incl_scan_u64(t);
      const unsigned long long tot =
          total == kTotalFromChunks ? __shfl_sync(0xffffffffu, ti, 31) : total;
      const unsigned long long th =
          static_cast<unsigned long long>(static_cast<double>(u) * static_cast<double>(tot));
      const bool fb = fallback && dw.q && static_cast<double>(tot) <= kResidualFallback * 4503599627370496.0;
      const bool hit = !fb && l < kWarps && ti - t <= th && th < ti;
      const unsigned ball = __ballot_sync(0xffffffffu, hit);
      if (hit) r.bu[2] = ti - t;  // one lane at most: the prefix before the crossing chunk
      if (l == 0) {
        r.bi[3] = fb ? kDrawFallback : (ball ? __ffs(ball) - 1 : -1);
        r.bu[3] = th;
      }
    }
    __syncthreads();
  }
  const int cw = r.bi[3];
  const unsigned long long thr = r.bu[3];
  if (cw == kDrawFallback) {
    __syncthreads();
    return kDrawFallback;
  }
  if (cw < 0)  // u * total rounded up to total
    return last_pos == kLastPosLazy ? last_positive(dw, V, r) : last_pos;
  unsigned long long run = r.bu[2];  // exact prefix before the current tile
  const int b0 = cw * chunk, b1 = min(V, b0 + chunk);
  __syncthreads();
  for (int base = b0; base < b1; base += 4 * kT) {
    const int x0 = base + threadIdx.x * 4;
    unsigned long long f[4];
    unsigned long long mine = 0;
    if (vec && x0 + 3 < b1) {
      const float4 va = __ldcg(reinterpret_cast<const float4*>(src + x0));
      const float4 vb = dw.q ? __ldcg(reinterpret_cast<const float4*>(dw.q + x0)) : make_float4(0.f, 0.f, 0.f, 0.f);
      f[0] = dw.fx_of(va.x, vb.x);
      f[1] = dw.fx_of(va.y, vb.y);
      f[2] = dw.fx_of(va.z, vb.z);
      f[3] = dw.fx_of(va.w, vb.w);
    } else {
#pragma unroll
      for (int k = 0; k < 4; ++k) f[k] = (x0 + k < b1) ? dw.fx(x0 + k) : 0ull;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) mine += f[k];
    const unsigned long long incl_w = warp_incl_scan_u64(mine);
    __syncthreads();
    if (l == 31) r.u[w] = incl_w;
    __syncthreads();
    if (w == 0) {
      unsigned long long t = l < kWarps ? r.u[l] : 0ull;
      const unsigned long long ti = warp_incl_scan_u64(t);
      if (l < kWarps) r.u[l] = ti - t;  // exclusive prefix of warp totals
      if (l == kWarps - 1) r.bu[2] = ti;
    }
    __syncthreads();
    const unsigned long long excl = run + r.u[w] + (incl_w - mine);
    const unsigned long long tile_total = r.bu[2];
    if (threadIdx.x == 0) r.bi[2] = -1;
    __syncthreads();
    if (excl <= thr && thr < excl + mine) {
      unsigned long long c = excl;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        c += f[k];
        if (c > thr) {
          r.bi[2] = x0 + k;
          break;
        }
      }
    }
    __syncthreads();
    if (r.bi[2] >= 0) return r.bi[2];
    run += tile_total;
    __syncthreads();
  }
  return last_pos;
}

// The last id with a positive draw weight (-1: none).
template <class DW>
__device__ int last_positive(const DW& dw, int V, Red& r) {
  int lp = -1;
  visit_row(dw.src(), dw.q, V, [&](int x, float sv, float qv) {
    if (dw.fx_of(sv, qv)) lp = max(lp, x);
  });
  __syncthreads();
  return block_max_i(lp, r);
}

// Exact fixed-point total and last positive id of the draw weights.
template <class DW>
__device__ void weights_total(const DW& dw, int V, Red& r, unsigned long long& total,
                              int& last_pos) {
  unsigned long long s = 0;
  int lp = -1;
  visit_row(dw.src(), dw.q, V, [&](int x, float sv, float qv) {
    const unsigned long long f = dw.fx_of(sv, qv);
    s += f;
    if (f) lp = max(lp, x);
  });
  total = block_sum_u64(s, r);
  last_pos = block_max_i(lp, r);
}

// ------------------------------------------------------- accept per sequence
// One CTA per sequence (batches with more than kAcceptGridRows rows): rows are
// visited lazily up to the first rejection.
__global__ void __launch_bounds__(kT, 1) accept_seq_kernel(const AcceptParams p) {
  __shared__ Red red;
  extern __shared__ unsigned dyn_hist[];  // kHistBytes
  __shared__ int s_flag;
  const int b = blockIdx.x;
  const int gamma = p.gamma, V = p.V, n = gamma + 1;
  const float* zb = p.logits + static_cast<long long>(b) * n * V;
  const int32_t* xb = p.draft + static_cast<long long>(b) * gamma;
  int32_t* out = p.out + static_cast<long long>(b) * n;
  for (int i = threadIdx.x; i < n; i += kT) out[i] = -1;
  __syncthreads();

  if (p.T == 0.f) {
    int acc = 0;
    for (int i = 0; i <= gamma; ++i) {
      const int a = row_argmax(zb + static_cast<long long>(i) * V, V, red);
      if (threadIdx.x == 0) out[i] = a;
      if (i < gamma && __ldg(xb + i) == a) {
        ++acc;
        continue;
      }
      break;
    }
    if (threadIdx.x == 0) p.n_acc[b] = acc;
    return;
  }

  const float* qb = p.q + static_cast<long long>(b) * gamma * V;
  const float* ub = p.u + static_cast<long long>(b) * n;
  int j = gamma;
  RowDist dist;
  for (int i = 0; i < gamma; ++i) {
    dist = make_dist(zb + static_cast<long long>(i) * V, V, p.T, p.top_p, red, dyn_hist);
    if (threadIdx.x == 0) {
      int x = __ldg(xb + i);
      bool accept = false;
      if (x < 0 || x >= V) {
        set_status(p.status, SPEC_DEV_BAD_TOKEN);
      } else {
        const float qx = __ldg(qb + static_cast<long long>(i) * V + x);
        if (!(qx > 0.f)) {
          set_status(p.status, SPEC_DEV_Q_ZERO);
        } else {
          const float a = fminf(1.0f, dist.p(x) / qx);
          accept = __ldg(ub + i) < a;
        }
      }
      if (accept) out[i] = x;
      s_flag = accept;
    }
    __syncthreads();
    if (!s_flag) {
      j = i;
      break;
    }
  }
  DrawWeights dw;
  if (j == gamma) {
    dist = make_dist(zb + static_cast<long long>(gamma) * V, V, p.T, p.top_p, red, dyn_hist);
    dw.p = dist;
    dw.q = nullptr;
  } else {
    dw.p = dist;
    dw.q = qb + static_cast<long long>(j) * V;
  }
  const float ug = __ldg(ub + gamma);
  int t = draw(dw, V, ug, kTotalFromChunks, kLastPosLazy, red, true);
  if (t == kDrawFallback) {
    dw.q = nullptr;  // residual mass numerically zero: draw from p
    t = draw(dw, V, ug, kTotalFromChunks, kLastPosLazy, red);
  }
  if (threadIdx.x == 0) {
    out[j] = t < 0 ? 0 : t;
    p.n_acc[b] = j;
  }
}

// ------------------------------------------------------------- accept grid
// The acceptance step as one cooperative grid over (sequence, row, vocabulary
// chunk) units, phases separated by grid-wide barriers:
//   P1  per chunk: online (max, sum exp2) of z / T, or (greedy) the chunk's
//       argmax; with top_p < 1 the nucleus histograms and totals are cleared.
//   N0..N3 (top_p < 1 only)  the mass-weighted radix select of the nucleus
//       threshold over global integer histograms (one 8-bit digit per phase;
//       the last digit is chosen where the row statistics are merged, and the
//       kept mass is the mass above the threshold plus its own bin).
//   P2  per (sequence, chunk): every unit takes the same accept decisions
//       (they only need the merged row statistics and one id per row) and
//       sums the chunk's 2^-52 fixed-point draw weights (residual and p).
//   P3  per sequence: the chunk where the cumulative weight crosses
//       u * total, then one block scan of that chunk.
// Row statistics are merged from the chunk partials in a fixed order by one
// warp, so every CTA derives bit-identical values; the fixed-point sums are
// exact integers, so the draw is the single-scan inverse CDF in id order.
constexpr int kAT = 512;
constexpr int kAW = kAT / 32;
constexpr int kAPer = kAcceptMaxChunk / kAT;  // ids per thread in a chunk scan
constexpr int kMaxRows = 128;

struct ASmem {
  float f[kAW];
  float g[kAW];
  int i[kAW];
  unsigned long long u[kAW];
  unsigned hist[kAW / 2][3 * 256];  // nucleus bins: one set per pair of warps
  float rm[kMaxRows];   // row max (greedy: argmax value)
  float rz[kMaxRows];   // row normaliser (kept mass with a nucleus)
  float rtau[kMaxRows]; // nucleus threshold on e(x) (0: none)
  int ri[kMaxRows];     // greedy: argmax id
  float bf[2];
  unsigned long long bu[3];
  int bi[3];
  uint32_t prefix;
  int j, tok, abort;
};

SPEC_DEVINL bool agrid_sync(const AcceptParams& p, unsigned target, ASmem& s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(p.bar, 1u);
    if (ld_acquire(p.bar) < target) {
      const unsigned long long t0 = globaltimer();
      while (ld_acquire(p.bar) < target) {
        if (globaltimer() - t0 > kWaitLimitNs) {
          set_status(p.status, SPEC_DEV_TIMEOUT);
          s.abort = 1;
          break;
        }
        __nanosleep(32);
      }
    }
  }
  __syncthreads();
  return s.abort == 0;
}

// Block (max, sum exp2((z - max) c)) over ids [x0, x1), fixed merge order.
__device__ float2 chunk_ms(const float* z, int x0, int x1, float c, ASmem& s) {
  float m = -INFINITY, sum = 0.f;
  for (int xs = x0; xs < x1; xs += kAPer * kAT) {
    float zv[kAPer];  // this thread's ids xs + threadIdx.x + k kAT, loaded together
#pragma unroll
    for (int k = 0; k < kAPer; ++k) {
      const int x = xs + threadIdx.x + k * kAT;
      zv[k] = x < x1 ? __ldcg(z + x) : -INFINITY;
    }
#pragma unroll
    for (int k = 0; k < kAPer; ++k) {
      const float v = zv[k];
      if (v > m) {
        sum = (m == -INFINITY ? 0.f : sum * exp2f((m - v) * c)) + 1.0f;
        m = v;
      } else if (v != -INFINITY) {  // masked-out logits (-inf) weigh nothing
        sum += exp2f((v - m) * c);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    ms_merge(m, sum, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sum, o), c);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    s.f[w] = m;
    s.g[w] = sum;
  }
  __syncthreads();
  if (w == 0) {
    m = l < kAW ? s.f[l] : -INFINITY;
    sum = l < kAW ? s.g[l] : 0.f;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      ms_merge(m, sum, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sum, o), c);
    if (l == 0) {
      s.bf[0] = m;
      s.bf[1] = sum;
    }
  }
  __syncthreads();
  const float2 r = make_float2(s.bf[0], s.bf[1]);
  __syncthreads();
  return r;
}

SPEC_DEVINL void arg_merge(float& v, int& i, float v2, int i2) {
  if (v2 > v || (v2 == v && i2 < i)) {
    v = v2;
    i = i2;
  }
}

// Block argmax over [x0, x1), lowest id on ties.
__device__ float2 chunk_argmax(const float* z, int x0, int x1, ASmem& s) {
  float best = -INFINITY;
  int bi = 0x7fffffff;
  for (int x = x0 + threadIdx.x; x < x1; x += kAT) arg_merge(best, bi, __ldcg(z + x), x);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    arg_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bi, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) {
    s.f[w] = best;
    s.i[w] = bi;
  }
  __syncthreads();
  if (w == 0) {
    best = l < kAW ? s.f[l] : -INFINITY;
    bi = l < kAW ? s.i[l] : 0x7fffffff;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      arg_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, o), __shfl_xor_sync(0xffffffffu, bi, o));
    if (l == 0) {
      s.bf[0] = best;
      s.bi[0] = bi;
    }
  }
  __syncthreads();
  const float2 r = make_float2(s.bf[0], __int_as_float(s.bi[0]));
  __syncthreads();
  return r;
}

// Block sums (fixed order): a uint64 and a float.
__device__ unsigned long long ablock_sum_u64(unsigned long long v, ASmem& s) {
  v = warp_sum_u64(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) s.u[w] = v;
  __syncthreads();
  if (w == 0) {
    unsigned long long t = l < kAW ? s.u[l] : 0ull;
    t = warp_sum_u64(t);
    if (l == 0) s.bu[0] = t;
  }
  __syncthreads();
  const unsigned long long r = s.bu[0];
  __syncthreads();
  return r;
}

__device__ float ablock_sum_f(float v, ASmem& s) {
  v = warp_sum(v);
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) s.f[w] = v;
  __syncthreads();
  if (w == 0) {
    float t = l < kAW ? s.f[l] : 0.f;
    t = warp_sum(t);
    if (l == 0) s.bf[0] = t;
  }
  __syncthreads();
  const float r = s.bf[0];
  __syncthreads();
  return r;
}

__device__ int ablock_max_i(int v, ASmem& s) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  if (l == 0) s.i[w] = v;
  __syncthreads();
  if (w == 0) {
    int t = l < kAW ? s.i[l] : INT_MIN;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) t = max(t, __shfl_xor_sync(0xffffffffu, t, o));
    if (l == 0) s.bi[0] = t;
  }
  __syncthreads();
  const int r = s.bi[0];
  __syncthreads();
  return r;
}

// One warp: merged (max, sum) of a row from its S chunk partials.
SPEC_DEVINL float2 warp_row_ms(const float2* part, int S, float c) {
  float m = -INFINITY, sum = 0.f;
  for (int k = threadIdx.x & 31; k < S; k += 32) {
    const float2 v = __ldcg(part + k);
    ms_merge(m, sum, v.x, v.y, c);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    ms_merge(m, sum, __shfl_xor_sync(0xffffffffu, m, o), __shfl_xor_sync(0xffffffffu, sum, o), c);
  return make_float2(m, sum);
}

// One warp: one digit of the mass-weighted radix select.  Among the 256
// buckets of `hist` (values sharing the digits chosen so far), scanning from
// the top with `above` = the mass strictly above them, pick the first bucket
// at which the cumulative mass reaches `target`; `above` becomes the mass
// strictly above that bucket.  If rounding leaves the target unreached, the
// lowest nonempty bucket (0 if none) with `above` = the whole mass.
SPEC_DEVINL int warp_select(const unsigned long long* hist, double target,
                            unsigned long long& above) {
  const int lane = threadIdx.x & 31;
  unsigned long long h[8], ls = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    h[k] = __ldcg(hist + 255 - 8 * lane - k);
    ls += h[k];
  }
  unsigned long long incl = ls;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += t;
  }
  unsigned long long acc = above + incl - ls;
  int cand = -1;
  unsigned long long cacc = 0;
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    if (cand < 0) {
      if (h[k] && static_cast<double>(acc + h[k]) >= target) {
        cand = 255 - 8 * lane - k;
        cacc = acc;
      } else {
        acc += h[k];
      }
    }
  }
  const unsigned ball = __ballot_sync(0xffffffffu, cand >= 0);
  const unsigned long long total = above + __shfl_sync(0xffffffffu, incl, 31);
  if (ball) {
    const int src = __ffs(ball) - 1;
    above = __shfl_sync(0xffffffffu, cacc, src);
    return __shfl_sync(0xffffffffu, cand, src);
  }
  int low = -1;
#pragma unroll
  for (int k = 0; k < 8; ++k)
    if (h[k]) low = 255 - 8 * lane - k;
  const unsigned nb = __ballot_sync(0xffffffffu, low >= 0);
  above = total;
  return nb ? __shfl_sync(0xffffffffu, low, 31 - __clz(nb)) : 0;
}

struct ARow {  // the distribution of one row: e = exp2((z - m) c), kept iff e >= tau
  const float* z;
  float m, c, tau, Z;
  SPEC_DEVINL float p_of(float zx) const {
    const float e = exp2f((zx - m) * c);
    return e >= tau ? e / Z : 0.f;
  }
  SPEC_DEVINL float p(int x) const { return p_of(__ldcg(z + x)); }
};

// This thread's ids xs + threadIdx.x + k kAT (k < kAPer) below x1, loaded
// together (0 past x1).
SPEC_DEVINL void load_block(const float* z, int xs, int x1, float (&zv)[kAPer]) {
#pragma unroll
  for (int k = 0; k < kAPer; ++k) {
    const int x = xs + threadIdx.x + k * kAT;
    zv[k] = x < x1 ? __ldcg(z + x) : 0.f;
  }
}

// Id ranges per row of the nucleus select's work units: about one unit per
// CTA, so that a unit's fixed costs (the row's statistics and the digits
// chosen so far, read by one warp; block barriers) are paid once per range.
// Units per row of the chunk statistics (P1) and of the nucleus select,
// chosen by the launcher for the grid it launches.
SPEC_DEVINL int stats_split(const AcceptParams& p) { return p.S1; }
SPEC_DEVINL int nucleus_split(const AcceptParams& p) { return p.SL; }

// Statistics of every row of sequence b into shared memory (all warps).
__device__ void seq_stats(const AcceptParams& p, int b, float c, bool nucleus, ASmem& s) {
  const int n = p.gamma + 1;
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  for (int i = w; i < n; i += kAW) {
    const long long row = static_cast<long long>(b) * n + i;
    const float2 ms = warp_row_ms(p.part_ms + row * p.S, stats_split(p), c);
    float Z = ms.y, tau = 0.f;
    if (nucleus) {
      // the last digit of the threshold, and the kept mass: everything
      // strictly above it plus its own bin, from the exact histograms
      unsigned long long above = __ldcg(p.sel + (row * 4 + 2) * 2 + 1);
      const uint32_t prefix = static_cast<uint32_t>(__ldcg(p.sel + (row * 4 + 2) * 2));
      const unsigned long long tot = __ldcg(p.tot40 + row);
      const double target = static_cast<double>(p.top_p) * static_cast<double>(tot);
      const int chosen = warp_select(p.hist + (row * 4 + 3) * 256, target, above);
      const unsigned long long kept = above + __ldcg(p.hist + (row * 4 + 3) * 256 + chosen);
      Z = static_cast<float>(static_cast<double>(kept < tot ? kept : tot) / 1099511627776.0);
      tau = __uint_as_float(prefix | static_cast<uint32_t>(chosen));
    }
    if (l == 0) {
      s.rm[i] = ms.x;
      s.rz[i] = Z;
      s.rtau[i] = tau;
    }
  }
  __syncthreads();
}

SPEC_DEVINL ARow arow(const AcceptParams& p, int b, int i, float c, const ASmem& s) {
  ARow r;
  r.z = p.logits + (static_cast<long long>(b) * (p.gamma + 1) + i) * p.V;
  r.m = s.rm[i];
  r.c = c;
  r.tau = s.rtau[i];
  r.Z = s.rz[i];
  return r;
}

// Warp 0 (every lane): the first rejected draft of sequence b (gamma if
// none), with the device status flag of that draft when `flag`.  Each lane
// tests one draft (its token, q and p loads in flight together); the answer
// is the first draft that is rejected or invalid, as in the sequential rule.
__device__ int decide_warp(const AcceptParams& p, int b, float c, const ASmem& s, bool flag) {
  const int l = threadIdx.x & 31;
  const int32_t* xb = p.draft + static_cast<long long>(b) * p.gamma;
  const float* qb = p.q + static_cast<long long>(b) * p.gamma * p.V;
  const float* ub = p.u + static_cast<long long>(b) * (p.gamma + 1);
  for (int i0 = 0; i0 < p.gamma; i0 += 32) {
    const int i = i0 + l;
    int why = 0;  // 0 accepted, 1 rejected, 2 token out of range, 3 q(x) = 0
    if (i < p.gamma) {
      const int x = __ldg(xb + i);
      if (x < 0 || x >= p.V) {
        why = 2;
      } else {
        const float qx = __ldg(qb + static_cast<long long>(i) * p.V + x);
        const float px = arow(p, b, i, c, s).p(x);
        const float ui = __ldg(ub + i);
        if (!(qx > 0.f))
          why = 3;
        else if (!(ui < fminf(1.0f, px / qx)))
          why = 1;
      }
    }
    const unsigned stop = __ballot_sync(0xffffffffu, why != 0);
    if (stop) {
      const int first = __ffs(stop) - 1;
      const int w = __shfl_sync(0xffffffffu, why, first);
      if (flag && l == 0 && w >= 2) set_status(p.status, w == 2 ? SPEC_DEV_BAD_TOKEN : SPEC_DEV_Q_ZERO);
      return i0 + first;
    }
  }
  return p.gamma;
}

// Fixed-point draw weights of an id with p = pv, q = qv: k = 0 residual
// max(0, p_j - q_j), k = 1 p_r.
SPEC_DEVINL unsigned long long fx_of(float pv, float qv, int k) {
  const float w = k == 0 ? fmaxf(pv - qv, 0.f) : pv;
  return static_cast<unsigned long long>(w * kFix52);
}
SPEC_DEVINL unsigned long long fx_weight(const ARow& r, const float* qrow, int x, int k) {
  const float pv = r.p(x);
  return fx_of(pv, k == 0 ? __ldcg(qrow + x) : 0.f, k);
}

__global__ void __launch_bounds__(kAT) accept_grid_kernel(const AcceptParams p) {
  __shared__ ASmem s;
  const int n = p.gamma + 1, S = p.S, C = p.C, V = p.V, B = p.B;
  const int G = gridDim.x;
  const bool greedy = !(p.T > 0.f);
  const bool nucleus = !greedy && p.top_p < 1.0f;
  const float c = greedy ? 0.f : kLog2e / p.T;
  unsigned nbar = 0;
  if (threadIdx.x == 0) s.abort = 0;
  __syncthreads();

  // ---- P1: chunk statistics
  if (nucleus) {
    const long long nh = static_cast<long long>(B) * n * 4 * 256;
    for (long long k = static_cast<long long>(blockIdx.x) * kAT + threadIdx.x; k < nh;
         k += static_cast<long long>(G) * kAT)
      p.hist[k] = 0ull;
    for (long long k = static_cast<long long>(blockIdx.x) * kAT + threadIdx.x;
         k < static_cast<long long>(B) * n; k += static_cast<long long>(G) * kAT)
      p.tot40[k] = 0ull;
  }
  const int S1 = stats_split(p);  // P1 units per row
  const long long units1 = static_cast<long long>(B) * n * S1;
  for (long long u = blockIdx.x; u < units1; u += G) {
    const int k = static_cast<int>(u % S1);
    const long long row = u / S1;
    const float* z = p.logits + row * V;
    const int x0 = static_cast<int>(static_cast<long long>(k) * V / S1);
    const int x1 = static_cast<int>(static_cast<long long>(k + 1) * V / S1);
    p.part_ms[row * S + k] = greedy ? chunk_argmax(z, x0, x1, s) : chunk_ms(z, x0, x1, c, s);
  }
  if (!agrid_sync(p, ++nbar * G, s)) return;

  if (greedy) {
    for (int b = blockIdx.x; b < B; b += G) {
      const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
      for (int i = w; i < n; i += kAW) {
        const float2* part = p.part_ms + (static_cast<long long>(b) * n + i) * S;
        float best = -INFINITY;
        int bi = 0x7fffffff;
        for (int k = l; k < S1; k += 32) {
          const float2 v = __ldcg(part + k);
          arg_merge(best, bi, v.x, __float_as_int(v.y));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1)
          arg_merge(best, bi, __shfl_xor_sync(0xffffffffu, best, o),
                    __shfl_xor_sync(0xffffffffu, bi, o));
        if (l == 0) s.ri[i] = bi == 0x7fffffff ? 0 : bi;
      }
      __syncthreads();
      if (threadIdx.x == 0) {
        const int32_t* xb = p.draft + static_cast<long long>(b) * p.gamma;
        int32_t* out = p.out + static_cast<long long>(b) * n;
        int acc = 0, i = 0;
        for (; i <= p.gamma; ++i) {
          out[i] = s.ri[i];
          if (i < p.gamma && __ldg(xb + i) == s.ri[i]) {
            ++acc;
            continue;
          }
          break;
        }
        for (++i; i < n; ++i) out[i] = -1;
        p.n_acc[b] = acc;
      }
      __syncthreads();
    }
    return;
  }

  // ---- N0..N3: the digits of the nucleus threshold of every row
  if (nucleus) {
    const int SL = nucleus_split(p);
    const long long units_l = static_cast<long long>(B) * n * SL;
    for (int level = 0; level <= 3; ++level) {
      for (long long u = blockIdx.x; u < units_l; u += G) {
        const int kr = static_cast<int>(u % SL);
        const long long row = u / SL;
        const float* z = p.logits + row * V;
        const int x0 = static_cast<int>(static_cast<long long>(kr) * V / SL);
        const int x1 = static_cast<int>(static_cast<long long>(kr + 1) * V / SL);
        if (threadIdx.x < 32) {
          const float2 ms = warp_row_ms(p.part_ms + row * S, S1, c);
          uint32_t prefix = 0;
          if (level >= 1) {
            unsigned long long above = 0;
            if (level >= 2) {
              prefix = static_cast<uint32_t>(__ldcg(p.sel + (row * 4 + level - 2) * 2));
              above = __ldcg(p.sel + (row * 4 + level - 2) * 2 + 1);
            }
            const double target = static_cast<double>(p.top_p) * static_cast<double>(__ldcg(p.tot40 + row));
            const int chosen = warp_select(p.hist + (row * 4 + level - 1) * 256, target, above);
            prefix |= static_cast<uint32_t>(chosen) << (24 - 8 * (level - 1));
            if (threadIdx.x == 0 && kr == 0) {
              p.sel[(row * 4 + level - 1) * 2] = prefix;
              p.sel[(row * 4 + level - 1) * 2 + 1] = above;
            }
          }
          if (threadIdx.x == 0) {
            s.bf[0] = ms.x;
            s.prefix = prefix;
          }
        }
        for (int k = threadIdx.x; k < kAW / 2 * 3 * 256; k += kAT) (&s.hist[0][0])[k] = 0u;
        __syncthreads();
        const float m = s.bf[0];
        const uint32_t prefix = s.prefix;
        {
          const int shift = 24 - 8 * level;
          const uint32_t hi_mask = level == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
          unsigned long long mass = 0;
          // this warp pair's bins: same-bin atomics contend within the pair only
          unsigned* wh = s.hist[threadIdx.x >> 6];
          float zv[kAPer];
          load_block(z, x0, x1, zv);
          for (int xs = x0; xs < x1; xs += kAPer * kAT) {
            float zn[kAPer];  // the next block's loads in flight during this one
            load_block(z, xs + kAPer * kAT, x1, zn);
#pragma unroll
            for (int k = 0; k < kAPer; ++k) {
              // every lane takes part in each step (the peer sums below)
              const bool valid = xs + static_cast<int>(threadIdx.x) + k * kAT < x1;
              const float e = valid ? exp2f((zv[k] - m) * c) : 0.f;
              const uint32_t bits = __float_as_uint(e);
              const unsigned long long fx = static_cast<unsigned long long>(e * kFix40);
              mass += fx;
              if (valid && (bits & hi_mask) == prefix) bins_add(wh, static_cast<int>((bits >> shift) & 0xFFu), fx);
            }
#pragma unroll
            for (int k = 0; k < kAPer; ++k) zv[k] = zn[k];
          }
          if (level == 0) {
            mass = ablock_sum_u64(mass, s);
            if (threadIdx.x == 0) atomicAdd(p.tot40 + row, mass);
          }
          __syncthreads();
          for (int k = threadIdx.x; k < 256; k += kAT) {
            unsigned long long t = 0;  // integer sums: exact in any order
#pragma unroll
            for (int w = 0; w < kAW / 2; ++w) t += bins_get(s.hist[w], k);
            if (t) atomicAdd(p.hist + (row * 4 + level) * 256 + k, t);
          }
        }
        __syncthreads();
      }
      if (!agrid_sync(p, ++nbar * G, s)) return;
    }
  }

  // ---- P2: decisions and the chunk sums of the draw weights
  const long long units2 = static_cast<long long>(B) * S;
  for (long long u = blockIdx.x; u < units2; u += G) {
    const int b = static_cast<int>(u / S), ch = static_cast<int>(u % S);
    seq_stats(p, b, c, nucleus, s);
    if (threadIdx.x < 32) {
      const int jd = decide_warp(p, b, c, s, ch == 0);
      if (threadIdx.x == 0) s.j = jd;
    }
    __syncthreads();
    const int j = s.j;
    const ARow r = arow(p, b, j, c, s);
    const float* qrow = p.q + (static_cast<long long>(b) * p.gamma + (j < p.gamma ? j : 0)) * V;
    const int x0 = ch * C, x1 = min(x0 + C, V);
    unsigned long long tr = 0, tp = 0;
    int lr = -1, lp = -1;
    float zv[kAPer], qv[kAPer];  // this thread's ids, loaded together
#pragma unroll
    for (int k = 0; k < kAPer; ++k) {
      const int x = x0 + threadIdx.x + k * kAT;
      zv[k] = x < x1 ? __ldcg(r.z + x) : -INFINITY;
      qv[k] = x < x1 && j < p.gamma ? __ldcg(qrow + x) : 0.f;
    }
#pragma unroll
    for (int k = 0; k < kAPer; ++k) {
      const int x = x0 + threadIdx.x + k * kAT;
      if (x >= x1) break;
      const float pv = r.p_of(zv[k]);
      const unsigned long long fp = fx_of(pv, 0.f, 1);
      tp += fp;
      if (fp) lp = x;
      if (j < p.gamma) {
        const unsigned long long fr = fx_of(pv, qv[k], 0);
        tr += fr;
        if (fr) lr = x;
      }
    }
    tr = ablock_sum_u64(tr, s);
    tp = ablock_sum_u64(tp, s);
    lr = ablock_max_i(lr, s);
    lp = ablock_max_i(lp, s);
    if (threadIdx.x == 0) {
      p.part_tot[u * 2] = tr;
      p.part_tot[u * 2 + 1] = tp;
      p.part_last[u * 2] = lr;
      p.part_last[u * 2 + 1] = lp;
    }
    __syncthreads();
  }
  if (!agrid_sync(p, ++nbar * G, s)) return;

  // ---- P3: the draw
  for (int b = blockIdx.x; b < B; b += G) {
    seq_stats(p, b, c, nucleus, s);
    if (threadIdx.x < 32) {
      // warp 0: the decision, the totals and the chunk holding the draw
      const int l = threadIdx.x;
      const int j = decide_warp(p, b, c, s, false);
      const unsigned long long* tot = p.part_tot + static_cast<long long>(b) * S * 2;
      const int* last = p.part_last + static_cast<long long>(b) * S * 2;
      unsigned long long total_r = 0, total_p = 0;
      for (int k = l; k < S; k += 32) {
        total_r += __ldcg(tot + 2 * k);
        total_p += __ldcg(tot + 2 * k + 1);
      }
      total_r = warp_sum_u64(total_r);  // integer sums: exact in any order
      total_p = warp_sum_u64(total_p);
      int kind = 1;
      if (j < p.gamma && !(static_cast<double>(total_r) <= kResidualFallback * 4503599627370496.0))
        kind = 0;
      const unsigned long long total = kind == 0 ? total_r : total_p;
      const float uu = __ldg(p.u + static_cast<long long>(b) * n + p.gamma);
      const unsigned long long thr =
          static_cast<unsigned long long>(static_cast<double>(uu) * static_cast<double>(total));
      // the first chunk k with thr < (sum of chunks 0..k): 32 chunks a round
      unsigned long long run = 0, base = 0;
      int found = -1, lastpos = -1;
      for (int k0 = 0; k0 < S; k0 += 32) {
        const int k = k0 + l;
        const unsigned long long t = k < S ? __ldcg(tot + 2 * k + kind) : 0ull;
        if (k < S) lastpos = max(lastpos, __ldcg(last + 2 * k + kind));
        unsigned long long incl = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const unsigned long long v = __shfl_up_sync(0xffffffffu, incl, o);
          if (l >= o) incl += v;
        }
        if (found < 0) {
          const unsigned hit = __ballot_sync(0xffffffffu, k < S && thr < base + incl);
          if (hit) {
            const int f = __ffs(hit) - 1;
            found = k0 + f;
            run = base + __shfl_sync(0xffffffffu, incl - t, f);
          }
        }
        base += __shfl_sync(0xffffffffu, incl, 31);
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) lastpos = max(lastpos, __shfl_xor_sync(0xffffffffu, lastpos, o));
      if (l == 0) {
        s.j = j;
        s.bi[0] = found;
        s.bi[1] = kind;
        s.bi[2] = lastpos;
        s.bu[1] = run;
        s.bu[2] = thr;
        s.tok = -1;
      }
    }
    __syncthreads();
    const int j = s.j, found = s.bi[0], kind = s.bi[1];
    int tok = s.bi[2];
    if (found >= 0) {
      const ARow r = arow(p, b, j, c, s);
      const float* qrow = p.q + (static_cast<long long>(b) * p.gamma + (j < p.gamma ? j : 0)) * V;
      const int x0 = found * C + threadIdx.x * kAPer;
      const int x1 = min(found * C + C, V);
      unsigned long long f[kAPer], mine = 0;
#pragma unroll
      for (int k = 0; k < kAPer; ++k) {
        f[k] = x0 + k < x1 ? fx_weight(r, qrow, x0 + k, kind) : 0ull;
        mine += f[k];
      }
      const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
      unsigned long long incl = mine;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const unsigned long long t = __shfl_up_sync(0xffffffffu, incl, o);
        if (l >= o) incl += t;
      }
      if (l == 31) s.u[w] = incl;
      __syncthreads();
      unsigned long long wex = 0;
      for (int k = 0; k < w; ++k) wex += s.u[k];
      const unsigned long long thr = s.bu[2];
      unsigned long long acc = s.bu[1] + wex + (incl - mine);
      if (acc <= thr && thr < acc + mine) {
#pragma unroll
        for (int k = 0; k < kAPer; ++k) {
          acc += f[k];
          if (acc > thr) {
            s.tok = x0 + k;
            break;
          }
        }
      }
      __syncthreads();
      if (s.tok >= 0) tok = s.tok;
    }
    if (threadIdx.x == 0) {
      const int32_t* xb = p.draft + static_cast<long long>(b) * p.gamma;
      int32_t* out = p.out + static_cast<long long>(b) * n;
      for (int i = 0; i < j; ++i) out[i] = __ldg(xb + i);
      out[j] = tok < 0 ? 0 : tok;
      for (int i = j + 1; i < n; ++i) out[i] = -1;
      p.n_acc[b] = j;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(kT, 1) sample_kernel(const SampleParams p) {
  __shared__ Red red;
  extern __shared__ unsigned dyn_hist[];  // kHistBytes
  const int row = blockIdx.x;
  const int V = p.V;
  const float* z = p.logits + static_cast<long long>(row) * V;
  float* probs = p.probs ? p.probs + static_cast<long long>(row) * V : nullptr;
  if (p.T == 0.f) {
    const int a = row_argmax(z, V, red);
    if (probs)
      for (int x = threadIdx.x; x < V; x += kT) probs[x] = x == a ? 1.f : 0.f;
    if (threadIdx.x == 0) p.tokens[row] = a;
    return;
  }
  RowDist dist = make_dist(z, V, p.T, p.top_p, red, dyn_hist);
  if (probs)
        visit_row(z, nullptr, V, [&](int x, float zv, float) { probs[x] = dist.p_of(zv); });
  DrawWeights dw;
  dw.p = dist;
  dw.q = nullptr;
  const int t = draw(dw, V, __ldg(p.u + row), kTotalFromChunks, kLastPosLazy, red);
  if (threadIdx.x == 0) p.tokens[row] = t < 0 ? 0 : t;
}

// ------------------------------------------------------- constrained rows
// Constrained generation ("Build a Speculative Decoding Engine ...", the
// question on JSON / grammar constraints): the target and the draft apply the
// same allowed-token mask before their probabilities are formed.  A masked
// logit becomes -inf, so its probability is 0 after the softmax and the rule
// runs unchanged.  Grid (row, 256-word chunk); a thread owns one mask word
// (32 ids) and rewrites only the float4 groups holding a disallowed id.  Every
// CTA first counts its row's allowed ids (the whole mask row, from L2): a row
// whose mask allows nothing is left as it is and flagged.
constexpr int kMaskThreads = 256;

__global__ void __launch_bounds__(kMaskThreads) mask_logits_kernel(float* logits, const uint32_t* allowed,
                                                                   int V, int vec4, int32_t* status) {
  __shared__ int s_cnt[kMaskThreads / 32];
  const int row = blockIdx.y;
  const int W = (V + 31) / 32;
  const uint32_t* a = allowed + static_cast<long long>(row) * W;
  float* z = logits + static_cast<long long>(row) * V;
  int cnt = 0;
  // 8 mask words per thread in flight at a time (the count is latency-bound)
  for (int w0 = threadIdx.x; w0 < W; w0 += 8 * kMaskThreads) {
    uint32_t bits[8];
#pragma unroll
    for (int k = 0; k < 8; ++k) {
      const int w = w0 + k * kMaskThreads;
      bits[k] = w < W ? __ldg(a + w) : 0u;
      if (w == W - 1 && (V & 31)) bits[k] &= (1u << (V & 31)) - 1u;  // ids past V are not tokens
    }
#pragma unroll
    for (int k = 0; k < 8; ++k) cnt += __popc(bits[k]);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) cnt += __shfl_xor_sync(0xffffffffu, cnt, o);
  if ((threadIdx.x & 31) == 0) s_cnt[threadIdx.x >> 5] = cnt;
  __syncthreads();
  int total = 0;
#pragma unroll
  for (int k = 0; k < kMaskThreads / 32; ++k) total += s_cnt[k];
  if (total == 0) {
    if (threadIdx.x == 0 && blockIdx.x == 0) set_status(status, SPEC_DEV_EMPTY_MASK);
    return;
  }
  const int w = blockIdx.x * kMaskThreads + threadIdx.x;
  if (w >= W) return;
  const uint32_t bits = __ldg(a + w);
  const int x0 = w * 32, n = min(32, V - x0);
  if (n == 32 && bits == 0xffffffffu) return;
  if (vec4 && n == 32) {
    float4* z4 = reinterpret_cast<float4*>(z + x0);
#pragma unroll
    for (int g = 0; g < 8; ++g) {
      const uint32_t nib = (bits >> (4 * g)) & 0xFu;
      if (nib == 0xFu) continue;
      float4 v = z4[g];
      if (!(nib & 1u)) v.x = -INFINITY;
      if (!(nib & 2u)) v.y = -INFINITY;
      if (!(nib & 4u)) v.z = -INFINITY;
      if (!(nib & 8u)) v.w = -INFINITY;
      z4[g] = v;
    }
  } else {
    for (int k = 0; k < n; ++k)
      if (!((bits >> k) & 1u)) z[x0 + k] = -INFINITY;
  }
}

// ------------------------------------------------------------- tree accept
// The acceptance walk over one sequence's draft tree ("Speculative Decoding:
// Speeding Sequential Generation", Tree-Based Drafting: the accept/reject test
// applied per node), one CTA per sequence.  At the current node the children
// are tried in index order with the node's target distribution p' (after T /
// top-p): child c is accepted iff u[c] < min(1, p'(x_c) / q(x_c)), q being the
// distribution the siblings were drawn from; after each rejected child p' is
// replaced by norm(max(0, p' - q)) (kept when that mass is <= 1e-8).  The
// first accepted child becomes the current node; when none is (or the node is
// a leaf) one token is drawn from p' with u[0] and the walk ends.  T = 0: move
// to the first child whose token is the argmax, else emit the argmax.
//
// p' starts as the softmax row itself (recomputed from the logits); the
// residuals after rejected siblings are kept in closed form (below).  Sums
// and the draw use the same 2^-52 fixed-point weights as the chain rule.

// The current node's target distribution during the walk.  After k rejected
// siblings (all drawn from the node's draft distribution q) the residual
// p_k = norm(max(0, p_{k-1} - q)) has the closed form
//   p_k = max(0, p - C_k q) / T_k,  C_k = C_{k-1} + T_{k-1},
//   T_k = sum_x max(0, p - C_k q),  C_0 = 0, T_0 = 1,
// (max(0, max(0, p - C q) / T - q) = max(0, p - (C + T) q) / T), so the walk
// carries two scalars instead of materialising a row per rejection.
// Weights: max(0, p - c q) with q set (unnormalised), p itself without.
struct TreeWeights {
  RowDist p;
  const float* q;   // the node's draft distribution, or nullptr: p itself
  float c;          // coefficient of q
  float inv_t;      // 1 / sum of the weights (base() is a distribution)
  SPEC_DEVINL const float* src() const { return p.z; }
  SPEC_DEVINL float w_of(float sv, float qv) const {
    const float v = p.p_of(sv);
    return q ? fmaxf(v - c * qv, 0.f) : v;
  }
  SPEC_DEVINL float base(int x) const {
    return q ? w_of(__ldcg(p.z + x), __ldcg(q + x)) * inv_t : p.p(x);
  }
  SPEC_DEVINL unsigned long long fx_of(float sv, float qv) const {
    return static_cast<unsigned long long>(w_of(sv, qv) * kFix52);
  }
  SPEC_DEVINL unsigned long long fx(int x) const {
    return fx_of(__ldcg(p.z + x), q ? __ldcg(q + x) : 0.f);
  }
};

__global__ void __launch_bounds__(kT, 1) tree_accept_kernel(const TreeAcceptParams p) {
  __shared__ Red red;
  extern __shared__ unsigned dyn_hist[];  // kHistBytes
  __shared__ int s_flag;
  const int b = blockIdx.x;
  const int n = p.n, V = p.V;
  const long long row0 = static_cast<long long>(b) * n;
  const float* zb = p.logits + row0 * V;
  const int32_t* tok = p.tokens + row0;
  const int32_t* par = p.parents + row0;
  int32_t* out = p.out + row0;
  int32_t* path = p.path + row0;
  for (int i = threadIdx.x; i < n; i += kT) {
    out[i] = -1;
    path[i] = -1;
  }
  if (threadIdx.x == 0) {
    bool ok = __ldg(par) == -1;
    for (int i = 1; i < n; ++i) {
      const int pi = __ldg(par + i);
      ok = ok && pi >= 0 && pi < i;
    }
    if (!ok) {
      set_status(p.status, SPEC_DEV_BAD_TREE);
      p.n_acc[b] = 0;
    }
    s_flag = ok;
  }
  __syncthreads();
  if (!s_flag) return;

  int cur = 0, m = 0;
  if (p.T == 0.f) {
    for (;;) {
      const int a = row_argmax(zb + static_cast<long long>(cur) * V, V, red);
      if (threadIdx.x == 0) {
        int nxt = -1;
        for (int c = cur + 1; c < n && nxt < 0; ++c)
          if (__ldg(par + c) == cur && __ldg(tok + c) == a) nxt = c;
        out[m] = a;
        if (nxt >= 0) path[m] = nxt;
        else p.n_acc[b] = m;
        s_flag = nxt;
      }
      __syncthreads();
      if (s_flag < 0) return;
      cur = s_flag;
      ++m;
    }
  }

  const float* ub = p.u + row0;
  for (;;) {
    const float* qrow = p.q + (row0 + cur) * V;
    TreeWeights tw;
    tw.p = make_dist(zb + static_cast<long long>(cur) * V, V, p.T, p.top_p, red, dyn_hist);
    tw.q = nullptr;
    tw.c = 0.f;
    tw.inv_t = 1.f;
    int nxt = -1;
    for (int c = cur + 1; c < n; ++c) {
      if (__ldg(par + c) != cur) continue;
      if (threadIdx.x == 0) {
        const int x = __ldg(tok + c);
        bool accept = false;
        if (x < 0 || x >= V) {
          set_status(p.status, SPEC_DEV_BAD_TOKEN);
        } else {
          const float qx = __ldcg(qrow + x);
          if (!(qx > 0.f)) {
            set_status(p.status, SPEC_DEV_Q_ZERO);
          } else {
            const float a = fminf(1.0f, tw.base(x) / qx);
            accept = __ldg(ub + c) < a;
          }
        }
        s_flag = accept;
      }
      __syncthreads();
      if (s_flag) {
        nxt = c;
        break;
      }
      // rejected: p' <- norm(max(0, p' - q)) unless that mass is ~0
      TreeWeights nx = tw;
      const float t_cur = tw.q ? 1.f / tw.inv_t : 1.f;
      nx.q = qrow;
      nx.c = (tw.q ? tw.c : 0.f) + t_cur;
      unsigned long long total;
      int last_pos;
      weights_total(nx, V, red, total, last_pos);
      const double t_new = static_cast<double>(total) / 4503599627370496.0;
      if (t_new > kResidualFallback * static_cast<double>(t_cur)) {
        nx.inv_t = static_cast<float>(1.0 / t_new);
        tw = nx;
      }
    }
    if (nxt >= 0) {
      if (threadIdx.x == 0) {
        path[m] = nxt;
        out[m] = __ldg(tok + nxt);
      }
      cur = nxt;
      ++m;
      continue;
    }
    const int t = draw(tw, V, __ldg(ub), kTotalFromChunks, kLastPosLazy, red);
    if (threadIdx.x == 0) {
      out[m] = t < 0 ? 0 : t;
      p.n_acc[b] = m;
    }
    return;
  }
}

// ------------------------------------------------------------- tree commit
// Moves the accepted path's keys / values from the flattened slots L0 + node
// to L0 + 1 .. L0 + m (depth order); one CTA per (layer, sequence, KV head).
// A destination may be the source of an earlier path entry (path [2, 5]
// reads slot 2 and writes it), so every source row is loaded before any row
// is stored.
constexpr int kCommitThreads = 256;
constexpr int kCommitPer = 8;  // uint4 per thread: 64 nodes x (K, V) x 128 dims / 256 threads

SPEC_DEVINL bool tree_path_ok(const int32_t* path, int m, int n) {
  int prev = 0;
  for (int d = 0; d < m; ++d) {
    const int s = __ldg(path + d);
    if (s <= prev || s >= n) return false;
    prev = s;
  }
  return true;
}

__global__ void __launch_bounds__(kCommitThreads) tree_commit_kernel(const TreeCommitParams p) {
  const int layer = blockIdx.y;
  const int b = blockIdx.x / p.Hkv, h = blockIdx.x % p.Hkv;
  const int n = p.n;
  const int m = __ldg(p.n_acc + b);
  const int len = p.len[b];
  const int L0 = len - n;
  const int32_t* path = p.path + static_cast<long long>(b) * n;
  if (m < 0 || m >= n || L0 < 0 || len > p.cap || !tree_path_ok(path, m, n)) return;
  const long long base =
      ((static_cast<long long>(layer) * p.B + b) * p.Hkv + h) * p.cap * p.hd;
  const int vec = p.hd / 8;  // uint4 per row
  const int per_side = m * vec;
  uint4 r[kCommitPer];
  int dst[kCommitPer];
#pragma unroll
  for (int k = 0; k < kCommitPer; ++k) {
    const int e = threadIdx.x + k * kCommitThreads;  // over [side][depth][vec]
    dst[k] = -1;
    if (e < 2 * per_side) {
      const int side = e / per_side, rem = e % per_side;
      const int d = rem / vec, c = rem % vec;
      const int src = __ldg(path + d);
      if (src != d + 1) {
        const uint4* s = reinterpret_cast<const uint4*>((side ? p.v : p.k) + base +
                                                         static_cast<long long>(L0 + src) * p.hd) + c;
        r[k] = *s;
        dst[k] = e;
      }
    }
  }
  __syncthreads();
#pragma unroll
  for (int k = 0; k < kCommitPer; ++k) {
    const int e = dst[k];
    if (e < 0) continue;
    const int side = e / per_side, rem = e % per_side;
    const int d = rem / vec, c = rem % vec;
    uint4* t = reinterpret_cast<uint4*>((side ? p.v : p.k) + base +
                                        static_cast<long long>(L0 + d + 1) * p.hd) + c;
    *t = r[k];
  }
}

// len = L0 + 1 + m after the copies (a separate launch: the copies read len).
__global__ void tree_len_kernel(int32_t* len, const int32_t* path, const int32_t* n_acc, int B,
                                int n, int cap, int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int m = n_acc[b];
  const int l = len[b];
  if (m < 0 || m >= n || !tree_path_ok(path + static_cast<long long>(b) * n, m, n)) {
    set_status(status, SPEC_DEV_BAD_TREE);
    return;
  }
  if (l < n || l > cap) {
    set_status(status, SPEC_DEV_KV_OVERFLOW);
    return;
  }
  len[b] = l - n + 1 + m;
}

__global__ void truncate_kernel(int32_t* len, const int32_t* n_acc, int B, int gamma,
                                int32_t* status) {
  grid_dep_wait();
  grid_dep_launch();
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int n = n_acc[b];
  if (n < 0 || n > gamma) {
    set_status(status, SPEC_DEV_BAD_NACC);
    return;
  }
  const int drop = gamma - n;
  if (len[b] < drop) {
    set_status(status, SPEC_DEV_KV_OVERFLOW);
    return;
  }
  len[b] -= drop;
}

cudaError_t launch_pdl(const void* fn, dim3 grid, dim3 block, void** args, cudaStream_t stream,
                       bool pdl) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelExC(&cfg, fn, args);
}

}  // namespace

// The per-sequence kernels take kHistBytes of dynamic shared memory (above
// the 48 KB default): set once per device.
cudaError_t per_seq_smem_attrs() {
  static PerDevice<cudaError_t> done;
  cudaError_t e = cudaErrorInvalidDevice;
  if (!done.get(
          [] {
            const void* fns[3] = {reinterpret_cast<const void*>(accept_seq_kernel),
                                  reinterpret_cast<const void*>(sample_kernel),
                                  reinterpret_cast<const void*>(tree_accept_kernel)};
            for (const void* f : fns) {
              const cudaError_t r = cudaFuncSetAttribute(
                  f, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kHistBytes));
              if (r != cudaSuccess) return r;
            }
            return cudaSuccess;
          },
          &e))
    return cudaErrorInvalidDevice;
  return e;
}

// CTAs of the cooperative accept grid the current device keeps resident.
int accept_grid_capacity() {
  static PerDevice<int> cap;
  int v = 0;
  if (!cap.get(
          [] {
            int dev = 0, sms = 0, per = 0;
            if (cudaGetDevice(&dev) != cudaSuccess) return 0;
            if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
              return 0;
            if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per, accept_grid_kernel, kAT, 0) !=
                cudaSuccess)
              return 0;
            return sms * per;
          },
          &v))
    return 0;
  return v;
}

// Work units per row of a grid pass over every row: the count (at most
// max_units) that minimises the busiest CTA's share -- rounds of units over
// the grid times the ids of a unit plus a fixed cost per unit (its
// reductions, row statistics and bin flush), in ids.
int accept_row_split(long long rows, int V, int max_units, int grid, long long fixed) {
  int best = 1;
  long long best_cost = -1;
  for (int sl = 1; sl <= max_units; ++sl) {
    const long long rounds = (rows * sl + grid - 1) / grid;
    const long long cost = rounds * ((V + sl - 1) / sl + fixed);
    if (best_cost < 0 || cost < best_cost) {
      best_cost = cost;
      best = sl;
    }
  }
  return best;
}

cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  const long long rows = static_cast<long long>(p.B) * (p.gamma + 1);
  const int cap = accept_grid_capacity();
  if (!p.grid || rows > kAcceptGridRows || cap <= 0) {
    const cudaError_t e = per_seq_smem_attrs();
    if (e != cudaSuccess) return e;
    AcceptParams a = p;
    accept_seq_kernel<<<p.B, kT, kHistBytes, stream>>>(a);
    return cudaGetLastError();
  }
  const long long units = rows * p.S;
  const int grid = static_cast<int>(std::min<long long>(cap, std::max<long long>(units, 1)));
  AcceptParams a = p;
  a.S1 = accept_row_split(rows, p.V, p.S, grid, 2048);
  a.SL = accept_row_split(rows, p.V, p.S, grid, 4096);
  cudaError_t e = cudaMemsetAsync(p.bar, 0, sizeof(unsigned), stream);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kAT);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, accept_grid_kernel, a);
}

cudaError_t launch_sample(const SampleParams& p, cudaStream_t stream) {
  if (p.R == 0) return cudaSuccess;
  const cudaError_t e = per_seq_smem_attrs();
  if (e != cudaSuccess) return e;
  sample_kernel<<<p.R, kT, kHistBytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_truncate(int32_t* len, const int32_t* n_acc, int B, int gamma, int32_t* status,
                            cudaStream_t stream, bool pdl) {
  if (B == 0) return cudaSuccess;
  void* args[] = {&len, const_cast<int32_t**>(&n_acc), &B, &gamma, &status};
  return launch_pdl(reinterpret_cast<const void*>(truncate_kernel), dim3((B + 127) / 128),
                    dim3(128), args, stream, pdl);
}

cudaError_t launch_mask_logits(float* logits, const uint32_t* allowed, int rows, int V, int32_t* status,
                               cudaStream_t stream) {
  if (rows == 0) return cudaSuccess;
  const int W = (V + 31) / 32;
  const int vec4 = (V % 4 == 0 && reinterpret_cast<uintptr_t>(logits) % 16 == 0) ? 1 : 0;
  const dim3 grid((W + kMaskThreads - 1) / kMaskThreads, rows);
  mask_logits_kernel<<<grid, kMaskThreads, 0, stream>>>(logits, allowed, V, vec4, status);
  return cudaGetLastError();
}

cudaError_t launch_tree_accept(const TreeAcceptParams& p, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  const cudaError_t e = per_seq_smem_attrs();
  if (e != cudaSuccess) return e;
  tree_accept_kernel<<<p.B, kT, kHistBytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_tree_commit(const TreeCommitParams& p, cudaStream_t stream) {
  if (p.B == 0) return cudaSuccess;
  if (p.n > 1 && p.L > 0 && p.Hkv > 0) {
    tree_commit_kernel<<<dim3(p.B * p.Hkv, p.L), kCommitThreads, 0, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
  }
  int32_t* len = p.len;
  const int32_t* path = p.path;
  const int32_t* n_acc = p.n_acc;
  int B = p.B, n = p.n, cap = p.cap;
  int32_t* status = p.status;
  void* args[] = {&len, const_cast<int32_t**>(&path), const_cast<int32_t**>(&n_acc), &B, &n, &cap,
                  &status};
  return launch_pdl(reinterpret_cast<const void*>(tree_len_kernel), dim3((B + 127) / 128),
                    dim3(128), args, stream, true);
}

}  // namespace spec
