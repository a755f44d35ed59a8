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
// Structure per CTA (1024 threads):
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

// Row statistics of softmax(z / T): block max and sum of exp2((z-max)*c).
__device__ void row_stats(const float* z, int V, float c, Red& r, float& m_out, float& s_out) {
  float m = -INFINITY, s = 0.f;
  for (int x = threadIdx.x; x < V; x += kT) {
    const float v = __ldcg(z + x);
    if (v > m) {
      s = (m == -INFINITY ? 0.f : s * exp2f((m - v) * c)) + 1.0f;
      m = v;
    } else {
      s += exp2f((v - m) * c);
    }
  }
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
  for (int x = threadIdx.x; x < V; x += kT) {
    const float v = __ldcg(z + x);
    if (v > best || (v == best && x < bi)) {
      best = v;
      bi = x;
    }
  }
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
  SPEC_DEVINL float e(int x) const { return exp2f((__ldcg(z + x) - m) * c); }
  SPEC_DEVINL float p(int x) const {
    const float v = e(x);
    return v >= tau ? v / Z : 0.f;
  }
};

// Softmax statistics and (top_p < 1) the nucleus threshold of one row.
__device__ RowDist make_dist(const float* z, int V, float T, float top_p, Red& r) {
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
  for (int x = threadIdx.x; x < V; x += kT) tot += static_cast<unsigned long long>(d.e(x) * kFix40);
  tot = block_sum_u64(tot, r);
  const double target = static_cast<double>(top_p) * static_cast<double>(tot);
  uint32_t prefix = 0;
  unsigned long long above = 0;  // mass strictly above the current prefix range
  for (int level = 0; level < 4; ++level) {
    const int shift = 24 - 8 * level;
    const uint32_t hi_mask = level == 0 ? 0u : (0xFFFFFFFFu << (shift + 8));
    for (int i = threadIdx.x; i < 256; i += kT) r.hist[i] = 0ull;
    __syncthreads();
    for (int x = threadIdx.x; x < V; x += kT) {
      const float v = d.e(x);
      const uint32_t bits = __float_as_uint(v);
      if ((bits & hi_mask) == prefix)
        atomicAdd(&r.hist[(bits >> shift) & 0xFFu], static_cast<unsigned long long>(v * kFix40));
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
  for (int x = threadIdx.x; x < V; x += kT) {
    const float v = d.e(x);
    z_kept += v >= d.tau ? v : 0.f;
  }
  d.Z = block_sum_f(z_kept, r);
  return d;
}

// Weight of id x for the final draw: the residual max(0, p - q) or p itself.
struct DrawWeights {
  RowDist p;
  const float* q;  // nullptr: draw from p
  SPEC_DEVINL float w(int x) const {
    const float pv = p.p(x);
    return q ? fmaxf(pv - __ldcg(q + x), 0.f) : pv;
  }
  SPEC_DEVINL unsigned long long fx(int x) const {
    return static_cast<unsigned long long>(w(x) * kFix52);
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

// Inverse-CDF draw: the smallest id t with sum_{x<=t} fx(x) > floor(u * total).
// `total` is the exact fixed-point sum; `last_pos` the last id with fx > 0.
__device__ int draw(const DrawWeights& dw, int V, float u, unsigned long long total,
                    int last_pos, Red& r) {
  const unsigned long long thr =
      static_cast<unsigned long long>(static_cast<double>(u) * static_cast<double>(total));
  unsigned long long run = 0;  // exact prefix before the current tile
  const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
  for (int base = 0; base < V; base += 4 * kT) {
    const int x0 = base + threadIdx.x * 4;
    unsigned long long f[4];
    unsigned long long mine = 0;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      f[k] = (x0 + k < V) ? dw.fx(x0 + k) : 0ull;
      mine += f[k];
    }
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

// Exact fixed-point total and last positive id of the draw weights.
__device__ void weights_total(const DrawWeights& dw, int V, Red& r, unsigned long long& total,
                              int& last_pos) {
  unsigned long long s = 0;
  int lp = -1;
  for (int x = threadIdx.x; x < V; x += kT) {
    const unsigned long long f = dw.fx(x);
    s += f;
    if (f) lp = x;
  }
  total = block_sum_u64(s, r);
  last_pos = block_max_i(lp, r);
}

__global__ void __launch_bounds__(kT, 1) accept_kernel(const AcceptParams p) {
  __shared__ Red red;
  __shared__ int s_flag;
  const int b = blockIdx.x;
  const int gamma = p.gamma, V = p.V, n = gamma + 1;
  grid_dep_wait();
  grid_dep_launch();
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
    dist = make_dist(zb + static_cast<long long>(i) * V, V, p.T, p.top_p, red);
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
    dist = make_dist(zb + static_cast<long long>(gamma) * V, V, p.T, p.top_p, red);
    dw.p = dist;
    dw.q = nullptr;
  } else {
    dw.p = dist;
    dw.q = qb + static_cast<long long>(j) * V;
  }
  unsigned long long total;
  int last_pos;
  weights_total(dw, V, red, total, last_pos);
  if (dw.q && static_cast<double>(total) <= kResidualFallback * 4503599627370496.0) {
    dw.q = nullptr;  // residual mass numerically zero: draw from p
    weights_total(dw, V, red, total, last_pos);
  }
  const int t = draw(dw, V, __ldg(ub + gamma), total, last_pos, red);
  if (threadIdx.x == 0) {
    out[j] = t < 0 ? 0 : t;
    p.n_acc[b] = j;
  }
}

__global__ void __launch_bounds__(kT, 1) sample_kernel(const SampleParams p) {
  __shared__ Red red;
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
  RowDist dist = make_dist(z, V, p.T, p.top_p, red);
  if (probs)
    for (int x = threadIdx.x; x < V; x += kT) probs[x] = dist.p(x);
  DrawWeights dw;
  dw.p = dist;
  dw.q = nullptr;
  unsigned long long total;
  int last_pos;
  weights_total(dw, V, red, total, last_pos);
  const int t = draw(dw, V, __ldg(p.u + row), total, last_pos, red);
  if (threadIdx.x == 0) p.tokens[row] = t < 0 ? 0 : t;
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

cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream, bool pdl) {
  if (p.B == 0) return cudaSuccess;
  AcceptParams a = p;
  void* args[] = {&a};
  return launch_pdl(reinterpret_cast<const void*>(accept_kernel), dim3(p.B), dim3(kT), args,
                    stream, pdl);
}

cudaError_t launch_sample(const SampleParams& p, cudaStream_t stream) {
  if (p.R == 0) return cudaSuccess;
  sample_kernel<<<p.R, kT, 0, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_truncate(int32_t* len, const int32_t* n_acc, int B, int gamma, int32_t* status,
                            cudaStream_t stream, bool pdl) {
  if (B == 0) return cudaSuccess;
  void* args[] = {&len, const_cast<int32_t**>(&n_acc), &B, &gamma, &status};
  return launch_pdl(reinterpret_cast<const void*>(truncate_kernel), dim3((B + 127) / 128),
                    dim3(128), args, stream, pdl);
}

}  // namespace spec
