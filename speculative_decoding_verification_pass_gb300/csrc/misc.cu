// Small kernels of the verification pass: the embedding gather that opens a
// pass (and owns the per-pass cache bookkeeping), the seeded weight
// generator, and constant tables.
#include "common.cuh"
#include "internal.h"

namespace spec {

namespace {

// ---------------------------------------------------------------- embedding
// h[m] = E[token[m]] (fp32 residual stream), hb[m] = bf16(h[m] * g0) (the
// next GEMM's input; its RMSNorm scale is applied in that GEMM's epilogue
// from the sum-of-squares partials written here, one per 128 features).
// Block 0 also opens the pass: zeroes the stream-K / attention counters and,
// per sequence, records the current cache length as the position base,
// checks that gamma+1 new slots fit and advances the length.
__global__ void __launch_bounds__(256) embed_kernel(const EmbedParams p) {
  grid_dep_wait();
  grid_dep_launch();
  const int m = blockIdx.x;
  if (m == 0) {
    for (int i = threadIdx.x; i < p.n_counters; i += blockDim.x) p.counters[i] = 0;
    for (int b = threadIdx.x; b < p.B; b += blockDim.x) {
      const int L = p.len[b];
      const int32_t bad = seq_fit(L, p.n, p.cap, p.kv_table, p.kv_max_pages, p.kv_n_pages, b);
      p.pos_base[b] = L < 0 ? 0 : L;
      p.seq_ok[b] = bad ? 0 : 1;
      if (!bad)
        p.len[b] = L + p.n;
      else
        set_status(p.status, bad);
    }
  }
  int tok = p.tokens[m];
  if (tok < 0 || tok >= p.V) {
    if (threadIdx.x == 0) set_status(p.status, SPEC_DEV_BAD_TOKEN);
    tok = 0;
  }
  const uint16_t* row = p.embed + static_cast<long long>(tok) * p.d;
  // every lane of a warp runs the same iterations (the shuffles below)
  for (int base = 0; base < p.d; base += blockDim.x * 16) {
    const int f0 = base + threadIdx.x * 16;
    const bool act = f0 < p.d;
    float sq = 0.f;
    if (act) {
      const uint4 a = *reinterpret_cast<const uint4*>(row + f0);
      const uint4 c = *reinterpret_cast<const uint4*>(row + f0 + 8);
      const uint32_t w[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
      float g[16];  // gains loaded before any store (the stores could alias them)
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const float4 v = __ldg(reinterpret_cast<const float4*>(p.g0 + f0) + k);
        g[4 * k] = v.x;
        g[4 * k + 1] = v.y;
        g[4 * k + 2] = v.z;
        g[4 * k + 3] = v.w;
      }
      float* h = p.h + static_cast<long long>(m) * p.d + f0;
      uint16_t* hb = p.hb + static_cast<long long>(m) * p.d + f0;
#pragma unroll
      for (int k = 0; k < 8; ++k) {
        const float lo = bf16lo(w[k]), hi = bf16hi(w[k]);
        h[2 * k] = lo;
        h[2 * k + 1] = hi;
        const float x0 = lo * g[2 * k], x1 = hi * g[2 * k + 1];
        const uint16_t b0 = f32_to_bf16(x0), b1 = f32_to_bf16(x1);
        hb[2 * k] = b0;
        hb[2 * k + 1] = b1;
        if (p.hb_lo) {
          uint16_t* hl = p.hb_lo + static_cast<long long>(m) * p.d + f0;
          hl[2 * k] = f32_to_bf16(x0 - bf16_to_f32(b0));
          hl[2 * k + 1] = f32_to_bf16(x1 - bf16_to_f32(b1));
        }
        sq += lo * lo;
        sq += hi * hi;
      }
    }
    // 8 consecutive threads cover one 128-feature tile
    sq += __shfl_xor_sync(0xffffffffu, sq, 1);
    sq += __shfl_xor_sync(0xffffffffu, sq, 2);
    sq += __shfl_xor_sync(0xffffffffu, sq, 4);
    if (act && (threadIdx.x & 7) == 0)
      p.ssq[static_cast<long long>(f0 / 128) * p.ssq_ld + m] = sq;
  }
}

// ------------------------------------------------------------ weight init
// Philox4x64-10 (Salmon, Moraes, Dror, Shaw, SC 2011): 10 rounds of two
// 64x64->128-bit multiplies with the key bumped by the Weyl constants
// between rounds.
SPEC_DEVINL void philox4x64_10(uint64_t c0, uint64_t c1, uint64_t c2, uint64_t c3, uint64_t k0,
                               uint64_t k1, uint64_t (&o)[4]) {
  const uint64_t M0 = 0xD2E7470EE14C6C93ull, M1 = 0xCA5A826395121157ull;
  const uint64_t W0 = 0x9E3779B97F4A7C15ull, W1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += W0;
      k1 += W1;
    }
    const uint64_t hi0 = __umul64hi(M0, c0), lo0 = M0 * c0;
    const uint64_t hi1 = __umul64hi(M1, c2), lo1 = M1 * c2;
    const uint64_t n0 = hi1 ^ c1 ^ k0, n1 = lo1, n2 = hi0 ^ c3 ^ k1, n3 = lo0;
    c0 = n0;
    c1 = n1;
    c2 = n2;
    c3 = n3;
  }
  o[0] = c0;
  o[1] = c1;
  o[2] = c2;
  o[3] = c3;
}

// Nearest bf16 of a double (ties to even), on the fp64 bit pattern.
SPEC_DEVINL uint16_t f64_to_bf16(double x) {
  unsigned long long u = static_cast<unsigned long long>(__double_as_longlong(x));
  const unsigned long long lsb = (u >> 45) & 1ull;
  u = (u + 0x0FFFFFFFFFFFull + lsb) & ~0x1FFFFFFFFFFFull;
  const float f = static_cast<float>(__longlong_as_double(static_cast<long long>(u)));
  return static_cast<uint16_t>(__float_as_uint(f) >> 16);
}

__global__ void init_weights_kernel(uint16_t* dst, long long rows, long long cols, int tid,
                                    uint64_t seed, int block_rows, int row_stride_rows) {
  const long long n = rows * cols;
  const long long nblk = (n + 3) / 4;
  const double kTwoM53 = 1.1102230246251565e-16;  // 2^-53
  const double kTwoPi = 6.283185307179586;         // 2 * fl(pi)
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < nblk;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    uint64_t o[4];
    philox4x64_10(static_cast<uint64_t>(i) + 1ull, static_cast<uint64_t>(tid), 0ull, 0ull, seed,
                  0ull, o);
#pragma unroll
    for (int pr = 0; pr < 2; ++pr) {
      const double u = (static_cast<double>(o[2 * pr] >> 11) + 0.5) * kTwoM53;
      const double v = (static_cast<double>(o[2 * pr + 1] >> 11) + 0.5) * kTwoM53;
      const double rad = sqrt(-2.0 * log(u));
      double s, c;
      sincos(kTwoPi * v, &s, &c);
      const double z[2] = {rad * c, rad * s};
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const long long e = 4 * i + 2 * pr + k;
        if (e >= n) continue;
        const long long row = e / cols, col = e - row * cols;
        const long long prow = (row / block_rows) * row_stride_rows + row % block_rows;
        dst[prow * cols + col] = f64_to_bf16(0.02 * z[k]);
      }
    }
  }
}

__global__ void fill_f32_kernel(float* dst, long long n, float v) {
  for (long long i = blockIdx.x * static_cast<long long>(blockDim.x) + threadIdx.x; i < n;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    dst[i] = v;
}

// Rotary frequency of pair i in turns per position, theta^(-2i/hd) / (2 pi),
// split as hi + lo floats (the QKV epilogue removes whole turns exactly, so
// the sine is evaluated on a reduced argument at any position).
__global__ void rope_table_kernel(float2* dst, int hd, double theta) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= hd / 2) return;
  const double two_pi = 6.283185307179586;
  const double f = pow(theta, -2.0 * i / hd) / two_pi;
  const float hi = static_cast<float>(f);
  dst[i] = make_float2(hi, static_cast<float>(f - static_cast<double>(hi)));
}

// One bounded wait of the persistent forward's grid barrier on a caller's
// counter: the self-test of the timeout path (a counter that nothing
// advances ends the wait with the timeout bit set, and the kernel returns).
__global__ void wait_probe_kernel(const unsigned* ctr, unsigned target, unsigned long long limit_ns,
                                  int32_t* status) {
  __shared__ int abort;
  if (threadIdx.x == 0) {
    abort = 0;
    wait_count(ctr, target, &abort, status, limit_ns);
  }
}

}  // namespace

cudaError_t launch_wait_probe(const unsigned* ctr, unsigned target, unsigned long long limit_ns,
                              int32_t* status, cudaStream_t stream) {
  wait_probe_kernel<<<1, 32, 0, stream>>>(ctr, target, limit_ns, status);
  return cudaGetLastError();
}

cudaError_t launch_embed(const EmbedParams& p, cudaStream_t stream, bool pdl) {
  const int M = p.B * p.n;
  if (M == 0) return cudaSuccess;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(M);
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, embed_kernel, p);
}

cudaError_t launch_init_weights(uint16_t* dst, long long rows, long long cols, int tid,
                                uint64_t seed, int block_rows, int row_stride_rows,
                                cudaStream_t stream) {
  const long long nblk = (rows * cols + 3) / 4;
  long long grid = (nblk + 255) / 256;
  if (grid > 152 * 32) grid = 152 * 32;
  if (grid < 1) grid = 1;
  init_weights_kernel<<<static_cast<int>(grid), 256, 0, stream>>>(dst, rows, cols, tid, seed,
                                                                   block_rows, row_stride_rows);
  return cudaGetLastError();
}

cudaError_t launch_fill_f32(float* dst, long long n, float v, cudaStream_t stream) {
  fill_f32_kernel<<<64, 256, 0, stream>>>(dst, n, v);
  return cudaGetLastError();
}

cudaError_t launch_rope_table(float2* dst, int hd, double theta, cudaStream_t stream) {
  rope_table_kernel<<<1, 128, 0, stream>>>(dst, hd, theta);
  return cudaGetLastError();
}

}  // namespace spec
