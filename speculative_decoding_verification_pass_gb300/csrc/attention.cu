// Split-KV attention of the gamma+1 new positions over the bf16 KV cache.
//
// One verification pass feeds gamma+1 queries per sequence through attention
// over the cached context plus the new block (lattice notes: the target
// scores all k drafted positions and the next-token slot in one call; the
// pass still reads "the KV cache" on top of the weights).  Query j of the
// block sits at position len+j and sees keys 0..len+j (causal inside the
// block).  Grouped-query attention: the G = n_heads / n_kv_heads query heads
// of a KV head share its keys, so a CTA takes one (sequence, KV head, chunk
// of 128 keys) and all n*G query rows of that group, reading each key and
// value once.
//
// Per CTA: the key/value chunk is staged in shared memory with cp.async
// (16-byte copies, XOR-swizzled rows so ldmatrix is conflict-free); query rows
// go through in tiles of 16; each warp takes 32 of the 128 keys and computes
// S = Q K^T and O = P V with mma.m16n8k16 (bf16 in, fp32 accumulate) and an
// exp2-domain softmax; q and P enter as bf16 pairs (hi + lo, two MMAs each),
// so only the cache itself is bf16-rounded; the four warps' (max, sum, O) are merged in shared
// memory into the CTA's partial.  The last CTA of a (sequence, KV head) to
// finish (atomic counter) merges all chunks' partials in chunk order by
// log-sum-exp and writes the bf16 output rows: deterministic, no waits on
// other CTAs.
#include "attn_common.cuh"
#include "common.cuh"
#include "internal.h"

namespace spec {

namespace {

constexpr int kThreads = 128;
constexpr int kChunk = kAttnChunk;  // keys per CTA
constexpr int kKeysPerWarp = kChunk / 4;
constexpr int kMaxChunks = kAttnMaxChunks;
// the combine stages [chunks][16] maxima and sums in the key/value area
static_assert(2 * 16 * kMaxChunks * 4 <= 2 * kChunk * 64 * 2, "combine scratch exceeds the K/V area");

template <int HD>
struct AttnSmem {
  static constexpr int kRowB = HD * 2;
  static constexpr int kOStride = HD + 8;  // floats per row of a warp partial
  static constexpr size_t kK = 0;
  static constexpr size_t kV = kK + static_cast<size_t>(kChunk) * kRowB;
  static constexpr size_t kQ = kV + static_cast<size_t>(kChunk) * kRowB;
  static constexpr size_t kQlo = kQ + 16 * kRowB;
  static constexpr size_t kO = kQlo + 16 * kRowB;
  static constexpr size_t kM = kO + 4ull * 16 * kOStride * 4;
  static constexpr size_t kL = kM + 4 * 16 * 4;
  static constexpr size_t kFlag = kL + 4 * 16 * 4;
  static constexpr size_t kBytes = kFlag + 16;
};

template <int HD>
__global__ void __launch_bounds__(kThreads) attn_splitkv_kernel(const AttnParams p) {
  using L = AttnSmem<HD>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int s = blockIdx.x, kvh = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.H / p.Hkv;
  grid_dep_wait();
  grid_dep_launch();

  const int Lb = p.pos_base[b];
  const int Tk = min(Lb + p.n, p.cap);
  const int k0 = s * kChunk;
  if (k0 >= Tk) return;  // this chunk is past the sequence
  const int ns = (Tk + kChunk - 1) / kChunk;
  const int nk = min(kChunk, Tk - k0);

  const uint32_t sK = smem_u32(smem + L::kK), sV = smem_u32(smem + L::kV),
                 sQ = smem_u32(smem + L::kQ), sQlo = smem_u32(smem + L::kQlo);
  const bool lo = p.q_lo != nullptr;
  float* Ow = reinterpret_cast<float*>(smem + L::kO);
  float* Mw = reinterpret_cast<float*>(smem + L::kM);
  float* Lw = reinterpret_cast<float*>(smem + L::kL);
  int* flag = reinterpret_cast<int*>(smem + L::kFlag);

  // ---- stage this chunk's keys and values (rows past the end are zero)
  const KVMap map{p.kv_table, p.kv_max_pages, p.kv_n_pages, p.Hkv, p.cap, HD};
  constexpr int kCPR = HD / 8;  // 16-byte chunks per row
  for (int idx = tid; idx < kChunk * kCPR; idx += kThreads) {
    const int i = idx / kCPR, c = idx % kCPR;
    const int row = i < nk ? i : 0;
    const long long g = map.row(b, kvh, k0 + row) + c * 8;
    const int bytes = i < nk ? 16 : 0;
    cp_async16(sK + swz<HD>(i, c), p.kcache + g, bytes);
    cp_async16(sV + swz<HD>(i, c), p.vcache + g, bytes);
  }
  cp_async_wait_all();
  __syncthreads();

  const int R = p.R;
  const int qdim = p.H * HD;
  const int kw0 = warp * kKeysPerWarp;
  const int g8 = lane >> 2, t4 = lane & 3;
  float* part_o = p.part_o + ((static_cast<long long>(b) * p.Hkv + kvh) * p.splits + s) * R * HD;
  float* part_ml = p.part_ml + ((static_cast<long long>(b) * p.Hkv + kvh) * p.splits + s) * R * 2;

  for (int qt = 0; qt * 16 < R; ++qt) {
    // ---- query tile: rows r = qt*16 + i, r = j*G + g -> token b*n+j, head kvh*G+g
    for (int idx = tid; idx < 16 * kCPR; idx += kThreads) {
      const int i = idx / kCPR, c = idx % kCPR;
      const int r = qt * 16 + i;
      uint4 val = make_uint4(0, 0, 0, 0), vlo = make_uint4(0, 0, 0, 0);
      if (r < R) {
        const int j = r / G, g = r % G;
        const long long off = (static_cast<long long>(b) * p.n + j) * qdim + (kvh * G + g) * HD + c * 8;
        val = *reinterpret_cast<const uint4*>(p.q + off);
        if (lo) vlo = *reinterpret_cast<const uint4*>(p.q_lo + off);
      }
      *reinterpret_cast<uint4*>(smem + L::kQ + swz<HD>(i, c)) = val;
      *reinterpret_cast<uint4*>(smem + L::kQlo + swz<HD>(i, c)) = vlo;
    }
    __syncthreads();

    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.f, 0.f};
    float oacc[HD / 8][4];
#pragma unroll
    for (int i = 0; i < HD / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;

    if (kw0 < nk) {
      // ---- S = Q K^T over this warp's 32 keys (4 n8 tiles)
      float sacc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
        ldsm_x4(sQ + swz<HD>(lane & 15, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
        if (lo) ldsm_x4(sQlo + swz<HD>(lane & 15, kk * 2 + (lane >> 4)), l0, l1, l2, l3);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int key = kw0 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sK + swz<HD>(key, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma_bf16(sacc[np * 2], a0, a1, a2, a3, b0, b1);
          mma_bf16(sacc[np * 2 + 1], a0, a1, a2, a3, b2, b3);
          if (lo) {  // q = q_hi + q_lo
            mma_bf16(sacc[np * 2], l0, l1, l2, l3, b0, b1);
            mma_bf16(sacc[np * 2 + 1], l0, l1, l2, l3, b2, b3);
          }
        }
      }
      // ---- mask (causal within the block, chunk end) and exp2-domain softmax
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = qt * 16 + g8 + hr * 8;
        const bool rv = r < R;
        const int jn = rv ? r / G : 0;
        const uint64_t am = (p.anc && rv) ? __ldg(p.anc + static_cast<long long>(b) * p.n + jn) : 0ull;
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kabs = k0 + kw0 + nt * 8 + t4 * 2 + e;
            const bool ok = rv && kabs < k0 + nk && key_visible(kabs, Lb, jn, p.anc, am);
            const float v = ok ? sacc[nt][hr * 2 + e] * p.scale_log2 : -INFINITY;
            sacc[nt][hr * 2 + e] = v;
            mx = fmaxf(mx, v);
          }
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        float sum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float v = sacc[nt][hr * 2 + e];
            const float pe = mx == -INFINITY ? 0.f : exp2f(v - mx);
            sacc[nt][hr * 2 + e] = pe;
            sum += pe;
          }
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        mrow[hr] = mx;
        lrow[hr] = sum;
      }
      // ---- O = P V, with P = P_hi + P_lo (bf16 pair)
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const uint32_t a0 = pack_bf16x2(sacc[2 * k2][0], sacc[2 * k2][1]);
        const uint32_t a1 = pack_bf16x2(sacc[2 * k2][2], sacc[2 * k2][3]);
        const uint32_t a2 = pack_bf16x2(sacc[2 * k2 + 1][0], sacc[2 * k2 + 1][1]);
        const uint32_t a3 = pack_bf16x2(sacc[2 * k2 + 1][2], sacc[2 * k2 + 1][3]);
        const uint32_t l0 = pack_bf16x2(sacc[2 * k2][0] - bf16lo(a0), sacc[2 * k2][1] - bf16hi(a0));
        const uint32_t l1 = pack_bf16x2(sacc[2 * k2][2] - bf16lo(a1), sacc[2 * k2][3] - bf16hi(a1));
        const uint32_t l2 =
            pack_bf16x2(sacc[2 * k2 + 1][0] - bf16lo(a2), sacc[2 * k2 + 1][1] - bf16hi(a2));
        const uint32_t l3 =
            pack_bf16x2(sacc[2 * k2 + 1][2] - bf16lo(a3), sacc[2 * k2 + 1][3] - bf16hi(a3));
        const int key = kw0 + k2 * 16 + (lane & 15);
#pragma unroll
        for (int dn = 0; dn < HD / 16; ++dn) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sV + swz<HD>(key, dn * 2 + (lane >> 4)), b0, b1, b2, b3);
          mma_bf16(oacc[2 * dn], a0, a1, a2, a3, b0, b1);
          mma_bf16(oacc[2 * dn + 1], a0, a1, a2, a3, b2, b3);
          mma_bf16(oacc[2 * dn], l0, l1, l2, l3, b0, b1);
          mma_bf16(oacc[2 * dn + 1], l0, l1, l2, l3, b2, b3);
        }
      }
    }
    // ---- this warp's partial to shared memory
    if (t4 == 0) {
      Mw[warp * 16 + g8] = mrow[0];
      Mw[warp * 16 + g8 + 8] = mrow[1];
      Lw[warp * 16 + g8] = lrow[0];
      Lw[warp * 16 + g8 + 8] = lrow[1];
    }
#pragma unroll
    for (int nd = 0; nd < HD / 8; ++nd) {
      float* o0 = Ow + (warp * 16 + g8) * L::kOStride + nd * 8 + t4 * 2;
      float* o1 = o0 + 8 * L::kOStride;
      *reinterpret_cast<float2*>(o0) = make_float2(oacc[nd][0], oacc[nd][1]);
      *reinterpret_cast<float2*>(o1) = make_float2(oacc[nd][2], oacc[nd][3]);
    }
    __syncthreads();
    // ---- merge the four warps: thread -> (row tid/8, dims (tid%8)*HD/8 ..)
    {
      const int i = tid >> 3;
      const int r = qt * 16 + i;
      constexpr int kDims = HD / 8;
      const int d0 = (tid & 7) * kDims;
      float m = -INFINITY;
#pragma unroll
      for (int w = 0; w < 4; ++w) m = fmaxf(m, Mw[w * 16 + i]);
      float wgt[4], l = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        wgt[w] = Mw[w * 16 + i] == -INFINITY ? 0.f : exp2f(Mw[w * 16 + i] - m);
        l += wgt[w] * Lw[w * 16 + i];
      }
      if (r < R) {
#pragma unroll
        for (int dd = 0; dd < kDims; dd += 4) {
          float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
          for (int w = 0; w < 4; ++w) {
            const float4 v =
                *reinterpret_cast<const float4*>(Ow + (w * 16 + i) * L::kOStride + d0 + dd);
            acc.x += wgt[w] * v.x;
            acc.y += wgt[w] * v.y;
            acc.z += wgt[w] * v.z;
            acc.w += wgt[w] * v.w;
          }
          __stcg(reinterpret_cast<float4*>(part_o + static_cast<long long>(r) * HD + d0 + dd), acc);
        }
        if ((tid & 7) == 0) {
          __stcg(part_ml + r * 2, m);
          __stcg(part_ml + r * 2 + 1, l);
        }
      }
    }
    __syncthreads();
  }

  // ---- last chunk to finish merges all chunks of this (sequence, KV head)
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    int32_t* ctr = p.counters + b * p.Hkv + kvh;
    const int old = atomicAdd(ctr, 1);
    const int last = old == ns - 1;
    if (last) *ctr = 0;
    *flag = last;
  }
  __syncthreads();
  if (!*flag) return;
  __threadfence();
  const float* base_o = p.part_o + (static_cast<long long>(b) * p.Hkv + kvh) * p.splits * R * HD;
  const float* base_ml = p.part_ml + (static_cast<long long>(b) * p.Hkv + kvh) * p.splits * R * 2;
  // every chunk's (max, sum) of a 16-row tile is staged in shared memory in
  // one parallel round (the key/value area is free by now), then one thread
  // per row turns them into chunk weights 2^(m_c - m) and 1/l, and every
  // output element sums its chunks with independent loads in flight
  float* ms = reinterpret_cast<float*>(smem + L::kK);   // [ns][16]
  float* ls = ms + 16 * kMaxChunks;                      // [ns][16]
  float* wgt = ms;
  float* rinv = Ow;                                      // [16]
  for (int r0 = 0; r0 < R; r0 += 16) {
    const int rows = min(16, R - r0);
    for (int idx = tid; idx < ns * 16; idx += kThreads) {
      const int c = idx >> 4, i = idx & 15;
      float m = -INFINITY, l = 0.f;
      if (i < rows) {
        const float2 v = __ldcg(reinterpret_cast<const float2*>(
            base_ml + (static_cast<long long>(c) * R + r0 + i) * 2));
        m = v.x;
        l = v.y;
      }
      ms[idx] = m;
      ls[idx] = l;
    }
    __syncthreads();
    if (tid < rows) {
      float m = -INFINITY;
      for (int c = 0; c < ns; ++c) m = fmaxf(m, ms[c * 16 + tid]);
      float l = 0.f;
      for (int c = 0; c < ns; ++c) {
        const float mc = ms[c * 16 + tid];
        const float w = mc == -INFINITY ? 0.f : exp2f(mc - m);
        l += w * ls[c * 16 + tid];
        wgt[c * 16 + tid] = w;
      }
      rinv[tid] = 1.0f / l;
    }
    __syncthreads();
    for (int idx = tid; idx < rows * (HD / 4); idx += kThreads) {
      const int i = idx / (HD / 4), d4 = (idx % (HD / 4)) * 4;
      const int r = r0 + i;
      float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
      int c = 0;
      for (; c + 4 <= ns; c += 4) {
        float4 v[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
          v[k] = __ldcg(reinterpret_cast<const float4*>(
              base_o + (static_cast<long long>(c + k) * R + r) * HD + d4));
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const float w = wgt[(c + k) * 16 + i];
          acc.x += w * v[k].x;
          acc.y += w * v[k].y;
          acc.z += w * v[k].z;
          acc.w += w * v[k].w;
        }
      }
      for (; c < ns; ++c) {
        const float4 v = __ldcg(
            reinterpret_cast<const float4*>(base_o + (static_cast<long long>(c) * R + r) * HD + d4));
        const float w = wgt[c * 16 + i];
        acc.x += w * v.x;
        acc.y += w * v.y;
        acc.z += w * v.z;
        acc.w += w * v.w;
      }
      const float inv = rinv[i];
      const int j = r / G, g = r % G;
      const long long off = (static_cast<long long>(b) * p.n + j) * qdim + (kvh * G + g) * HD + d4;
      const float o0 = acc.x * inv, o1 = acc.y * inv, o2 = acc.z * inv, o3 = acc.w * inv;
      uint2 pk;
      pk.x = pack_bf16x2(o0, o1);
      pk.y = pack_bf16x2(o2, o3);
      *reinterpret_cast<uint2*>(p.o + off) = pk;
      if (p.o_lo) {
        uint2 lo;
        lo.x = pack_bf16x2(o0 - bf16lo(pk.x), o1 - bf16hi(pk.x));
        lo.y = pack_bf16x2(o2 - bf16lo(pk.y), o3 - bf16hi(pk.y));
        *reinterpret_cast<uint2*>(p.o_lo + off) = lo;
      }
    }
    __syncthreads();
  }
}

// ---------------------------------------------------------------------------
// Decode path (n*G <= 32 query rows per KV head): one thread-block cluster of
// CS CTAs per (sequence, KV head).  CTA rank r takes a contiguous slice of the
// keys, its 8 warps (2 query tiles x 4 key groups) run an online-softmax loop
// over 32-key blocks, the four key groups of a tile are merged in shared
// memory, and after a cluster barrier each rank merges a share of the rows
// from all ranks' partials through distributed shared memory.  No global
// partials, no counters, no waits other than the hardware cluster barrier.
constexpr int kClusterThreads = 256;

SPEC_DEVINL uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
SPEC_DEVINL void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                   : "memory");
}
SPEC_DEVINL uint32_t map_rank(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
// Plain (non-volatile) distributed-shared-memory load: only issued after a
// cluster barrier, so the compiler may overlap as many as it likes.
SPEC_DEVINL float ld_cluster(uint32_t addr) {
  float v;
  asm("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
  return v;
}

template <int HD>
struct ClusterSmem {
  static constexpr int kRowB = HD * 2;
  // [kpr][HD] K, [kpr][HD] V, Q hi/lo [32][HD], O [32][HD] f32, m/l [32]
  __host__ __device__ static size_t kv_bytes(int kpr) { return static_cast<size_t>(kpr) * kRowB; }
  __host__ __device__ static size_t bytes(int kpr) {
    return 2 * kv_bytes(kpr) + 2 * 32 * kRowB + 32 * HD * 4 + 2 * 32 * 4 + 16;
  }
};

template <int HD>
__global__ void __launch_bounds__(kClusterThreads)
    attn_cluster_kernel(const AttnParams p, int kpr_max) {
  using L = ClusterSmem<HD>;
  extern __shared__ __align__(128) uint8_t smem[];
  const int kvh = blockIdx.y, b = blockIdx.z;
  const uint32_t rank = cluster_rank();
  const int CS = gridDim.x;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.H / p.Hkv;
  const int R = p.R;  // <= 32
  grid_dep_wait();
  grid_dep_launch();

  const int Lb = p.pos_base[b];
  const int Tk = min(Lb + p.n, p.cap);
  const int per = (Tk + CS - 1) / CS;
  const int k_lo = min(Tk, static_cast<int>(rank) * per);
  const int nk = min(Tk, k_lo + per) - k_lo;  // keys of this rank (may be 0)

  uint8_t* sKp = smem;
  uint8_t* sVp = smem + L::kv_bytes(kpr_max);
  uint8_t* sQp = sVp + L::kv_bytes(kpr_max);
  uint8_t* sQlp = sQp + 32 * L::kRowB;
  float* Oc = reinterpret_cast<float*>(sQlp + 32 * L::kRowB);  // [32][HD]
  float* Mc = Oc + 32 * HD;
  float* Lc = Mc + 32;
  const uint32_t sK = smem_u32(sKp), sV = smem_u32(sVp), sQ = smem_u32(sQp), sQlo = smem_u32(sQlp);
  const bool lo = p.q_lo != nullptr;

  // ---- stage this rank's keys/values and the query rows (hi, lo)
  const KVMap map{p.kv_table, p.kv_max_pages, p.kv_n_pages, p.Hkv, p.cap, HD};
  constexpr int kCPR = HD / 8;
  const int nk_pad = (nk + 31) & ~31;
  for (int idx = tid; idx < nk_pad * kCPR; idx += kClusterThreads) {
    const int i = idx / kCPR, c = idx % kCPR;
    const int row = i < nk ? i : 0;
    const long long g = map.row(b, kvh, k_lo + row) + c * 8;
    const int bytes = i < nk ? 16 : 0;
    cp_async16(sK + swz<HD>(i, c), p.kcache + g, bytes);
    cp_async16(sV + swz<HD>(i, c), p.vcache + g, bytes);
  }
  const int qdim = p.H * HD;
  for (int idx = tid; idx < 32 * kCPR; idx += kClusterThreads) {
    const int r = idx / kCPR, c = idx % kCPR;
    uint4 val = make_uint4(0, 0, 0, 0), vlo = make_uint4(0, 0, 0, 0);
    if (r < R) {
      const int j = r / G, g = r % G;
      const long long off = (static_cast<long long>(b) * p.n + j) * qdim + (kvh * G + g) * HD + c * 8;
      val = *reinterpret_cast<const uint4*>(p.q + off);
      if (lo) vlo = *reinterpret_cast<const uint4*>(p.q_lo + off);
    }
    *reinterpret_cast<uint4*>(sQp + swz<HD>(r, c)) = val;
    *reinterpret_cast<uint4*>(sQlp + swz<HD>(r, c)) = vlo;
  }
  cp_async_wait_all();
  __syncthreads();

  // ---- warp (qt, kg): query tile qt (rows qt*16..), key blocks kg, kg+4, ...
  const int qt = warp >> 2, kg = warp & 3;
  const int g8 = lane >> 2, t4 = lane & 3;
  float mrow[2] = {-INFINITY, -INFINITY}, lrow[2] = {0.f, 0.f};
  float oacc[HD / 8][4];
#pragma unroll
  for (int i = 0; i < HD / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
  const bool tile_live = qt * 16 < R;
  const int nblk = nk_pad / 32;
  if (tile_live) {
    for (int kb = kg; kb < nblk; kb += 4) {
      const int kw0 = kb * 32;
      float sacc[4][4];
#pragma unroll
      for (int i = 0; i < 4; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < HD / 16; ++kk) {
        uint32_t a0, a1, a2, a3, l0, l1, l2, l3;
        const int qrow = qt * 16 + (lane & 15);
        ldsm_x4(sQ + swz<HD>(qrow, kk * 2 + (lane >> 4)), a0, a1, a2, a3);
        if (lo) ldsm_x4(sQlo + swz<HD>(qrow, kk * 2 + (lane >> 4)), l0, l1, l2, l3);
#pragma unroll
        for (int np = 0; np < 2; ++np) {
          const int key = kw0 + np * 16 + (lane & 7) + ((lane >> 4) << 3);
          uint32_t b0, b1, b2, b3;
          ldsm_x4(sK + swz<HD>(key, kk * 2 + ((lane >> 3) & 1)), b0, b1, b2, b3);
          mma_bf16(sacc[np * 2], a0, a1, a2, a3, b0, b1);
          mma_bf16(sacc[np * 2 + 1], a0, a1, a2, a3, b2, b3);
          if (lo) {
            mma_bf16(sacc[np * 2], l0, l1, l2, l3, b0, b1);
            mma_bf16(sacc[np * 2 + 1], l0, l1, l2, l3, b2, b3);
          }
        }
      }
      // mask + online softmax (exp2 domain)
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int r = qt * 16 + g8 + hr * 8;
        const bool rv = r < R;
        const int jn = rv ? r / G : 0;
        const uint64_t am = (p.anc && rv) ? __ldg(p.anc + static_cast<long long>(b) * p.n + jn) : 0ull;
        float mx = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int kl = kw0 + nt * 8 + t4 * 2 + e;
            const int kabs = k_lo + kl;
            const bool ok = rv && kl < nk && key_visible(kabs, Lb, jn, p.anc, am);
            const float v = ok ? sacc[nt][hr * 2 + e] * p.scale_log2 : -INFINITY;
            sacc[nt][hr * 2 + e] = v;
            mx = fmaxf(mx, v);
          }
        }
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        const float mnew = fmaxf(mrow[hr], mx);
        const float scale = mnew == -INFINITY ? 1.f : exp2f(mrow[hr] - mnew);
        float sum = 0.f;
#pragma unroll
        for (int nt = 0; nt < 4; ++nt) {
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const float v = sacc[nt][hr * 2 + e];
            const float pe = mnew == -INFINITY ? 0.f : exp2f(v - mnew);
            sacc[nt][hr * 2 + e] = pe;
            sum += pe;
          }
        }
        sum += __shfl_xor_sync(0xffffffffu, sum, 1);
        sum += __shfl_xor_sync(0xffffffffu, sum, 2);
        lrow[hr] = lrow[hr] * scale + sum;
        mrow[hr] = mnew;
#pragma unroll
        for (int nd = 0; nd < HD / 8; ++nd) {
          oacc[nd][hr * 2] *= scale;
          oacc[nd][hr * 2 + 1] *= scale;
        }
      }
      // O += P V with P = P_hi + P_lo
#pragma unroll
      for (int k2 = 0; k2 < 2; ++k2) {
        const uint32_t a0 = pack_bf16x2(sacc[2 * k2][0], sacc[2 * k2][1]);
        const uint32_t a1 = pack_bf16x2(sacc[2 * k2][2], sacc[2 * k2][3]);
        const uint32_t a2 = pack_bf16x2(sacc[2 * k2 + 1][0], sacc[2 * k2 + 1][1]);
        const uint32_t a3 = pack_bf16x2(sacc[2 * k2 + 1][2], sacc[2 * k2 + 1][3]);
        const uint32_t l0 = pack_bf16x2(sacc[2 * k2][0] - bf16lo(a0), sacc[2 * k2][1] - bf16hi(a0));
        const uint32_t l1 = pack_bf16x2(sacc[2 * k2][2] - bf16lo(a1), sacc[2 * k2][3] - bf16hi(a1));
        const uint32_t l2 =
            pack_bf16x2(sacc[2 * k2 + 1][0] - bf16lo(a2), sacc[2 * k2 + 1][1] - bf16hi(a2));
        const uint32_t l3 =
            pack_bf16x2(sacc[2 * k2 + 1][2] - bf16lo(a3), sacc[2 * k2 + 1][3] - bf16hi(a3));
        const int key = kw0 + k2 * 16 + (lane & 15);
#pragma unroll
        for (int dn = 0; dn < HD / 16; ++dn) {
          uint32_t b0, b1, b2, b3;
          ldsm_x4_t(sV + swz<HD>(key, dn * 2 + (lane >> 4)), b0, b1, b2, b3);
          mma_bf16(oacc[2 * dn], a0, a1, a2, a3, b0, b1);
          mma_bf16(oacc[2 * dn + 1], a0, a1, a2, a3, b2, b3);
          mma_bf16(oacc[2 * dn], l0, l1, l2, l3, b0, b1);
          mma_bf16(oacc[2 * dn + 1], l0, l1, l2, l3, b2, b3);
        }
      }
    }
  }
  // ---- merge the four key groups of each query tile into the CTA partial
  for (int step = 0; step < 4; ++step) {
    if (kg == step && tile_live) {
#pragma unroll
      for (int hr = 0; hr < 2; ++hr) {
        const int rr = qt * 16 + g8 + hr * 8;
        const float mo = step ? Mc[rr] : -INFINITY;
        const float lo_ = step ? Lc[rr] : 0.f;
        const float mn = fmaxf(mo, mrow[hr]);
        const float so = mo == -INFINITY ? 0.f : exp2f(mo - mn);
        const float sn = mrow[hr] == -INFINITY ? 0.f : exp2f(mrow[hr] - mn);
#pragma unroll
        for (int nd = 0; nd < HD / 8; ++nd) {
          float* o = Oc + rr * HD + nd * 8 + t4 * 2;
          const float x0 = step ? o[0] : 0.f, x1 = step ? o[1] : 0.f;
          o[0] = x0 * so + oacc[nd][hr * 2] * sn;
          o[1] = x1 * so + oacc[nd][hr * 2 + 1] * sn;
        }
        __syncwarp();
        if (t4 == 0) {
          Mc[rr] = mn;
          Lc[rr] = lo_ * so + lrow[hr] * sn;
        }
      }
    }
    __syncthreads();
  }
  // ---- cluster merge: rank r owns rows r, r+CS, ...  (1) every rank's
  // (max, sum) of the owned rows in one parallel round, (2) chunk weights per
  // row, (3) one thread per (row, dim) with all ranks' loads in flight
  cluster_sync();
  const uint32_t oc_addr = smem_u32(Oc), mc_addr = smem_u32(Mc), lc_addr = smem_u32(Lc);
  const int own = (R - static_cast<int>(rank) + CS - 1) / CS;  // rows owned (<= 2 for CS 16)
  float* Wg = reinterpret_cast<float*>(sQp);                   // [CS][own] weights (Q area is free)
  float* Lg = Wg + 16 * 32;                                     // [CS][own] sums
  float* Rinv = Lg + 16 * 32;                                   // [own]
  for (int i = tid; i < CS * own; i += kClusterThreads) {
    const int c = i / own, lr = i % own;
    const int rr = static_cast<int>(rank) + lr * CS;
    Wg[c * 32 + lr] = ld_cluster(map_rank(mc_addr + rr * 4, c));
    Lg[c * 32 + lr] = ld_cluster(map_rank(lc_addr + rr * 4, c));
  }
  __syncthreads();
  if (tid < own) {
    float m = -INFINITY;
    for (int c = 0; c < CS; ++c) m = fmaxf(m, Wg[c * 32 + tid]);
    float l = 0.f;
    for (int c = 0; c < CS; ++c) {
      const float mc = Wg[c * 32 + tid];
      const float w = mc == -INFINITY ? 0.f : exp2f(mc - m);
      Wg[c * 32 + tid] = w;
      l += w * Lg[c * 32 + tid];
    }
    Rinv[tid] = 1.0f / l;
  }
  __syncthreads();
  for (int item = tid; item < own * HD; item += kClusterThreads) {
    const int lr = item / HD, dim = item % HD;
    const int rr = static_cast<int>(rank) + lr * CS;
    const uint32_t src = oc_addr + (rr * HD + dim) * 4;
    float v[16];
#pragma unroll
    for (int c = 0; c < 16; ++c) v[c] = c < CS ? ld_cluster(map_rank(src, c)) : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int c = 0; c < 16; ++c) acc += c < CS ? Wg[c * 32 + lr] * v[c] : 0.f;
    const float o = acc * Rinv[lr];
    const int j = rr / G, g = rr % G;
    const long long off = (static_cast<long long>(b) * p.n + j) * qdim + (kvh * G + g) * HD + dim;
    const uint16_t hi = f32_to_bf16(o);
    p.o[off] = hi;
    if (p.o_lo) p.o_lo[off] = f32_to_bf16(o - bf16_to_f32(hi));
  }
  cluster_sync();  // peers' shared memory stays alive until every rank has read it
}

// Dynamic shared memory up to the per-CTA maximum and clusters above the
// portable size, set once per device.
constexpr int kMaxDynSmem = 227 * 1024;

template <int HD>
cudaError_t configure_cluster(size_t smem) {
  if (smem > static_cast<size_t>(kMaxDynSmem)) return cudaErrorInvalidValue;
  static PerDevice<cudaError_t> done;
  cudaError_t e = cudaErrorInvalidDevice;
  if (!done.get(
          [] {
            cudaError_t r = cudaFuncSetAttribute(attn_cluster_kernel<HD>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                 kMaxDynSmem);
            if (r != cudaSuccess) return r;
            return cudaFuncSetAttribute(attn_cluster_kernel<HD>,
                                        cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
          },
          &e))
    return cudaErrorInvalidDevice;
  return e;
}

// Can clusters of `cs` CTAs with this much shared memory be placed at all?
template <int HD>
bool cluster_fits(int cs, size_t smem) {
  if (configure_cluster<HD>(smem) != cudaSuccess) return false;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cs, 1, 1);
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  return cudaOccupancyMaxActiveClusters(&n, attn_cluster_kernel<HD>, &cfg) == cudaSuccess && n > 0;
}

template <int HD>
cudaError_t launch_cluster(const AttnParams& p, cudaStream_t stream, bool pdl) {
  const int CS = p.cluster;
  const int kpr = ((p.cap + CS - 1) / CS + 31) & ~31;
  const size_t smem = ClusterSmem<HD>::bytes(kpr);
  cudaError_t e = configure_cluster<HD>(smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(CS, p.Hkv, p.B);
  cfg.blockDim = dim3(kClusterThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = CS;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, attn_cluster_kernel<HD>, p, kpr);
}

template <int HD>
cudaError_t launch_hd(const AttnParams& p, cudaStream_t stream, bool pdl) {
  static PerDevice<cudaError_t> configured;
  const size_t smem = AttnSmem<HD>::kBytes;
  cudaError_t ce = cudaErrorInvalidDevice;
  if (!configured.get([smem] { return cudaFuncSetAttribute(attn_splitkv_kernel<HD>,
                                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                           static_cast<int>(smem)); },
                      &ce) || ce != cudaSuccess)
    return ce;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.splits, p.Hkv, p.B);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, attn_splitkv_kernel<HD>, p);
}

}  // namespace

int attention_cluster_size(int hd, int cap, size_t smem_limit) {
  // the last answer per device, keyed by the arguments
  struct Entry {
    int hd = -1, cap = -1;
    size_t lim = 0;
    int val = 0;
  };
  static std::mutex mu;
  static Entry cache[kMaxDevices];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  {
    std::lock_guard<std::mutex> lock(mu);
    const Entry& c = cache[dev];
    if (c.hd == hd && c.cap == cap && c.lim == smem_limit) return c.val;
  }
  int best = 0;
  int cs = (cap + 127) / 128;
  cs = cs < 1 ? 1 : (cs > 16 ? 16 : cs);
  for (; cs >= 1 && !best; cs = cs > 8 ? 8 : cs - 1) {
    const int kpr = ((cap + cs - 1) / cs + 31) & ~31;
    const size_t smem = hd == 128 ? ClusterSmem<128>::bytes(kpr) : ClusterSmem<64>::bytes(kpr);
    if (smem > smem_limit) break;
    const bool ok = hd == 128 ? cluster_fits<128>(cs, smem) : cluster_fits<64>(cs, smem);
    if (ok) best = cs;
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[dev] = Entry{hd, cap, smem_limit, best};
  return best;
}

cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream, bool pdl) {
  if (p.cluster > 0) {
    if (p.hd == 128) return launch_cluster<128>(p, stream, pdl);
    if (p.hd == 64) return launch_cluster<64>(p, stream, pdl);
    return cudaErrorInvalidValue;
  }
  if (p.hd == 128) return launch_hd<128>(p, stream, pdl);
  if (p.hd == 64) return launch_hd<64>(p, stream, pdl);
  return cudaErrorInvalidValue;
}

}  // namespace spec
