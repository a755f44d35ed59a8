// Skinny weight-streaming GEMM for the verification pass on sm_103a.
//
// One target pass multiplies every weight matrix by only M = batch*(gamma+1)
// token rows, so the pass is a stream of the weights through HBM ("verifying
// several tokens costs the same as one": pigeon guide, *The idea*; lattice
// notes: the k-token pass turns the matrix-vector op into a matrix-matrix op
// over the same weight read).  The kernel is built around that stream:
//
//  * swap-AB: the weight tile (128 output features x 64 K) is the UMMA "A"
//    operand (M = 128), the M token rows padded to ntok (16..256) are "B";
//    the accumulator D[feature][token] lives in tensor memory.  Activations
//    arrive as a bf16 pair (x = hi + lo) so the GEMM sees ~16-bit-mantissa
//    inputs while the weights are still read once: for ntok <= 128 the lo rows
//    are stacked under the hi rows in one B operand (UMMA N = 2 ntok, summed in
//    the epilogue; an N=32 MMA issues as fast as an N=16 one), for wider tiles
//    a second MMA accumulates the lo rows.
//  * warp 0 streams weight tiles and activation tiles with TMA
//    (cp.async.bulk.tensor, 128-byte swizzle, evict-first L2 policy for the
//    weights) through a ring of shared-memory stages guarded by mbarriers;
//    weight loads for the first ring pass are issued before the
//    programmatic-dependent-launch wait, i.e. while the previous kernel
//    finishes.
//  * warp 1 allocates TMEM and one lane issues tcgen05.mma (kind::f16, bf16 x
//    bf16 -> fp32), committing each stage back to the producer and each
//    finished accumulator to the epilogue (double-buffered in TMEM).
//  * warps 2-5 drain TMEM with tcgen05.ld and run the fused epilogue.
//  * Stream-K: the n_tiles x (K/64) work units are split into equal
//    contiguous ranges, one per CTA (grid <= SM count), so every SM streams
//    the same number of bytes.  A tile split across CTAs is finished by the
//    last CTA to arrive (atomic counter), which sums every contributor's
//    fp32 partial in CTA order: deterministic, no float atomics, no waits on
//    other CTAs.  With one CTA per SM (wide token tiles), the contributors
//    that have no later segment share the finishing instead: each waits
//    (bounded) until every contributor has arrived, then sums and runs the
//    epilogue of every n-th 16-column chunk.  After its last MMA a finisher
//    otherwise spends a few microseconds a chunk on the epilogue's per-column
//    chains, ten chunks at 160 token rows, while the other CTAs have exited.
//
// Epilogues: EPI_STORE (fp32 logits), EPI_RESID (residual add + next norm's
// bf16 input + sum-of-squares partials), EPI_QKV (RMSNorm scale, RoPE, q to
// the workspace, k/v appended to the bf16 cache), EPI_SWIGLU.
#include "common.cuh"
#include "gemm_common.cuh"
#include "internal.h"

namespace spec {

namespace {

constexpr int kThreads = 192;

}  // namespace

__global__ void __launch_bounds__(kThreads, 2)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmX,
                   const __grid_constant__ CUtensorMap tmXlo, const GemmParams p, int shared_finish) {
  extern __shared__ uint8_t smem_raw[];
  const int nb = p.split ? 2 * p.ntok : p.ntok;  // B rows per sub-tile: hi rows, then lo rows
  const int ncols = p.split == 1 ? 2 * p.ntok : p.ntok;  // accumulator columns (UMMA N)
  const int ksub = p.ksub;
  const Smem sm = carve(smem_raw, nb, p.stages, ksub);
  const int warp = threadIdx.x >> 5;
  const int S = p.stages;
  const Partition part{static_cast<uint32_t>(p.units), gridDim.x, static_cast<uint32_t>(p.kc)};
  const uint32_t me = blockIdx.x;
  const uint32_t u0 = part.start(me), u1 = part.start(me + 1);
  const uint32_t kc = static_cast<uint32_t>(p.kc);
  const uint32_t tcols = tmem_cols_for(ncols);
  const uint32_t sbytes = static_cast<uint32_t>(stage_bytes(nb, ksub));
  const uint32_t boff = static_cast<uint32_t>(kATileBytes) * ksub;  // B sub-tiles after the A ones
  const uint32_t bsub = static_cast<uint32_t>(nb) * 128;            // bytes of one B sub-tile

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&sm.full[s], 1);
      mbar_init(&sm.empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&sm.accfull[a], 1);
      mbar_init(&sm.accempty[a], 4);
    }
    *sm.abort = 0;
    fence_mbar_init();
    prefetch_tmap(&tmW);
    prefetch_tmap(&tmX);
    if (p.split) prefetch_tmap(&tmXlo);
  }
  if (warp == 1) {
    tmem_alloc(sm.tmem_slot, tcols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *sm.tmem_slot;
  grid_dep_launch();

  if (warp == 0) {
    if (elect_lane0() && u1 > u0) {
      // ------------------------------------------------------ TMA producer
      const uint64_t pol_w = l2_policy_evict_first();
      const uint64_t pol_x = l2_policy_evict_last();
      uint32_t issued[kMaxStages];
      for (int s = 0; s < S; ++s) issued[s] = 0;
      const uint32_t n = u1 - u0;
      const int pre = static_cast<int>(n < static_cast<uint32_t>(S) ? n : static_cast<uint32_t>(S));
      // (tile, k-chunk) of the next unit, advanced without divisions
      uint32_t tile = u0 / kc, kci = u0 - tile * kc;
      uint32_t kci_b = kci;
      auto load_a = [&](uint8_t* st, uint64_t* bar) {
        for (int s = 0; s < ksub; ++s)
          tma_load_2d(st + s * kATileBytes, &tmW, bar, static_cast<int>((kci * ksub + s) * kTileK),
                      static_cast<int>(tile * kTileN), pol_w);
      };
      auto load_b = [&](uint8_t* st, uint64_t* bar, uint32_t k) {
        for (int s = 0; s < ksub; ++s) {
          uint8_t* b = st + boff + s * bsub;
          const int x = static_cast<int>((k * ksub + s) * kTileK);
          tma_load_2d(b, &tmX, bar, x, p.tok0, pol_x);
          if (p.split) tma_load_2d(b + p.ntok * 128, &tmXlo, bar, x, p.tok0, pol_x);
        }
      };
      for (int i = 0; i < pre; ++i) {
        uint8_t* st = sm.stage_base + static_cast<size_t>(i) * sbytes;
        mbar_arrive_expect_tx(&sm.full[i], sbytes);
        load_a(st, &sm.full[i]);
        if (++kci == kc) {
          kci = 0;
          ++tile;
        }
      }
      grid_dep_wait();  // activations are produced by the previous kernel
      for (int i = 0; i < pre; ++i) {
        load_b(sm.stage_base + static_cast<size_t>(i) * sbytes, &sm.full[i], kci_b);
        issued[i] = 1;
        if (++kci_b == kc) kci_b = 0;
      }
      int stage = pre % S;
      uint32_t phase = pre == S ? 1u : 0u;
      for (uint32_t u = u0 + pre; u < u1; ++u) {
        if (!mbar_wait(&sm.empty[stage], phase ^ 1u, sm.abort)) break;
        uint8_t* st = sm.stage_base + static_cast<size_t>(stage) * sbytes;
        mbar_arrive_expect_tx(&sm.full[stage], sbytes);
        load_a(st, &sm.full[stage]);
        load_b(st, &sm.full[stage], kci);
        ++issued[stage];
        if (++kci == kc) {
          kci = 0;
          ++tile;
        }
        if (++stage == S) {
          stage = 0;
          phase ^= 1u;
        }
      }
      if (*sm.abort) {
        // let every copy still in flight land before the CTA may exit
        volatile int never = 0;
        for (int s = 0; s < S; ++s)
          if (issued[s]) mbar_wait(&sm.full[s], (issued[s] - 1) & 1u, &never);
      }
    } else {
      grid_dep_wait();
    }
  } else if (warp == 1) {
    grid_dep_wait();
    if (elect_lane0() && u1 > u0) {
      // -------------------------------------------------------- MMA issuer
      const uint32_t idesc = idesc_bf16(kTileN, ncols);
      int stage = 0;
      uint32_t phase = 0;
      int seg = 0;
      uint32_t u = u0;
      bool ok = true;
      while (u < u1 && ok) {
        const uint32_t t = part.tile_of(u);
        const uint32_t seg_end = min(u1, (t + 1) * kc);
        const int a = seg & 1;
        ok = mbar_wait(&sm.accempty[a], ((seg >> 1) & 1) ^ 1u, sm.abort);
        if (!ok) break;
        tc_fence_after();
        const uint32_t dcol = tmem_base + static_cast<uint32_t>(a * ncols);
        for (uint32_t v = u; v < seg_end; ++v) {
          if (!mbar_wait(&sm.full[stage], phase, sm.abort)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t sbase = smem_u32(sm.stage_base + static_cast<size_t>(stage) * sbytes);
          for (int s = 0; s < ksub; ++s) {
            const uint32_t abase = sbase + s * kATileBytes;
            const uint32_t bbase = sbase + boff + s * bsub;
            const uint32_t lbase = bbase + static_cast<uint32_t>(p.ntok) * 128;
#pragma unroll
            for (int kk = 0; kk < kTileK / 16; ++kk) {
              const uint64_t ad = sdesc_k128(abase + kk * 32);
              umma_bf16(dcol, ad, sdesc_k128(bbase + kk * 32), idesc,
                        (v > u || s > 0 || kk > 0) ? 1u : 0u);
              // split == 2: the bf16 residual of the activations into the same
              // accumulator (split == 1 has it stacked in the same MMA's N)
              if (p.split == 2) umma_bf16(dcol, ad, sdesc_k128(lbase + kk * 32), idesc, 1u);
            }
          }
          umma_commit(&sm.empty[stage]);
          if (++stage == S) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        umma_commit(&sm.accfull[a]);
        u = seg_end;
        ++seg;
      }
    }
  } else {
    // --------------------------------------------------------------- epilogue
    grid_dep_wait();
    const int e = threadIdx.x - kEpiFirstThread;
    const int quarter = warp & 3;
    const int r = quarter * 32 + (threadIdx.x & 31);
    if (p.ssq_in) {
      for (int c = e; c < p.ntok; c += kEpiThreads) {
        const int m = p.tok0 + c;
        float s = 0.f;
        if (m < p.M)
          for (int t = 0; t < p.ssq_tiles; ++t) s += p.ssq_in[static_cast<long long>(t) * p.ssq_ld + m];
        sm.rs[c] = rsqrtf(s * p.inv_d + p.eps);
      }
    }
    named_bar(kEpiBar, kEpiThreads);
    const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
    int seg = 0;
    uint32_t u = u0;
    while (u < u1) {
      const uint32_t t = part.tile_of(u);
      const uint32_t seg_end = min(u1, (t + 1) * kc);
      const int a = seg & 1;
      mbar_wait(&sm.accfull[a], (seg >> 1) & 1, sm.abort);
      named_bar(kEpiBar, kEpiThreads);  // all four warps leave together on abort
      if (*sm.abort) break;
      tc_fence_after();
      const uint32_t tacc = tmem_base + lane_addr + static_cast<uint32_t>(a * ncols);
      const uint32_t c_first = part.cta_of(t * kc);
      const uint32_t c_last = part.cta_of((t + 1) * kc - 1);
      const int nc = static_cast<int>(c_last - c_first + 1);
      bool finisher = true;
      int chunk0 = 0, chunk_step = 1;  // this CTA's 16-column chunks: chunk0, chunk0 + chunk_step, ...
      // shared finishing: the contributors with no later segment, a prefix
      // of the tile's CTAs (the last one may go on into the next tile)
      const bool sharing = shared_finish && nc > 1;
      const int n_fin = part.start(c_last + 1) > (t + 1) * kc ? nc - 1 : nc;
      if (nc > 1) {
        const int slot = part.slot(me, t);
        float* dst = p.partials + (static_cast<long long>(me) * 2 + slot) * p.ntok * kTileN;
        for (int c0 = 0; c0 < p.ntok; c0 += 16) {
          float v[16];
          load_acc(tacc, c0, p.ntok, p.split, v);
#pragma unroll
          for (int j = 0; j < 16; ++j) __stcg(dst + (c0 + j) * kTileN + r, v[j]);
        }
        if (e < nc) sm.slots[e] = part.slot(c_first + e, t);  // for the finisher
        __threadfence();
        named_bar(kEpiBar, kEpiThreads);
        if (e == 0) {
          const int old = atomicAdd(&p.counters[t], 1);
          if (!sharing) {
            const int last = old == nc - 1;
            if (last) p.counters[t] = 0;
            *sm.flag = last;
          } else if (seg_end == u1) {
            // every contributor's partials are stored once the count is nc
            *sm.flag = wait_count(reinterpret_cast<const unsigned*>(p.counters + t), static_cast<unsigned>(nc),
                                  sm.abort, p.status)
                           ? 1
                           : 0;
          } else {
            *sm.flag = 0;  // a later segment follows: the others finish this tile
          }
        }
        named_bar(kEpiBar, kEpiThreads);
        finisher = *sm.flag != 0;
        __threadfence();
        if (sharing) {
          chunk0 = static_cast<int>(me - c_first);
          chunk_step = n_fin;
        }
      }
      if (finisher) {
        // per 16-column chunk: the residual rows (EPI_RESID) and up to four
        // contributors' partial sums in flight together, one L2 round trip
        // for most tiles (a tile has about five contributors at 152 CTAs
        // over 32 tiles)
        const bool pre_h = p.epi == EPI_RESID;
        const int f = static_cast<int>(t) * kTileN + r;
        for (int c0 = chunk0 * 16; c0 < p.ntok; c0 += chunk_step * 16) {
          float own[16], acc[16], hv[16];
          if (pre_h) {
#pragma unroll
            for (int j = 0; j < 16; ++j) {
              const int m = p.tok0 + c0 + j;
              hv[j] = (m < p.M && f < p.N) ? ldcg(p.h + static_cast<long long>(m) * p.d + f) : 0.f;
            }
          }
          load_acc(tacc, c0, p.ntok, p.split, own);
          if (nc == 1) {
#pragma unroll
            for (int j = 0; j < 16; ++j) acc[j] = own[j];
          } else {
            fixup_sum<4>(p.partials, p.ntok, c0, r, c_first, nc, me, sm.slots, own, acc);
          }
          epilogue_chunk_h(p, sm, t, r, c0, acc, hv, pre_h, EpiPre{});
        }
        if (sharing) {
          // the sharers' second arrivals: the last one clears the tile's
          // counter for the next launch (every sharer has seen nc by then)
          named_bar(kEpiBar, kEpiThreads);
          if (e == 0) {
            const int old = atomicAdd(&p.counters[t], 1);
            if (old == nc + n_fin - 1) p.counters[t] = 0;
          }
        }
      }
      tc_fence_before();
      __syncwarp();
      if ((threadIdx.x & 31) == 0) mbar_arrive(&sm.accempty[a]);
      u = seg_end;
      ++seg;
    }
  }

  if (*sm.abort && threadIdx.x == 0) set_status(p.status, SPEC_DEV_TIMEOUT);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tcols);
  }
}

size_t gemm_smem_bytes(int rows_b, int stages, int ksub) {
  return 1024 + stage_bytes(rows_b, ksub) * stages + kTailBytes;
}

int gemm_max_stages(int rows_b, size_t budget, int ksub) {
  int s = static_cast<int>((budget - 1024 - kTailBytes) / stage_bytes(rows_b, ksub));
  if (s > kMaxStages) s = kMaxStages;
  return s;
}

cudaError_t launch_gemm(const CUtensorMap* tmW, const CUtensorMap* tmX, const CUtensorMap* tmXlo,
                        const GemmParams& p, int grid, cudaStream_t stream, bool pdl) {
  const size_t smem = gemm_smem_bytes(p.split ? 2 * p.ntok : p.ntok, p.stages, p.ksub);
  // Shared finishing makes CTAs wait for one another: only where every CTA of
  // the grid is resident at once, one per SM (no two fit in an SM's 228 KB of
  // shared memory) and no more CTAs than SMs.
  static PerDevice<int> sms;
  int n_sm = 0;
  if (!sms.get([] {
        int dev = 0, v = 0;
        if (cudaGetDevice(&dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
          return 0;
        return v;
      },
      &n_sm))
    n_sm = 0;
  int shared_finish = (smem > 116 * 1024 && n_sm > 0 && grid <= n_sm) ? 1 : 0;
  static PerDevice<cudaError_t> configured;
  cudaError_t ce = cudaErrorInvalidDevice;
  if (!configured.get([] { return cudaFuncSetAttribute(gemm_tc_kernel,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       227 * 1024); },
                      &ce) || ce != cudaSuccess)
    return ce;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, gemm_tc_kernel, *tmW, *tmX, *tmXlo, p, shared_finish);
}

}  // namespace spec
