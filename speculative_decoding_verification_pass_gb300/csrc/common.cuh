// Device helpers shared by the sm_103a kernels: PTX wrappers for mbarriers,
// TMA, tcgen05 (UMMA + TMEM), programmatic dependent launch, bounded waits,
// the device status word and bf16 conversions.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

#define SPEC_DEVINL __device__ __forceinline__

namespace spec {

// ------------------------------------------------------------------ status
// The workspace begins with one int32 status word (SPEC_DEV_* bits).
SPEC_DEVINL void set_status(int32_t* status, int32_t bit) {
  if (status) atomicOr(status, bit);
}

// Load with acquire semantics at GPU scope (grid-barrier counters).
// 64-bit relaxed accesses at GPU scope: single-copy atomic, so a word that
// carries a value and a tag is seen whole or not at all.
SPEC_DEVINL void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}
SPEC_DEVINL unsigned long long ld_relaxed_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p));
  return v;
}

// *p += v at GPU scope with release semantics: writes this thread has made
// or observed (through a CTA barrier) are visible before the addition is.
SPEC_DEVINL void red_release_add(unsigned* p, unsigned v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

SPEC_DEVINL uint32_t ld_acquire(const unsigned* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// May the query of new-block node j see key slot kabs?  The block starts at
// slot Lb: cached keys always; a new slot Lb + s by the causal order (s <= j)
// for a chain, or, with a draft tree (anc != nullptr), iff bit s of the
// node's ancestor mask `am` is set (the node itself or one of its ancestors).
// Where (sequence b, KV head h, slot t)'s key / value row starts within one
// layer's cache, in elements: contiguous [B][Hkv][cap][hd], or paged through a
// block table (page = table[b][t / kPageSlots], rows [page][Hkv][kPageSlots][hd];
// a page id outside [0, n_pages) is clamped, the pass flags it beforehand).
constexpr int kPageSlots = SPEC_PAGE_SLOTS;

// The pass's slot check: len + n within the capacity and, for a paged cache,
// every page covering slots [0, len + n) a valid page id.  0 when it fits,
// else the status bit to raise.
SPEC_DEVINL int32_t seq_fit(int L, int n, int cap, const int32_t* table, int max_pages, int n_pages,
                            int b) {
  if (L < 0 || L + n > cap) return SPEC_DEV_KV_OVERFLOW;
  if (table) {
    const int np = (L + n + kPageSlots - 1) / kPageSlots;
    for (int j = 0; j < np; ++j) {
      const int pg = __ldg(table + static_cast<long long>(b) * max_pages + j);
      if (pg < 0 || pg >= n_pages) return SPEC_DEV_BAD_PAGE;
    }
  }
  return 0;
}
struct KVMap {
  const int32_t* table;  // [B][max_pages] physical page ids, or nullptr (contiguous)
  int max_pages, n_pages;
  int Hkv, cap, hd;
  // kLayout: 0 decided by `table` at run time, 1 contiguous, 2 paged
  template <int kLayout = 0>
  SPEC_DEVINL long long row(int b, int h, int t) const {
    if (kLayout == 1 || (kLayout == 0 && !table))
      return ((static_cast<long long>(b) * Hkv + h) * cap + t) * hd;
    int page = __ldg(table + static_cast<long long>(b) * max_pages + t / kPageSlots);
    page = page < 0 ? 0 : (page >= n_pages ? n_pages - 1 : page);
    return ((static_cast<long long>(page) * Hkv + h) * kPageSlots + (t % kPageSlots)) * hd;
  }
};

SPEC_DEVINL bool key_visible(int kabs, int Lb, int j, const uint64_t* anc, uint64_t am) {
  if (kabs < Lb) return true;
  const int s = kabs - Lb;
  return anc ? (s < 64 && ((am >> s) & 1ull) != 0) : s <= j;
}

// Wall-clock bound for every spin-wait in a kernel: about two seconds.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

SPEC_DEVINL unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Wait (one thread) until *ctr >= target, reading it with acquire semantics.
// Bounded: after limit_ns of wall-clock time it sets *abort and the timeout
// bit of *status and returns false; it also returns false once *abort is set
// by another thread.  The persistent forward's grid barrier waits through it.
SPEC_DEVINL bool wait_count(const unsigned* ctr, unsigned target, volatile int* abort,
                            int32_t* status, unsigned long long limit_ns = kWaitLimitNs) {
  if (ld_acquire(ctr) >= target) return true;
  const unsigned long long t0 = globaltimer();
  for (;;) {
    if (ld_acquire(ctr) >= target) return true;
    if (*abort) return false;
    if (globaltimer() - t0 > limit_ns) {
      *abort = 1;
      set_status(status, SPEC_DEV_TIMEOUT);
      return false;
    }
    __nanosleep(32);
  }
}

// ------------------------------------------------------- dependent launches
// Wait until the previous kernel in the stream has completed and its writes
// are visible (no-op when the launch had no programmatic dependency).
SPEC_DEVINL void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Allow the next kernel in the stream to start its prologue.
SPEC_DEVINL void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- smem/mbar
SPEC_DEVINL uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

SPEC_DEVINL void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count)
               : "memory");
}
SPEC_DEVINL void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
SPEC_DEVINL void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}
SPEC_DEVINL void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
SPEC_DEVINL bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase with the given parity.  Returns false (and the
// caller must abandon its loop) once `*abort` is set or the wall-clock limit
// is reached; the first waiter to time out sets *abort.
SPEC_DEVINL bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  for (uint32_t it = 0;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 63u) == 63u) {
      if (*abort) return false;
      if (globaltimer() - t0 > kWaitLimitNs) {
        *abort = 1;
        return false;
      }
    }
  }
}

// --------------------------------------------------------------------- TMA
SPEC_DEVINL void prefetch_tmap(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
SPEC_DEVINL uint64_t l2_policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
SPEC_DEVINL uint64_t l2_policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
// 2-D tiled load (x = innermost coordinate in elements, y = row) into shared
// memory, completing `bar`'s transaction count.
SPEC_DEVINL void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y,
                             uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}

// The same with a shared-memory address, and a 3-D box.
SPEC_DEVINL void tma_load_2d_s(uint32_t dst, const CUtensorMap* m, uint64_t* bar, int x, int y, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy)
      : "memory");
}
SPEC_DEVINL void tma_load_3d_s(uint32_t dst, const CUtensorMap* m, uint64_t* bar, int x, int y, int z,
                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4, %5}], [%2], %6;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "l"(policy)
      : "memory");
}

// ----------------------------------------------------------------- tcgen05
SPEC_DEVINL void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                   smem_u32(slot)),
               "r"(ncols)
               : "memory");
}
SPEC_DEVINL void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
SPEC_DEVINL void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
SPEC_DEVINL void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
SPEC_DEVINL void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// Shared-memory matrix descriptor of a K-major bf16 tile written by TMA with
// 128-byte swizzling: rows of 128 bytes (64 elements), 8-row groups 1024 bytes
// apart (stride byte offset), tile base 1024-byte aligned.  Advancing along K
// inside the 128-byte row is done by adding the byte offset to the start
// address field (bits 0-13, in 16-byte units).
SPEC_DEVINL uint64_t sdesc_k128(uint32_t saddr) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);  // start address
  d |= static_cast<uint64_t>(1) << 16;                   // leading byte offset (unused here)
  d |= static_cast<uint64_t>(1024 >> 4) << 32;           // stride byte offset
  d |= static_cast<uint64_t>(1) << 46;                   // descriptor version (sm_100 family)
  d |= static_cast<uint64_t>(2) << 61;                   // layout: 128-byte swizzle
  return d;
}

// Instruction descriptor of kind::f16 with bf16 A/B, fp32 accumulate, both
// operands K-major, shape M x N.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4)                                   // D = f32
         | (1u << 7)                                 // A = bf16
         | (1u << 10)                                // B = bf16
         | (static_cast<uint32_t>(N >> 3) << 17)     // N / 8
         | (static_cast<uint32_t>(M >> 4) << 24);    // M / 16
}

// D[tmem] (+)= A[smem] * B[smem]^T, issued by one thread.
SPEC_DEVINL void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                           uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on `bar` once every previously issued tcgen05.mma of this thread
// has completed.
SPEC_DEVINL void umma_commit(uint64_t* bar) {
  asm volatile(
      "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
          smem_u32(bar))
      : "memory");
}
// Each thread of the warp reads 16 consecutive 32-bit columns of its TMEM
// lane (lane = the warp's quarter * 32 + lane id, encoded in taddr[31:16]).
SPEC_DEVINL void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
        "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Named barrier among `nthreads` threads (ids 1..15; 0 is __syncthreads).
SPEC_DEVINL void named_bar(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

SPEC_DEVINL bool elect_lane0() { return (threadIdx.x & 31) == 0; }

// -------------------------------------------------------------------- bf16
// Round fp32 to bf16, nearest with ties to even (finite inputs).
SPEC_DEVINL uint16_t f32_to_bf16(float x) {
  uint32_t u = __float_as_uint(x);
  u += 0x7FFFu + ((u >> 16) & 1u);
  return static_cast<uint16_t>(u >> 16);
}
SPEC_DEVINL float bf16_to_f32(uint16_t b) { return __uint_as_float(static_cast<uint32_t>(b) << 16); }
SPEC_DEVINL float bf16lo(uint32_t w) { return __uint_as_float(w << 16); }
SPEC_DEVINL float bf16hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
SPEC_DEVINL uint32_t pack_bf16x2(float lo, float hi) {
  return static_cast<uint32_t>(f32_to_bf16(lo)) | (static_cast<uint32_t>(f32_to_bf16(hi)) << 16);
}

// --------------------------------------------------------------- reductions
SPEC_DEVINL float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}
SPEC_DEVINL float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

}  // namespace spec
