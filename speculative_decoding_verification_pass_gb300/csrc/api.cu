// The C ABI declared in include/spec_verify.h: argument validation, the
// weight and workspace layouts, TMA descriptors and the launch sequence of
// one verification pass.  No device memory is allocated here.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "internal.h"

using namespace spec;

namespace {

thread_local std::string g_cuda_error;

int cuda_fail(cudaError_t e) {
  g_cuda_error = cudaGetErrorString(e);
  return SPEC_ECUDA;
}

#define SPEC_CUDA(call)                        \
  do {                                         \
    cudaError_t e_ = (call);                   \
    if (e_ != cudaSuccess) return cuda_fail(e_); \
  } while (0)

constexpr size_t kAlign = 256;
constexpr int kMaxGrid = 512;      // stream-K grid cap (>= 3 x SM count of the part)
constexpr int kMaxTok = 256;       // token rows per GEMM launch (UMMA N limit)
constexpr int kMaxM = 512;         // token rows per pass
constexpr int kMaxN = 128;         // gamma + 1 per pass
// Shared-memory budget of one GEMM CTA (ring stages).  Two ~100 KB CTAs per SM
// stream faster than one CTA with a ring twice as deep (each CTA's stage
// round trip, not the bytes in flight, caps its rate).  Tunable with the
// environment variable SPEC_GEMM_SMEM_KB for sweeps.
size_t gemm_smem_budget() {
  static size_t v = [] {
    const char* e = getenv("SPEC_GEMM_SMEM_KB");
    long kb = e ? atol(e) : 100;
    if (kb < 48) kb = 48;
    if (kb > 220) kb = 220;
    return static_cast<size_t>(kb) * 1024;
  }();
  return v;
}
// K sub-tiles of 64 per pipeline stage (SPEC_GEMM_KSUB, default 2).
int gemm_ksub() {
  static int v = [] {
    const char* e = getenv("SPEC_GEMM_KSUB");
    int x = e ? atoi(e) : 2;
    return x == 1 ? 1 : 2;
  }();
  return v;
}
// Stream-K grid: SM count x SPEC_GEMM_CTAS_PER_SM (default 2).
int gemm_ctas_per_sm() {
  static int v = [] {
    const char* e = getenv("SPEC_GEMM_CTAS_PER_SM");
    int x = e ? atoi(e) : 2;
    return x < 1 ? 1 : (x > 3 ? 3 : x);
  }();
  return v;
}

// Shared-memory budget of the persistent decode forward's CTA (one per SM):
// SPEC_MK_SMEM_KB, default 220.
int mk_smem_kb() {
  static int v = [] {
    const char* e = getenv("SPEC_MK_SMEM_KB");
    int x = e ? atoi(e) : 220;
    return x < 64 ? 64 : (x > 224 ? 224 : x);
  }();
  return v;
}
// Decode-shaped passes run as one persistent kernel unless the environment
// sets SPEC_FORWARD_PERSISTENT=0 (read per call: the per-kernel schedule
// stays selectable for comparison).
bool mk_enabled() {
  const char* e = getenv("SPEC_FORWARD_PERSISTENT");
  return !(e && e[0] == '0');
}
// Its attention runs on the tensor cores where the shape allows, unless the
// environment sets SPEC_ATTENTION_TC=0 (read per call, for comparison).
// ... and loads its blocks with TMA unless SPEC_ATTENTION_TMA=0 (read per call).
bool mk_att_tma_enabled() {
  const char* e = getenv("SPEC_ATTENTION_TMA");
  return !(e && e[0] == '0');
}
bool mk_att_tc_enabled() {
  const char* e = getenv("SPEC_ATTENTION_TC");
  return !(e && e[0] == '0');
}

// The most key chunks a (sequence, KV head) of the persistent forward's
// attention may be cut into (the workspace's partials): enough for about four
// units per CTA of any grid up to kMaxGrid, at most one per 64 cache slots.
int mk_att_chunks_max(int pairs, int slot_chunks) {
  const int p = std::max(1, pairs);
  return std::max(1, std::min(slot_chunks, std::max(kMaxGrid / p, (4 * kMaxGrid + p - 1) / p)));
}

size_t align_up(size_t x, size_t a = kAlign) { return (x + a - 1) / a * a; }
int round_up(int x, int a) { return (x + a - 1) / a * a; }

bool cfg_ok(const spec_model_config* c) {
  if (!c) return false;
  if (c->n_layers < 0 || c->d_model <= 0 || c->vocab <= 0) return false;
  if (c->d_model % 128) return false;
  if (c->n_layers == 0) return true;
  if (c->n_heads <= 0 || c->n_kv_heads <= 0 || c->n_heads % c->n_kv_heads) return false;
  if (c->d_model % c->n_heads) return false;
  const int hd = c->d_model / c->n_heads;
  if (hd != 64 && hd != 128) return false;
  if (c->d_ffn <= 0 || c->d_ffn % 64) return false;
  if (!(c->rms_eps > 0.f) || !(c->rope_theta > 1.f)) return false;
  return true;
}

struct Layout {
  size_t embed, head, gfinal, rope;
  std::vector<size_t> g_attn, g_mlp, wqkv, wo, wgu, wd;
  size_t total;
};

Layout layout_of(const spec_model_config& c) {
  Layout L;
  const size_t d = c.d_model, V = c.vocab;
  const int hd = c.n_layers ? c.d_model / c.n_heads : 128;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + bytes);
    return at;
  };
  L.embed = take(V * d * 2);
  L.head = take(V * d * 2);
  L.gfinal = take(d * 4);
  L.rope = take(static_cast<size_t>(hd / 2) * 8);
  for (int l = 0; l < c.n_layers; ++l) {
    const size_t qkv = static_cast<size_t>(c.n_heads + 2 * c.n_kv_heads) * hd;
    L.g_attn.push_back(take(d * 4));
    L.g_mlp.push_back(take(d * 4));
    L.wqkv.push_back(take(qkv * d * 2));
    L.wo.push_back(take(d * static_cast<size_t>(c.n_heads) * hd * 2));
    L.wgu.push_back(take(2ull * c.d_ffn * d * 2));
    L.wd.push_back(take(d * c.d_ffn * 2));
  }
  L.total = o;
  return L;
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D bf16 [rows][cols] row-major, box = box_rows x 64 columns, 128-byte swizzle;
// rows outside the tensor read as zero.
bool make_tmap(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {cols, rows};
  cuuint64_t strides[1] = {cols * 2};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// q (or its lo half) as a 3-D tensor [M tokens][H heads][hd]: a box of 64
// dimensions x G heads x 32 / G tokens is 32 attention rows (token-major).
bool make_tmap_q(CUtensorMap* m, const void* base, uint64_t M, uint64_t H, uint64_t hd, uint32_t G) {
  auto fn = encode_fn();
  if (!fn || G == 0 || 32 % G) return false;
  cuuint64_t dims[3] = {hd, H, M};
  cuuint64_t strides[2] = {hd * 2, H * hd * 2};
  cuuint32_t box[3] = {64, G, 32 / G};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

struct WsPlan {
  size_t status, pos_base, seq_ok, mk_bar, counters, ssq, h, hb, hb_lo, q, q_lo, o, o_lo, act,
      act_lo, gpart, apart_o, apart_ml, mk_att_o, mk_att_ml;
  size_t total;
  int n_counters, attn_counter0, ssq_ld, splits, R, M, n, att_pairs;
};

int max_tiles(const spec_model_config& c) {
  int t = (c.vocab + 127) / 128;
  if (c.n_layers) {
    const int hd = c.d_model / c.n_heads;
    t = std::max(t, (c.n_heads + 2 * c.n_kv_heads) * hd / 128 + 1);
    t = std::max(t, c.d_model / 128);
    t = std::max(t, 2 * c.d_ffn / 128);
  }
  return t;
}

WsPlan plan_ws(const spec_model_config& c, int B, int gamma, int cap) {
  WsPlan p{};
  p.n = gamma + 1;
  p.M = B * p.n;
  const int M = p.M;
  const int mpad = round_up(std::max(M, 1), 16);
  const int ntok = std::min(kMaxTok, mpad);
  const int hd = c.n_layers ? c.d_model / c.n_heads : 128;
  const int Hkv = c.n_layers ? c.n_kv_heads : 1;
  const int G = c.n_layers ? c.n_heads / c.n_kv_heads : 1;
  p.ssq_ld = mpad;
  p.splits = (std::max(cap, 1) + kAttnChunk - 1) / kAttnChunk;
  p.R = p.n * G;
  p.attn_counter0 = max_tiles(c);
  p.n_counters = p.attn_counter0 + B * Hkv;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    size_t at = o;
    o = align_up(o + std::max<size_t>(bytes, 1));
    return at;
  };
  const size_t d = c.d_model;
  const size_t qd = c.n_layers ? static_cast<size_t>(c.n_heads) * hd : 0;
  p.status = take(68);  // status word; the persistent kernel's launch epoch at +64
  p.pos_base = take(static_cast<size_t>(B) * 4);
  p.seq_ok = take(static_cast<size_t>(B) * 4);
  p.mk_bar = take(256);  // directly before the counters: one memset clears both
  p.counters = take(static_cast<size_t>(p.n_counters) * 4);
  p.ssq = take(d / 128 * mpad * 4);
  p.h = take(static_cast<size_t>(M) * d * 4);
  p.hb = take(static_cast<size_t>(M) * d * 2);
  p.hb_lo = take(static_cast<size_t>(M) * d * 2);
  p.q = take(static_cast<size_t>(M) * qd * 2);
  p.q_lo = take(static_cast<size_t>(M) * qd * 2);
  p.o = take(static_cast<size_t>(M) * qd * 2);
  p.o_lo = take(static_cast<size_t>(M) * qd * 2);
  p.act = take(static_cast<size_t>(M) * c.d_ffn * 2);
  p.act_lo = take(static_cast<size_t>(M) * c.d_ffn * 2);
  p.gpart = take(static_cast<size_t>(kMaxGrid) * 2 * ntok * 128 * 4);  // summed partials: ntok columns
  const size_t rows = c.n_layers ? static_cast<size_t>(B) * Hkv * p.splits * p.R : 0;
  p.apart_o = take(rows * hd * 4);
  p.apart_ml = take(rows * 2 * 4);
  p.att_pairs = mk_att_chunks_max(B * Hkv, (std::max(cap, 1) + 63) / 64);
  const size_t urows = c.n_layers ? static_cast<size_t>(B) * Hkv * p.att_pairs * kMkAttRows : 0;
  p.mk_att_o = take(urows * hd * 4);
  p.mk_att_ml = take(urows * 2 * 4);
  p.total = o;
  return p;
}

struct TimedLaunch {
  cudaEvent_t a, b;
  int kind;
  double bytes;
};

}  // namespace

struct spec_model {
  spec_model_config cfg;
  int hd, G, qkv_rows, sm_count;
  uint8_t* base;
  size_t bytes;
  Layout L;
  std::vector<CUtensorMap> tm_qkv, tm_o, tm_gu, tm_d;
  CUtensorMap tm_head;
  bool timing = false;
  std::vector<TimedLaunch> pending;
  std::vector<cudaEvent_t> free_events;
};

namespace {

cudaEvent_t take_event(spec_model* m) {
  if (!m->free_events.empty()) {
    cudaEvent_t e = m->free_events.back();
    m->free_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

struct Ctx {
  const spec_model* m;
  cudaStream_t st;
  bool timing;
};

// Launch one GEMM over all token chunks of M rows.  With x_lo (the bf16
// residual of the activations) both halves of x = hi + lo enter the MMA
// (near-fp32 inputs at no extra weight traffic).
int run_gemm(const Ctx& cx, const CUtensorMap* tmW, const void* x, const void* x_lo, int M, int N,
             int K, GemmParams base) {
  spec_model* mm = const_cast<spec_model*>(cx.m);
  const int split_req = x_lo ? 1 : 0;
  // as few launches as the UMMA N limit allows, their token chunks of equal
  // size: a chunk's activation rows fill most of each ring stage, so a full
  // 256-row chunk leaves the ring two stages deep (320 rows: 160 + 160 ran
  // 33.7 ms a batch-64 pass against 36.1 for 256 + 64)
  const int n_launch = (M + kMaxTok - 1) / kMaxTok;
  const int max_tok = round_up((M + n_launch - 1) / n_launch, 16);
  for (int tok0 = 0; tok0 < M; tok0 += max_tok) {
    const int rows = std::min(max_tok, M - tok0);
    GemmParams p = base;
    p.N = N;
    p.K = K;
    p.M = M;
    p.tok0 = tok0;
    p.ntok = round_up(rows, 16);
    const int split = split_req ? (p.ntok <= 128 ? 1 : 2) : 0;
    p.split = split;
    p.ksub = (K % 128 == 0) ? gemm_ksub() : 1;
    p.kc = K / (64 * p.ksub);
    p.n_tiles = (N + 127) / 128;
    p.units = static_cast<long long>(p.n_tiles) * p.kc;
    // wide token tiles (prefill) need a bigger ring budget: one CTA per SM then
    size_t budget = gemm_smem_budget();
    int cps = gemm_ctas_per_sm();
    p.stages = gemm_max_stages(p.ntok << (split ? 1 : 0), budget, p.ksub);
    if (p.stages < 2) {
      p.ksub = 1;
      p.kc = K / 64;
      p.units = static_cast<long long>(p.n_tiles) * p.kc;
      p.stages = gemm_max_stages(p.ntok << (split ? 1 : 0), budget, 1);
    }
    if (p.stages < 2) {
      budget = 220 * 1024;
      cps = 1;
      p.stages = gemm_max_stages(p.ntok << (split ? 1 : 0), budget, 1);
    }
    if (p.stages < 2) return SPEC_ESIZE;
    CUtensorMap tmX, tmXlo;
    if (!make_tmap(&tmX, x, static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                   static_cast<uint32_t>(p.ntok)))
      return SPEC_ECUDA;
    if (split && !make_tmap(&tmXlo, x_lo, static_cast<uint64_t>(M), static_cast<uint64_t>(K),
                            static_cast<uint32_t>(p.ntok)))
      return SPEC_ECUDA;
    if (!split) tmXlo = tmX;
    int grid = static_cast<int>(std::min<long long>(std::min(cx.m->sm_count * cps, kMaxGrid), p.units));
    // 32-bit partition arithmetic in the kernel; at most 64 CTAs per tile
    if (static_cast<unsigned long long>(p.units) * grid >= (1ull << 32)) return SPEC_ESIZE;
    while (grid > 1 && (static_cast<long long>(grid) * p.kc + p.units - 1) / p.units + 1 > 64) --grid;
    TimedLaunch t{};
    if (cx.timing) {
      t.a = take_event(mm);
      t.b = take_event(mm);
      t.kind = 0;
      t.bytes = static_cast<double>(N) * K * 2 + static_cast<double>(rows) * K * 2;
      cudaEventRecord(t.a, cx.st);
    }
    SPEC_CUDA(launch_gemm(tmW, &tmX, &tmXlo, p, grid, cx.st, !cx.timing));
    if (cx.timing) {
      cudaEventRecord(t.b, cx.st);
      mm->pending.push_back(t);
    }
  }
  return SPEC_OK;
}

}  // namespace

extern "C" {

const char* spec_status_string(int s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_EINVAL: return "invalid argument";
    case SPEC_ESIZE: return "size out of range or buffer too small";
    case SPEC_ECUDA: return "CUDA error";
    case SPEC_EDEVICE: return "the device reported an error (status word set)";
    case SPEC_ETIMEOUT: return "a bounded device wait gave up";
    case SPEC_ENOTSUP: return "unsupported device or configuration";
    default: return "unknown status";
  }
}

const char* spec_last_cuda_error(void) { return g_cuda_error.c_str(); }

size_t spec_model_weight_bytes(const spec_model_config* cfg) {
  if (!cfg_ok(cfg)) return 0;
  return layout_of(*cfg).total;
}

int spec_model_create(const spec_model_config* cfg, uint64_t seed, void* d_weights,
                      size_t weight_bytes, void* stream, spec_model** out) {
  if (!out || !d_weights) return SPEC_EINVAL;
  *out = nullptr;
  if (!cfg_ok(cfg)) return SPEC_EINVAL;
  const Layout L = layout_of(*cfg);
  if (weight_bytes < L.total) return SPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_weights) % kAlign) return SPEC_EINVAL;
  int dev = 0;
  SPEC_CUDA(cudaGetDevice(&dev));
  cudaDeviceProp prop;
  SPEC_CUDA(cudaGetDeviceProperties(&prop, dev));
  if (prop.major != 10 || prop.minor != 3) return SPEC_ENOTSUP;
  if (!encode_fn()) return SPEC_ENOTSUP;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const spec_model_config& c = *cfg;
  auto* m = new spec_model();
  m->cfg = c;
  m->hd = c.n_layers ? c.d_model / c.n_heads : 128;
  m->G = c.n_layers ? c.n_heads / c.n_kv_heads : 1;
  m->qkv_rows = c.n_layers ? (c.n_heads + 2 * c.n_kv_heads) * m->hd : 0;
  m->sm_count = prop.multiProcessorCount;
  m->base = static_cast<uint8_t*>(d_weights);
  m->bytes = weight_bytes;
  m->L = L;
  uint8_t* B = m->base;
  const long long d = c.d_model, V = c.vocab, hd = m->hd;
  auto fail = [&](int code) {
    delete m;
    return code;
  };
  auto gen = [&](size_t off, long long rows, long long cols, int tid, int brows, int stride) {
    return launch_init_weights(reinterpret_cast<uint16_t*>(B + off), rows, cols, tid, seed, brows,
                               stride, st);
  };
  cudaError_t e;
  if ((e = gen(L.embed, V, d, 0, static_cast<int>(V), static_cast<int>(V))) != cudaSuccess)
    return fail(cuda_fail(e));
  if ((e = gen(L.head, V, d, 1, static_cast<int>(V), static_cast<int>(V))) != cudaSuccess)
    return fail(cuda_fail(e));
  if ((e = launch_fill_f32(reinterpret_cast<float*>(B + L.gfinal), d, 1.0f, st)) != cudaSuccess)
    return fail(cuda_fail(e));
  if ((e = launch_rope_table(reinterpret_cast<float2*>(B + L.rope), static_cast<int>(hd),
                             c.rope_theta, st)) != cudaSuccess)
    return fail(cuda_fail(e));
  const long long qd = static_cast<long long>(c.n_heads) * hd, kd = static_cast<long long>(c.n_kv_heads) * hd;
  const long long ffn = c.d_ffn;
  for (int l = 0; l < c.n_layers; ++l) {
    const int t0 = 2 + 7 * l;
    const size_t qkv = L.wqkv[l];
    struct G {
      size_t off;
      long long rows, cols;
      int tid, brows, stride;
    } gs[] = {
        {qkv, qd, d, t0 + 0, static_cast<int>(qd), static_cast<int>(qd)},
        {qkv + static_cast<size_t>(qd * d * 2), kd, d, t0 + 1, static_cast<int>(kd), static_cast<int>(kd)},
        {qkv + static_cast<size_t>((qd + kd) * d * 2), kd, d, t0 + 2, static_cast<int>(kd), static_cast<int>(kd)},
        {L.wo[l], d, qd, t0 + 3, static_cast<int>(d), static_cast<int>(d)},
        {L.wgu[l], ffn, d, t0 + 4, 64, 128},
        {L.wgu[l] + static_cast<size_t>(64 * d * 2), ffn, d, t0 + 5, 64, 128},
        {L.wd[l], d, ffn, t0 + 6, static_cast<int>(d), static_cast<int>(d)},
    };
    for (const G& g : gs)
      if ((e = gen(g.off, g.rows, g.cols, g.tid, g.brows, g.stride)) != cudaSuccess)
        return fail(cuda_fail(e));
    if ((e = launch_fill_f32(reinterpret_cast<float*>(B + L.g_attn[l]), d, 1.0f, st)) != cudaSuccess)
      return fail(cuda_fail(e));
    if ((e = launch_fill_f32(reinterpret_cast<float*>(B + L.g_mlp[l]), d, 1.0f, st)) != cudaSuccess)
      return fail(cuda_fail(e));
    CUtensorMap t;
    if (!make_tmap(&t, B + L.wqkv[l], m->qkv_rows, d, 128)) return fail(SPEC_ECUDA);
    m->tm_qkv.push_back(t);
    if (!make_tmap(&t, B + L.wo[l], d, qd, 128)) return fail(SPEC_ECUDA);
    m->tm_o.push_back(t);
    if (!make_tmap(&t, B + L.wgu[l], 2 * ffn, d, 128)) return fail(SPEC_ECUDA);
    m->tm_gu.push_back(t);
    if (!make_tmap(&t, B + L.wd[l], d, ffn, 128)) return fail(SPEC_ECUDA);
    m->tm_d.push_back(t);
  }
  if (!make_tmap(&m->tm_head, B + L.head, V, d, 128)) return fail(SPEC_ECUDA);
  *out = m;
  return SPEC_OK;
}

int spec_model_destroy(spec_model* m) {
  if (!m) return SPEC_OK;
  for (auto& t : m->pending) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  for (auto e : m->free_events) cudaEventDestroy(e);
  delete m;
  return SPEC_OK;
}

int spec_model_tensor(const spec_model* m, int layer, int which, const void** d_ptr,
                      int64_t shape[2], int* block_rows, int* row_stride_rows) {
  if (!m || !d_ptr || !shape || !block_rows || !row_stride_rows) return SPEC_EINVAL;
  const spec_model_config& c = m->cfg;
  const int64_t d = c.d_model, V = c.vocab, hd = m->hd;
  const int64_t qd = static_cast<int64_t>(c.n_heads) * hd, kd = static_cast<int64_t>(c.n_kv_heads) * hd;
  const uint8_t* B = m->base;
  int64_t rows = 0, cols = 0;
  const uint8_t* p = nullptr;
  int brows = 0, stride = 0;
  if (layer == -1) {
    if (which == 0) p = B + m->L.embed;
    else if (which == 1) p = B + m->L.head;
    else return SPEC_EINVAL;
    rows = V;
    cols = d;
  } else {
    if (layer < 0 || layer >= c.n_layers) return SPEC_EINVAL;
    const size_t qkv = m->L.wqkv[layer];
    switch (which) {
      case 0: p = B + qkv; rows = qd; cols = d; break;
      case 1: p = B + qkv + qd * d * 2; rows = kd; cols = d; break;
      case 2: p = B + qkv + (qd + kd) * d * 2; rows = kd; cols = d; break;
      case 3: p = B + m->L.wo[layer]; rows = d; cols = qd; break;
      case 4: p = B + m->L.wgu[layer]; rows = c.d_ffn; cols = d; brows = 64; stride = 128; break;
      case 5: p = B + m->L.wgu[layer] + 64 * d * 2; rows = c.d_ffn; cols = d; brows = 64; stride = 128; break;
      case 6: p = B + m->L.wd[layer]; rows = d; cols = c.d_ffn; break;
      default: return SPEC_EINVAL;
    }
  }
  if (!brows) brows = stride = static_cast<int>(rows);
  *d_ptr = p;
  shape[0] = rows;
  shape[1] = cols;
  *block_rows = brows;
  *row_stride_rows = stride;
  return SPEC_OK;
}

size_t spec_kv_bytes(const spec_model_config* cfg, int batch, int capacity) {
  if (!cfg_ok(cfg) || batch < 0 || capacity < 0 || cfg->n_layers == 0) return 0;
  const size_t hd = cfg->d_model / cfg->n_heads;
  return static_cast<size_t>(cfg->n_layers) * batch * cfg->n_kv_heads * capacity * hd * 2;
}

size_t spec_workspace_bytes(const spec_model_config* cfg, int batch, int gamma, int capacity) {
  if (!cfg_ok(cfg) || batch < 0 || gamma < 0 || capacity < 0) return 0;
  return plan_ws(*cfg, batch, gamma, capacity).total;
}

// Page table of a paged cache (table == nullptr: the contiguous layout).
struct PageDesc {
  const int32_t* table = nullptr;
  int max_pages = 0, n_pages = 0;
};

// The verification forward; d_anc / d_depth describe a draft tree per
// sequence (nullptr: the chain, node j at position len + j seeing new slots
// 0..j); pg the page table of a paged cache (kv->capacity = its logical
// capacity).
static int verify_forward_impl(const spec_model* m, const int32_t* d_tokens, const uint64_t* d_anc,
                               const int32_t* d_depth, int batch, int gamma, const spec_kv_cache* kv,
                               float* d_logits, void* d_ws, size_t ws_bytes, void* stream,
                               const PageDesc& pg = PageDesc{}) {
  if (!m || !d_tokens || !kv || !d_logits || !d_ws) return SPEC_EINVAL;
  if (batch < 0 || gamma < 0) return SPEC_EINVAL;
  const spec_model_config& c = m->cfg;
  if (c.n_layers == 0) return SPEC_ENOTSUP;
  if (!kv->k || !kv->v || !kv->len) return SPEC_EINVAL;
  if (kv->batch != batch || kv->capacity <= 0) return SPEC_EINVAL;
  if (kv->capacity > kAttnChunk * kAttnMaxChunks) return SPEC_ESIZE;
  const int n = gamma + 1;
  if (n > kMaxN || static_cast<long long>(batch) * n > kMaxM) return SPEC_ESIZE;
  if (batch == 0) return SPEC_OK;
  const WsPlan P = plan_ws(c, batch, gamma, kv->capacity);
  if (ws_bytes < P.total) return SPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_ws) % kAlign) return SPEC_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* W = static_cast<uint8_t*>(d_ws);
  uint8_t* B = m->base;
  const Layout& L = m->L;
  const int M = P.M, d = c.d_model, hd = m->hd, H = c.n_heads, Hkv = c.n_kv_heads;
  const int qd = H * hd;
  int32_t* status = reinterpret_cast<int32_t*>(W + P.status);
  int32_t* counters = reinterpret_cast<int32_t*>(W + P.counters);
  float* ssq = reinterpret_cast<float*>(W + P.ssq);
  float* h = reinterpret_cast<float*>(W + P.h);
  uint16_t* hb = reinterpret_cast<uint16_t*>(W + P.hb);
  uint16_t* hb_lo = reinterpret_cast<uint16_t*>(W + P.hb_lo);
  uint16_t* q = reinterpret_cast<uint16_t*>(W + P.q);
  uint16_t* q_lo = reinterpret_cast<uint16_t*>(W + P.q_lo);
  uint16_t* o = reinterpret_cast<uint16_t*>(W + P.o);
  uint16_t* o_lo = reinterpret_cast<uint16_t*>(W + P.o_lo);
  uint16_t* act = reinterpret_cast<uint16_t*>(W + P.act);
  uint16_t* act_lo = reinterpret_cast<uint16_t*>(W + P.act_lo);
  int32_t* pos_base = reinterpret_cast<int32_t*>(W + P.pos_base);
  int32_t* seq_ok = reinterpret_cast<int32_t*>(W + P.seq_ok);
  const Ctx cx{m, st, m->timing};
  const bool pdl = !m->timing;

  // ---- decode shapes: the whole pass as one persistent cooperative kernel
  {
    const int ntok = round_up(M, 16);
    const int fpt = d / 128;
    const bool shape_ok = mk_enabled() && M <= 128 && P.R <= kMkAttRows && c.n_layers <= kMkMaxLayers &&
                          (fpt & (fpt - 1)) == 0 && fpt <= 128;
    // one CTA per SM with a deep ring (the ring also absorbs grid barriers)
    int stages = shape_ok ? forward_max_stages(ntok, hd, static_cast<size_t>(mk_smem_kb()) * 1024) : 0;
    const int cps = stages >= 2 ? forward_ctas_per_sm(ntok, stages, hd) : 0;
    const long long stride = c.n_layers > 1 ? static_cast<long long>(L.g_attn[1] - L.g_attn[0]) : 0;
    bool uniform = true;
    for (int l = 1; l < c.n_layers; ++l)
      uniform = uniform && static_cast<long long>(L.g_attn[l] - L.g_attn[0]) == stride * l &&
                static_cast<long long>(L.g_mlp[l] - L.g_mlp[0]) == stride * l;
    // the stream-K words (8 bytes each) of at most kMaxGrid / 2 CTAs fit the partials area
    if (shape_ok && cps >= 1 && uniform && m->sm_count * cps <= kMaxGrid / 2) {
      MkParams* mp = new MkParams();
      MkParams& Q = *mp;
      const void* xs[6] = {hb, hb_lo, o, o_lo, act, act_lo};
      const int xk[6] = {d, d, qd, qd, c.d_ffn, c.d_ffn};
      bool ok = true;
      for (int i = 0; i < 6 && ok; ++i)
        ok = make_tmap(&Q.xmap[i], xs[i], static_cast<uint64_t>(M), static_cast<uint64_t>(xk[i]),
                       static_cast<uint32_t>(ntok));
      if (!ok) {
        delete mp;
        return SPEC_ECUDA;
      }
      for (int l = 0; l < c.n_layers; ++l) {
        Q.wmap[4 * l + 0] = m->tm_qkv[l];
        Q.wmap[4 * l + 1] = m->tm_o[l];
        Q.wmap[4 * l + 2] = m->tm_gu[l];
        Q.wmap[4 * l + 3] = m->tm_d[l];
      }
      Q.wmap[4 * c.n_layers] = m->tm_head;
      Q.L = c.n_layers;
      Q.d = d;
      Q.H = H;
      Q.Hkv = Hkv;
      Q.hd = hd;
      Q.ffn = c.d_ffn;
      Q.V = c.vocab;
      Q.qkv_rows = m->qkv_rows;
      Q.B = batch;
      Q.n = n;
      Q.M = M;
      Q.ntok = ntok;
      Q.cap = kv->capacity;
      Q.stages = stages;
      Q.ssq_ld = P.ssq_ld;
      const int grid = std::min(m->sm_count * cps, kMaxGrid);
      Q.att_nch = P.att_pairs;  // the most chunks a sequence's keys may be cut into
      Q.att_tc = mk_att_tc_enabled() && forward_att_tc(ntok, stages, hd) ? 1 : 0;
      Q.nacc = forward_acc_buffers(ntok, Q.att_tc != 0);
      if (Q.att_tc && mk_att_tma_enabled() && hd == 128 && 32 % (H / Hkv) == 0) {
        const uint64_t kv_rows = pg.table ? static_cast<uint64_t>(c.n_layers) * pg.n_pages * Hkv * SPEC_PAGE_SLOTS
                                          : static_cast<uint64_t>(c.n_layers) * batch * Hkv * kv->capacity;
        const uint32_t box = pg.table ? SPEC_PAGE_SLOTS : 128;
        // the loads' row coordinates are 32-bit
        Q.att_tma = kv_rows + 128 < (1ull << 31) && make_tmap(&Q.kvmap[0], kv->k, kv_rows, hd, box) && make_tmap(&Q.kvmap[1], kv->v, kv_rows, hd, box) &&
                            make_tmap_q(&Q.qmap[0], q, M, H, hd, H / Hkv) && make_tmap_q(&Q.qmap[1], q_lo, M, H, hd, H / Hkv)
                        ? 1
                        : 0;
      }
      Q.eps = c.rms_eps;
      Q.inv_d = 1.0f / d;
      Q.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(hd)));
      Q.embed = reinterpret_cast<const uint16_t*>(B + L.embed);
      Q.rope = reinterpret_cast<const float2*>(B + L.rope);
      Q.anc = d_anc;
      Q.depth = d_depth;
      Q.gfinal = reinterpret_cast<const float*>(B + L.gfinal);
      Q.g_attn0 = reinterpret_cast<const float*>(B + L.g_attn[0]);
      Q.g_mlp0 = reinterpret_cast<const float*>(B + L.g_mlp[0]);
      Q.layer_stride = stride;
      Q.kc = static_cast<uint16_t*>(kv->k);
      Q.vc = static_cast<uint16_t*>(kv->v);
      Q.layer_kv = pg.table ? static_cast<long long>(pg.n_pages) * Hkv * SPEC_PAGE_SLOTS * hd
                            : static_cast<long long>(batch) * Hkv * kv->capacity * hd;
      Q.kv_table = pg.table;
      Q.kv_max_pages = pg.max_pages;
      Q.kv_n_pages = pg.n_pages;
      Q.len = kv->len;
      Q.tokens = d_tokens;
      Q.logits = d_logits;
      Q.h = h;
      Q.hb = hb;
      Q.hb_lo = hb_lo;
      Q.q = q;
      Q.q_lo = q_lo;
      Q.o = o;
      Q.o_lo = o_lo;
      Q.act = act;
      Q.act_lo = act_lo;
      Q.ssq = ssq;
      Q.partials = reinterpret_cast<float*>(W + P.gpart);
      Q.counters = counters;
      Q.bar = reinterpret_cast<unsigned*>(W + P.mk_bar);
      Q.epoch = reinterpret_cast<unsigned*>(W + P.status + 64);  // outside the per-launch memset
      Q.status = status;
      Q.pos_base = pos_base;
      Q.seq_ok = seq_ok;
      Q.att_o = reinterpret_cast<float*>(W + P.mk_att_o);
      Q.att_ml = reinterpret_cast<float*>(W + P.mk_att_ml);
      cudaError_t e = cudaMemsetAsync(W + P.mk_bar, 0, P.counters + P.n_counters * 4 - P.mk_bar, st);
      TimedLaunch t{};
      if (e == cudaSuccess && cx.timing) {
        t.a = take_event(const_cast<spec_model*>(m));
        t.b = take_event(const_cast<spec_model*>(m));
        t.kind = 2;
        double wbytes = static_cast<double>(c.vocab) * d * 2;
        for (int l = 0; l < c.n_layers; ++l)
          wbytes += (static_cast<double>(m->qkv_rows) * d + static_cast<double>(d) * qd +
                     2.0 * c.d_ffn * d + static_cast<double>(d) * c.d_ffn) * 2;
        t.bytes = wbytes;
        cudaEventRecord(t.a, st);
      }
      if (e == cudaSuccess) e = launch_forward(Q, grid, hd, st);
      if (e == cudaSuccess && cx.timing) {
        cudaEventRecord(t.b, st);
        const_cast<spec_model*>(m)->pending.push_back(t);
      }
      delete mp;
      if (e != cudaSuccess) return cuda_fail(e);
      return SPEC_OK;
    }
  }

  EmbedParams ep{};
  ep.tokens = d_tokens;
  ep.embed = reinterpret_cast<const uint16_t*>(B + L.embed);
  ep.g0 = reinterpret_cast<const float*>(B + L.g_attn[0]);
  ep.h = h;
  ep.hb = hb;
  ep.hb_lo = hb_lo;
  ep.ssq = ssq;
  ep.ssq_ld = P.ssq_ld;
  ep.len = kv->len;
  ep.pos_base = pos_base;
  ep.seq_ok = seq_ok;
  ep.counters = counters;
  ep.n_counters = P.n_counters;
  ep.status = status;
  ep.B = batch;
  ep.n = n;
  ep.d = d;
  ep.V = c.vocab;
  ep.cap = kv->capacity;
  ep.kv_table = pg.table;
  ep.kv_max_pages = pg.max_pages;
  ep.kv_n_pages = pg.n_pages;
  SPEC_CUDA(launch_embed(ep, st, pdl));

  GemmParams g0{};
  g0.inv_d = 1.0f / d;
  g0.eps = c.rms_eps;
  g0.ssq_tiles = d / 128;
  g0.ssq_ld = P.ssq_ld;
  g0.d = d;
  g0.partials = reinterpret_cast<float*>(W + P.gpart);
  g0.counters = counters;
  g0.status = status;

  const size_t layer_kv = pg.table ? static_cast<size_t>(pg.n_pages) * Hkv * SPEC_PAGE_SLOTS * hd
                                   : static_cast<size_t>(batch) * Hkv * kv->capacity * hd;
  // decode shapes of head dim 128 past the persistent kernel (more than 128
  // token rows): the attention on the tensor cores, as launches of its own
  MkParams* tq = nullptr;
  if (hd == 128 && P.R <= kMkAttRows && batch <= 128 && mk_att_tc_enabled()) {
    tq = new MkParams();
    MkParams& A = *tq;
    A.B = batch;
    A.n = n;
    A.M = M;
    A.H = H;
    A.Hkv = Hkv;
    A.hd = hd;
    A.cap = kv->capacity;
    A.stages = kStepAttStages;
    A.att_nch = P.att_pairs;
    A.att_tc = 1;
    A.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(hd)));
    A.anc = d_anc;
    A.kc = static_cast<uint16_t*>(kv->k);
    A.vc = static_cast<uint16_t*>(kv->v);
    A.layer_kv = layer_kv;
    A.kv_table = pg.table;
    A.kv_max_pages = pg.max_pages;
    A.kv_n_pages = pg.n_pages;
    A.q = q;
    A.q_lo = q_lo;
    A.o = o;
    A.o_lo = o_lo;
    A.pos_base = pos_base;
    A.status = status;
    A.att_o = reinterpret_cast<float*>(W + P.mk_att_o);
    A.att_ml = reinterpret_cast<float*>(W + P.mk_att_ml);
    if (mk_att_tma_enabled() && 32 % (H / Hkv) == 0) {
      const uint64_t kv_rows = pg.table ? static_cast<uint64_t>(c.n_layers) * pg.n_pages * Hkv * SPEC_PAGE_SLOTS
                                        : static_cast<uint64_t>(c.n_layers) * batch * Hkv * kv->capacity;
      const uint32_t box = pg.table ? SPEC_PAGE_SLOTS : 128;
      // the loads' row coordinates are 32-bit
      A.att_tma = kv_rows + 128 < (1ull << 31) && make_tmap(&A.kvmap[0], kv->k, kv_rows, hd, box) && make_tmap(&A.kvmap[1], kv->v, kv_rows, hd, box) &&
                          make_tmap_q(&A.qmap[0], q, M, H, hd, H / Hkv) && make_tmap_q(&A.qmap[1], q_lo, M, H, hd, H / Hkv)
                      ? 1
                      : 0;
    }
  }
  struct Free {
    MkParams* p;
    ~Free() { delete p; }
  } free_tq{tq};
  for (int l = 0; l < c.n_layers; ++l) {
    uint16_t* kc = static_cast<uint16_t*>(kv->k) + l * layer_kv;
    uint16_t* vc = static_cast<uint16_t*>(kv->v) + l * layer_kv;
    {  // QKV projection: RMSNorm scale, RoPE, KV append
      GemmParams p = g0;
      p.epi = EPI_QKV;
      p.ssq_in = ssq;
      p.q = q;
      p.q_lo = q_lo;
      p.kcache = kc;
      p.vcache = vc;
      p.pos_base = pos_base;
      p.seq_ok = seq_ok;
      p.rope = reinterpret_cast<const float2*>(B + L.rope);
      p.depth = d_depth;
      p.kv_table = pg.table;
      p.kv_max_pages = pg.max_pages;
      p.kv_n_pages = pg.n_pages;
      p.n_per_seq = n;
      p.H = H;
      p.Hkv = Hkv;
      p.hd = hd;
      p.cap = kv->capacity;
      int r = run_gemm(cx, &m->tm_qkv[l], hb, hb_lo, M, m->qkv_rows, d, p);
      if (r) return r;
    }
    {  // attention over the cache
      AttnParams a{};
      a.q = q;
      a.q_lo = q_lo;
      a.kcache = kc;
      a.vcache = vc;
      a.o = o;
      a.o_lo = o_lo;
      a.pos_base = pos_base;
      a.anc = d_anc;
      a.kv_table = pg.table;
      a.kv_max_pages = pg.max_pages;
      a.kv_n_pages = pg.n_pages;
      a.part_o = reinterpret_cast<float*>(W + P.apart_o);
      a.part_ml = reinterpret_cast<float*>(W + P.apart_ml);
      a.counters = counters + P.attn_counter0;
      a.status = status;
      a.B = batch;
      a.n = n;
      a.H = H;
      a.Hkv = Hkv;
      a.hd = hd;
      a.cap = kv->capacity;
      a.splits = P.splits;
      a.R = P.R;
      a.scale_log2 = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(hd)));
      // decode shapes (<= 32 query rows per KV head) take the cluster path when
      // a rank's slice of the cache fits in shared memory
      a.cluster = P.R <= 32 ? attention_cluster_size(hd, kv->capacity, 200 * 1024) : 0;
      TimedLaunch t{};
      if (cx.timing) {
        t.a = take_event(const_cast<spec_model*>(m));
        t.b = take_event(const_cast<spec_model*>(m));
        t.kind = 1;
        cudaEventRecord(t.a, st);
      }
      if (tq)
        SPEC_CUDA(launch_attention_tc(*tq, l, m->sm_count, st));
      else
        SPEC_CUDA(launch_attention(a, st, pdl));
      if (cx.timing) {
        cudaEventRecord(t.b, st);
        const_cast<spec_model*>(m)->pending.push_back(t);
      }
    }
    {  // O projection + residual
      GemmParams p = g0;
      p.epi = EPI_RESID;
      p.h = h;
      p.hb = hb;
      p.hb_lo = hb_lo;
      p.g_next = reinterpret_cast<const float*>(B + L.g_mlp[l]);
      p.ssq_out = ssq;
      int r = run_gemm(cx, &m->tm_o[l], o, o_lo, M, d, qd, p);
      if (r) return r;
    }
    {  // gate/up + SwiGLU
      GemmParams p = g0;
      p.epi = EPI_SWIGLU;
      p.ssq_in = ssq;
      p.act = act;
      p.act_lo = act_lo;
      p.ffn = c.d_ffn;
      int r = run_gemm(cx, &m->tm_gu[l], hb, hb_lo, M, 2 * c.d_ffn, d, p);
      if (r) return r;
    }
    {  // down + residual; writes the next norm's input
      GemmParams p = g0;
      p.epi = EPI_RESID;
      p.h = h;
      p.hb = hb;
      p.hb_lo = hb_lo;
      p.g_next = reinterpret_cast<const float*>(B + (l + 1 < c.n_layers ? L.g_attn[l + 1] : L.gfinal));
      p.ssq_out = ssq;
      int r = run_gemm(cx, &m->tm_d[l], act, act_lo, M, d, c.d_ffn, p);
      if (r) return r;
    }
  }
  {  // final norm (scale in the epilogue) + LM head
    GemmParams p = g0;
    p.epi = EPI_STORE;
    p.ssq_in = ssq;
    p.out = d_logits;
    p.ldo = c.vocab;
    int r = run_gemm(cx, &m->tm_head, hb, hb_lo, M, c.vocab, d, p);
    if (r) return r;
  }
  return SPEC_OK;
}

int spec_verify_forward(const spec_model* m, const int32_t* d_tokens, int batch, int gamma,
                        const spec_kv_cache* kv, float* d_logits, void* d_ws, size_t ws_bytes,
                        void* stream) {
  return verify_forward_impl(m, d_tokens, nullptr, nullptr, batch, gamma, kv, d_logits, d_ws, ws_bytes,
                             stream);
}

size_t spec_paged_kv_bytes(const spec_model_config* cfg, int n_pages) {
  if (!cfg_ok(cfg) || n_pages < 0 || cfg->n_layers == 0) return 0;
  const size_t hd = static_cast<size_t>(cfg->d_model / cfg->n_heads);
  return static_cast<size_t>(cfg->n_layers) * n_pages * cfg->n_kv_heads * SPEC_PAGE_SLOTS * hd * 2;
}

static int paged_view(const spec_paged_kv_cache* kv, spec_kv_cache* view, PageDesc* pg) {
  if (!kv || !kv->k || !kv->v || !kv->len || !kv->table) return SPEC_EINVAL;
  if (kv->batch < 0 || kv->n_pages <= 0 || kv->max_pages <= 0) return SPEC_EINVAL;
  if (static_cast<long long>(kv->max_pages) * SPEC_PAGE_SLOTS > kAttnChunk * kAttnMaxChunks) return SPEC_ESIZE;
  view->k = kv->k;
  view->v = kv->v;
  view->len = kv->len;
  view->batch = kv->batch;
  view->capacity = kv->max_pages * SPEC_PAGE_SLOTS;
  pg->table = kv->table;
  pg->max_pages = kv->max_pages;
  pg->n_pages = kv->n_pages;
  return SPEC_OK;
}

int spec_verify_forward_paged(const spec_model* m, const int32_t* d_tokens, int batch, int gamma,
                              const spec_paged_kv_cache* kv, float* d_logits, void* d_ws,
                              size_t ws_bytes, void* stream) {
  spec_kv_cache view{};
  PageDesc pg;
  const int r = paged_view(kv, &view, &pg);
  if (r) return r;
  return verify_forward_impl(m, d_tokens, nullptr, nullptr, batch, gamma, &view, d_logits, d_ws, ws_bytes,
                             stream, pg);
}

int spec_paged_kv_truncate(const spec_paged_kv_cache* kv, const int32_t* d_n_accepted, int gamma,
                           void* d_ws, void* stream) {
  spec_kv_cache view{};
  PageDesc pg;
  const int r = paged_view(kv, &view, &pg);
  if (r) return r;
  return spec_kv_truncate(&view, d_n_accepted, gamma, d_ws, stream);
}

int spec_tree_masks(const int32_t* parents, int n_nodes, uint64_t* out_anc, int32_t* out_depth) {
  if (!parents || !out_anc || !out_depth || n_nodes < 1) return SPEC_EINVAL;
  if (n_nodes > kTreeMaxNodes) return SPEC_ESIZE;
  if (parents[0] != -1) return SPEC_EINVAL;
  for (int i = 1; i < n_nodes; ++i)
    if (parents[i] < 0 || parents[i] >= i) return SPEC_EINVAL;
  for (int i = 0; i < n_nodes; ++i) {
    uint64_t mask = 0;
    int depth = -1;
    for (int j = i; j != -1; j = parents[j]) {
      mask |= 1ull << j;
      ++depth;
    }
    out_anc[i] = mask;
    out_depth[i] = depth;
  }
  return SPEC_OK;
}

int spec_verify_forward_tree(const spec_model* m, const int32_t* d_tokens, const uint64_t* d_anc,
                             const int32_t* d_depth, int batch, int n_nodes, const spec_kv_cache* kv,
                             float* d_logits, void* d_ws, size_t ws_bytes, void* stream) {
  if (!d_anc || !d_depth || n_nodes < 1) return SPEC_EINVAL;
  if (n_nodes > kTreeMaxNodes) return SPEC_ESIZE;
  return verify_forward_impl(m, d_tokens, d_anc, d_depth, batch, n_nodes - 1, kv, d_logits, d_ws,
                             ws_bytes, stream);
}

int spec_lm_head(const spec_model* m, const uint16_t* d_hidden, int rows, float* d_logits,
                 void* d_ws, size_t ws_bytes, void* stream) {
  if (!m || !d_hidden || !d_logits || !d_ws) return SPEC_EINVAL;
  if (rows < 0) return SPEC_EINVAL;
  if (rows > kMaxM) return SPEC_ESIZE;
  if (rows == 0) return SPEC_OK;
  const spec_model_config& c = m->cfg;
  const WsPlan P = plan_ws(c, rows, 0, 1);
  if (ws_bytes < P.total) return SPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_ws) % kAlign) return SPEC_EINVAL;
  if (reinterpret_cast<uintptr_t>(d_hidden) % 16) return SPEC_EINVAL;
  uint8_t* W = static_cast<uint8_t*>(d_ws);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SPEC_CUDA(cudaMemsetAsync(W + P.counters, 0, static_cast<size_t>(P.n_counters) * 4, st));
  GemmParams p{};
  p.epi = EPI_STORE;
  p.out = d_logits;
  p.ldo = c.vocab;
  p.partials = reinterpret_cast<float*>(W + P.gpart);
  p.counters = reinterpret_cast<int32_t*>(W + P.counters);
  p.status = reinterpret_cast<int32_t*>(W + P.status);
  const Ctx cx{m, st, m->timing};
  return run_gemm(cx, &m->tm_head, d_hidden, nullptr, rows, c.vocab, c.d_model, p);
}

// LM head on caller-supplied stream-K scratch (used by the entry point that
// keeps its scratch in a static device array instead of a workspace).
int spec_internal_lm_head(const spec_model* m, const uint16_t* d_hidden, int rows, float* d_logits,
                          float* partials, int32_t* counters, int32_t* status, int max_vocab,
                          int max_grid, void* stream) {
  if (!m || !d_hidden || !d_logits || !partials || !counters || !status) return SPEC_EINVAL;
  if (rows <= 0) return rows == 0 ? SPEC_OK : SPEC_EINVAL;
  if (m->cfg.vocab > max_vocab || kMaxGrid > max_grid || rows > 16) return SPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_hidden) % 16) return SPEC_EINVAL;
  GemmParams p{};
  p.epi = EPI_STORE;
  p.out = d_logits;
  p.ldo = m->cfg.vocab;
  p.partials = partials;
  p.counters = counters;
  p.status = status;
  const Ctx cx{m, static_cast<cudaStream_t>(stream), false};
  return run_gemm(cx, &m->tm_head, d_hidden, nullptr, rows, m->cfg.vocab, m->cfg.d_model, p);
}

}  // extern "C"

namespace {

// Accept workspace: status word and grid-barrier counter, then the chunk
// partials of the cooperative accept grid, sized for the largest chunk count
// a launch may choose.
struct AcceptWs {
  size_t bar, part_ms, tot40, hist, sel, part_tot, part_last, total;
  int s_max;
};

int accept_chunks_max(int V) {
  const int by_size = (V + kAcceptMaxChunk - 1) / kAcceptMaxChunk;
  return std::min(V, std::max(512, by_size));
}

AcceptWs plan_accept(int B, int gamma, int V) {
  AcceptWs w{};
  const size_t n = static_cast<size_t>(gamma) + 1;
  w.s_max = accept_chunks_max(V);
  const size_t S = static_cast<size_t>(w.s_max);
  // the grid schedule serves batches of up to kAcceptGridRows rows; larger
  // ones run one CTA per sequence and need only the status word
  if (static_cast<long long>(B) * static_cast<long long>(n) > kAcceptGridRows) B = 0;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes);
    return o;
  };
  take(64);  // status word
  w.bar = take(64);
  w.part_ms = take(B * n * S * 8);
  w.tot40 = take(B * n * 8);
  w.hist = take(B * n * 4 * 256 * 8);
  w.sel = take(B * n * 4 * 2 * 8);
  w.part_tot = take(B * S * 2 * 8);
  w.part_last = take(B * S * 2 * 4);
  w.total = off;
  return w;
}

int device_sm_count() {
  static PerDevice<int> sms;
  int v = 0;
  if (!sms.get(
          [] {
            int dev = 0, n = 0;
            if (cudaGetDevice(&dev) != cudaSuccess) return 0;
            if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
              return 0;
            return n;
          },
          &v))
    return 0;
  return v;
}

}  // namespace

extern "C" {

size_t spec_accept_workspace_bytes(int batch, int gamma, int vocab) {
  if (batch < 0 || gamma < 0 || vocab <= 0) return 0;
  return plan_accept(batch, gamma, vocab).total;
}

static int accept_common_checks(int batch, int gamma, int vocab, float T, float top_p) {
  if (batch < 0 || gamma < 0 || vocab <= 0) return SPEC_EINVAL;
  if (!(T >= 0.f) || std::isinf(T)) return SPEC_EINVAL;
  if (!(top_p > 0.f && top_p <= 1.f)) return SPEC_EINVAL;
  // the nucleus select's exact 32-bit bin limbs hold up to 2^21 ids a row
  if (top_p < 1.f && vocab > kNucleusMaxVocab) return SPEC_ESIZE;
  return SPEC_OK;
}

int spec_accept(const float* d_target_logits, const float* d_draft_probs,
                const int32_t* d_draft_tokens, const float* d_uniforms, int batch, int gamma,
                int vocab, float temperature, float top_p, int32_t* d_out_tokens,
                int32_t* d_n_accepted, void* d_ws, size_t ws_bytes, void* stream) {
  int r = accept_common_checks(batch, gamma, vocab, temperature, top_p);
  if (r) return r;
  if (!d_target_logits || !d_out_tokens || !d_n_accepted || !d_ws) return SPEC_EINVAL;
  if (gamma > 0 && !d_draft_tokens) return SPEC_EINVAL;
  if (temperature > 0.f && ((gamma > 0 && !d_draft_probs) || !d_uniforms)) return SPEC_EINVAL;
  if (gamma + 1 > kAcceptMaxRows) return SPEC_ESIZE;
  const AcceptWs A = plan_accept(batch, gamma, vocab);
  if (ws_bytes < A.total) return SPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_ws) % 16) return SPEC_EINVAL;
  if (batch == 0) return SPEC_OK;
  uint8_t* W = static_cast<uint8_t*>(d_ws);
  AcceptParams p{};
  const char* ge = getenv("SPEC_ACCEPT_GRID");  // 0: one CTA per sequence (read per call)
  p.grid = (ge && ge[0] == '0') ? 0 : 1;
  // chunks: at most kAcceptMaxChunk ids each, and about two units per SM
  const int rows = batch * (gamma + 1);
  const int want = std::max(1, (2 * device_sm_count() + rows - 1) / rows);
  int S = std::min(A.s_max, std::max((vocab + kAcceptMaxChunk - 1) / kAcceptMaxChunk, want));
  const int C = (vocab + S - 1) / S;
  S = (vocab + C - 1) / C;
  p.S = S;
  p.C = C;
  p.bar = reinterpret_cast<unsigned*>(W + A.bar);
  p.part_ms = reinterpret_cast<float2*>(W + A.part_ms);
  p.tot40 = reinterpret_cast<unsigned long long*>(W + A.tot40);
  p.hist = reinterpret_cast<unsigned long long*>(W + A.hist);
  p.sel = reinterpret_cast<unsigned long long*>(W + A.sel);
  p.part_tot = reinterpret_cast<unsigned long long*>(W + A.part_tot);
  p.part_last = reinterpret_cast<int*>(W + A.part_last);
  p.logits = d_target_logits;
  p.q = d_draft_probs;
  p.draft = d_draft_tokens;
  p.u = d_uniforms;
  p.out = d_out_tokens;
  p.n_acc = d_n_accepted;
  p.status = static_cast<int32_t*>(d_ws);
  p.B = batch;
  p.gamma = gamma;
  p.V = vocab;
  p.T = temperature;
  p.top_p = top_p;
  SPEC_CUDA(launch_accept(p, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

int spec_draft_sample(const float* d_logits, int rows, int vocab, float temperature, float top_p,
                      const float* d_uniforms, float* d_probs, int32_t* d_tokens, void* d_ws,
                      size_t ws_bytes, void* stream) {
  int r = accept_common_checks(rows, 0, vocab, temperature, top_p);
  if (r) return r;
  if (!d_logits || !d_tokens || !d_ws) return SPEC_EINVAL;
  if (temperature > 0.f && !d_uniforms) return SPEC_EINVAL;
  if (ws_bytes < spec_accept_workspace_bytes(rows, 0, vocab)) return SPEC_ESIZE;
  if (rows == 0) return SPEC_OK;
  SampleParams p{};
  p.logits = d_logits;
  p.u = d_uniforms;
  p.probs = d_probs;
  p.tokens = d_tokens;
  p.status = static_cast<int32_t*>(d_ws);
  p.R = rows;
  p.V = vocab;
  p.T = temperature;
  p.top_p = top_p;
  SPEC_CUDA(launch_sample(p, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

int spec_kv_truncate(const spec_kv_cache* kv, const int32_t* d_n_accepted, int gamma, void* d_ws,
                     void* stream) {
  if (!kv || !kv->len || !d_n_accepted || !d_ws) return SPEC_EINVAL;
  if (gamma < 0 || kv->batch < 0) return SPEC_EINVAL;
  SPEC_CUDA(launch_truncate(kv->len, d_n_accepted, kv->batch, gamma, static_cast<int32_t*>(d_ws),
                            static_cast<cudaStream_t>(stream), true));
  return SPEC_OK;
}

int spec_mask_logits(float* d_logits, const uint32_t* d_allowed, int rows, int vocab, void* d_ws,
                     void* stream) {
  if (!d_logits || !d_allowed || !d_ws || rows < 0 || vocab <= 0) return SPEC_EINVAL;
  if (rows > 65535) return SPEC_ESIZE;
  SPEC_CUDA(launch_mask_logits(d_logits, d_allowed, rows, vocab, static_cast<int32_t*>(d_ws),
                               static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

size_t spec_tree_accept_workspace_bytes(int batch, int vocab) {
  if (batch < 0 || vocab <= 0) return 0;
  return kAlign;  // the status word: the walk keeps its residuals in closed form
}

int spec_tree_accept(const float* d_target_logits, const float* d_draft_probs,
                     const int32_t* d_node_tokens, const int32_t* d_parents,
                     const float* d_uniforms, int batch, int n_nodes, int vocab, float temperature,
                     float top_p, int32_t* d_out_tokens, int32_t* d_out_path,
                     int32_t* d_n_accepted, void* d_ws, size_t ws_bytes, void* stream) {
  int r = accept_common_checks(batch, 0, vocab, temperature, top_p);
  if (r) return r;
  if (n_nodes < 1) return SPEC_EINVAL;
  if (n_nodes > kTreeMaxNodes) return SPEC_ESIZE;
  if (!d_target_logits || !d_node_tokens || !d_parents || !d_out_tokens || !d_out_path ||
      !d_n_accepted || !d_ws)
    return SPEC_EINVAL;
  if (temperature > 0.f && (!d_draft_probs || !d_uniforms)) return SPEC_EINVAL;
  if (ws_bytes < spec_tree_accept_workspace_bytes(batch, vocab)) return SPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(d_ws) % 16) return SPEC_EINVAL;
  if (batch == 0) return SPEC_OK;
  TreeAcceptParams p{};
  p.logits = d_target_logits;
  p.q = d_draft_probs;
  p.tokens = d_node_tokens;
  p.parents = d_parents;
  p.u = d_uniforms;
  p.out = d_out_tokens;
  p.path = d_out_path;
  p.n_acc = d_n_accepted;
  p.status = static_cast<int32_t*>(d_ws);
  p.B = batch;
  p.n = n_nodes;
  p.V = vocab;
  p.T = temperature;
  p.top_p = top_p;
  SPEC_CUDA(launch_tree_accept(p, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

int spec_kv_tree_commit(const spec_model* m, const spec_kv_cache* kv, const int32_t* d_path,
                        const int32_t* d_n_accepted, int n_nodes, void* d_ws, void* stream) {
  if (!m || !kv || !kv->k || !kv->v || !kv->len || !d_path || !d_n_accepted || !d_ws)
    return SPEC_EINVAL;
  if (n_nodes < 1 || kv->batch < 0 || kv->capacity < 0) return SPEC_EINVAL;
  if (n_nodes > kTreeMaxNodes) return SPEC_ESIZE;
  if (reinterpret_cast<uintptr_t>(kv->k) % 16 || reinterpret_cast<uintptr_t>(kv->v) % 16)
    return SPEC_EINVAL;
  const spec_model_config& c = m->cfg;
  TreeCommitParams p{};
  p.k = static_cast<uint16_t*>(kv->k);
  p.v = static_cast<uint16_t*>(kv->v);
  p.len = kv->len;
  p.path = d_path;
  p.n_acc = d_n_accepted;
  p.status = static_cast<int32_t*>(d_ws);
  p.L = c.n_layers;
  p.B = kv->batch;
  p.Hkv = c.n_kv_heads;
  p.hd = m->hd;
  p.cap = kv->capacity;
  p.n = n_nodes;
  SPEC_CUDA(launch_tree_commit(p, static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

int spec_device_status(void* d_ws, void* stream, int32_t* out) {
  if (!d_ws || !out) return SPEC_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  SPEC_CUDA(cudaStreamSynchronize(st));
  int32_t v = 0;
  SPEC_CUDA(cudaMemcpy(&v, d_ws, 4, cudaMemcpyDeviceToHost));
  SPEC_CUDA(cudaMemset(d_ws, 0, 4));
  *out = v;
  if (v == 0) return SPEC_OK;
  return (v & SPEC_DEV_TIMEOUT) ? SPEC_ETIMEOUT : SPEC_EDEVICE;
}

int spec_wait_selftest(const uint32_t* d_counter, uint32_t target, double limit_ms, void* d_ws,
                       size_t ws_bytes, void* stream) {
  if (!d_counter || !d_ws || ws_bytes < 4 || !(limit_ms > 0.0) || limit_ms > 2000.0) return SPEC_EINVAL;
  if (reinterpret_cast<uintptr_t>(d_counter) % 4 || reinterpret_cast<uintptr_t>(d_ws) % 4) return SPEC_EINVAL;
  const auto ns = static_cast<unsigned long long>(limit_ms * 1e6);
  SPEC_CUDA(launch_wait_probe(d_counter, target, ns, static_cast<int32_t*>(d_ws),
                              static_cast<cudaStream_t>(stream)));
  return SPEC_OK;
}

int spec_timing_enable(spec_model* m, int enable) {
  if (!m) return SPEC_EINVAL;
  m->timing = enable != 0;
  return SPEC_OK;
}

int spec_timing_read(spec_model* m, double ms[3], int64_t launches[3], double bytes[3]) {
  if (!m || !ms || !launches || !bytes) return SPEC_EINVAL;
  for (int k = 0; k < 3; ++k) {
    ms[k] = 0;
    launches[k] = 0;
    bytes[k] = 0;
  }
  for (auto& t : m->pending) {
    SPEC_CUDA(cudaEventSynchronize(t.b));
    float x = 0.f;
    SPEC_CUDA(cudaEventElapsedTime(&x, t.a, t.b));
    ms[t.kind] += x;
    launches[t.kind] += 1;
    bytes[t.kind] += t.bytes;
    m->free_events.push_back(t.a);
    m->free_events.push_back(t.b);
  }
  m->pending.clear();
  return SPEC_OK;
}

}  // extern "C"
