// Host-side declarations shared by the C-ABI translation unit and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "spec_verify.h"

namespace spec {

// One value per device, made once per device by the first call with that
// device current.  CUDA keeps function attributes (e.g. the dynamic shared
// memory limit) and occupancy per device, so a process that drives several
// GPUs needs every such set-up on each of them.  Thread-safe.
constexpr int kMaxDevices = 64;
template <typename T>
class PerDevice {
 public:
  // false when the current device cannot be read or is out of range
  template <typename F>
  bool get(F make, T* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return false;
    std::call_once(once_[dev], [&] { val_[dev] = make(); });
    *out = val_[dev];
    return true;
  }

 private:
  std::once_flag once_[kMaxDevices];
  T val_[kMaxDevices] = {};
};

// ------------------------------------------------------------------ GEMM
// Y[m][n] = sum_k X[m][k] * W[n][k]; W bf16 [N][K] (TMA map tmW), X bf16
// [rows][K] (TMA map tmX); N-tiles of 128 rows, K-chunks of 64.
enum EpiKind { EPI_STORE = 0, EPI_RESID = 1, EPI_QKV = 2, EPI_SWIGLU = 3 };

struct GemmParams {
  int N, K;        // weight rows (output features) and reduction length
  int M;           // valid token rows in total (rows >= M are padding)
  int tok0;        // first token row handled by this launch
  int ntok;        // token tile (multiple of 16, <= 256)
  int split;       // 0: bf16 X only; 1: [X_hi ; X_lo] stacked in N (2*ntok <= 256);
                   // 2: X_lo accumulated by a second MMA
  int ksub;        // 64-wide K sub-tiles per stage (1 or 2)
  int kc;          // K / (64 * ksub): K-chunks per tile
  int n_tiles;     // ceil(N / 128)
  long long units; // n_tiles * kc
  int stages;      // smem ring depth
  int epi;         // EpiKind
  // RMSNorm of the consumer: rs[m] = rsqrt(sum_t ssq_in[t][m] / d + eps)
  const float* ssq_in;  // nullptr: no norm scale
  int ssq_tiles;
  int ssq_ld;
  float inv_d, eps;
  // EPI_STORE
  float* out;
  int ldo;
  // EPI_RESID: h[m][f] += y; hb[m][f] = bf16(h * g_next[f]); ssq_out[tile][m]
  float* h;
  uint16_t* hb;
  uint16_t* hb_lo;        // bf16(x - bf16(x)) or nullptr
  const float* g_next;
  float* ssq_out;
  int d;
  // EPI_QKV
  uint16_t* q;           // [M][H*hd]
  uint16_t* q_lo;        // bf16 residual of q, or nullptr
  uint16_t* kcache;      // this layer's K base [B][Hkv][cap][hd]
  uint16_t* vcache;
  const int32_t* pos_base;
  const int32_t* seq_ok;  // per sequence: 1 if its slots fit in the cache
  const float2* rope;     // [hd/2] frequency (hi, lo)
  const int32_t* depth;   // [M] draft-tree node depths (position = base + depth), or nullptr
  const int32_t* kv_table;  // [B][kv_max_pages] page table of a paged cache, or nullptr
  int kv_max_pages, kv_n_pages;
  int n_per_seq, H, Hkv, hd, cap;
  // EPI_SWIGLU: rows 0-63 of a tile are gate features, 64-127 up features
  uint16_t* act;  // [M][ffn]
  uint16_t* act_lo;
  int ffn;
  // stream-K workspace
  float* partials;    // [grid][2][ntok][128]
  int32_t* counters;  // [n_tiles], zero on entry, left zero
  int32_t* status;
};

// Shared memory a launch needs for `stages` ring stages.
// `rows_b` = token rows of the B operand per stage (ntok << split).
size_t gemm_smem_bytes(int rows_b, int stages, int ksub);
int gemm_max_stages(int rows_b, size_t smem_budget, int ksub);
cudaError_t launch_gemm(const CUtensorMap* tmW, const CUtensorMap* tmX, const CUtensorMap* tmXlo,
                        const GemmParams& p, int grid, cudaStream_t stream, bool pdl);

// -------------------------------------------------------------- attention
struct AttnParams {
  const uint16_t* q;      // [M][H*hd] bf16 (RoPE applied)
  const uint16_t* q_lo;   // bf16 residual of q, or nullptr
  const uint16_t* kcache; // this layer's [B][Hkv][cap][hd]
  const uint16_t* vcache;
  uint16_t* o;            // [M][H*hd] bf16
  uint16_t* o_lo;         // bf16 residual of o, or nullptr
  const int32_t* pos_base;
  const uint64_t* anc;    // [B][n] draft-tree ancestor masks, or nullptr (chain)
  const int32_t* kv_table;  // [B][kv_max_pages] page table of a paged cache, or nullptr
  int kv_max_pages, kv_n_pages;
  float* part_o;          // [B][Hkv][splits][R][hd]
  float* part_ml;         // [B][Hkv][splits][R][2]
  int32_t* counters;      // [B*Hkv], zero on entry, left zero
  int32_t* status;
  int B, n, H, Hkv, hd, cap, splits, R;
  int cluster;            // > 0: decode path, clusters of this many CTAs (R <= 32)
  float scale_log2;       // log2(e) / sqrt(hd)
};
constexpr int kAttnChunk = 128;      // keys per CTA
constexpr int kAttnMaxChunks = 256;  // capacity <= 32768 slots
cudaError_t launch_attention(const AttnParams& p, cudaStream_t stream, bool pdl);
// Cluster size of the decode attention path for this cache capacity (0: the
// cache slice per CTA would not fit in smem_limit, or no cluster can be placed).
int attention_cluster_size(int hd, int cap, size_t smem_limit);

// --------------------------------------------------- persistent decode forward
constexpr int kMkMaxLayers = 48;
constexpr int kMkAttRows = 64;  // query rows per (sequence, KV head) of the persistent forward
constexpr int kMkMaxAcc = 4;    // TMEM accumulator buffers of the persistent forward, at most
struct MkParams {
  CUtensorMap xmap[6];                    // hb, hb_lo, o, o_lo, act, act_lo (box rows = ntok)
  CUtensorMap wmap[4 * kMkMaxLayers + 1]; // per layer W_qkv, W_o, W_gu, W_d; then the LM head
  CUtensorMap kvmap[2];                   // K, V caches of all layers as [rows][hd], boxes [64][128 | 64 rows]
  CUtensorMap qmap[2];                    // q hi, lo as [M][H][hd], boxes [64][G][32 / G]
  int L, d, H, Hkv, hd, ffn, V, qkv_rows;
  int B, n, M, ntok, cap, stages, ssq_ld;
  int att_nch;                            // the most key chunks per (sequence, KV head): the partials' slots
  int att_tc;                             // attention on the tensor cores (forward_att_tc)
  int att_tma;                            // ... with its q, K and V blocks as TMA loads (kvmap, qmap)
  int nacc;                               // TMEM accumulator buffers, 2..kMkMaxAcc (forward_acc_buffers)
  float eps, inv_d, scale_log2;
  const uint16_t* embed;
  const float2* rope;
  const float* gfinal;
  const float* g_attn0;                   // layer 0's gains; layer l is + l * layer_stride bytes
  const float* g_mlp0;
  long long layer_stride;
  uint16_t* kc;                           // KV cache base; layer l is + l * layer_kv elements
  uint16_t* vc;
  long long layer_kv;
  const int32_t* kv_table;                // [B][kv_max_pages] page table, or nullptr (contiguous)
  int kv_max_pages, kv_n_pages;
  int32_t* len;
  const int32_t* tokens;
  float* logits;
  float* h;
  uint16_t *hb, *hb_lo, *q, *q_lo, *o, *o_lo, *act, *act_lo;
  float* ssq;
  float* partials;                        // stream-K words: [grid][2][ntok][128] x 8 bytes
  int32_t* counters;
  unsigned* bar;                          // grid-barrier arrivals, zero at launch
  unsigned* epoch;                        // launch epoch (advanced by every launch; never cleared)
  int32_t* status;
  int32_t* pos_base;
  int32_t* seq_ok;
  const uint64_t* anc;                    // [B][n] draft-tree ancestor masks, or nullptr (chain)
  const int32_t* depth;                   // [B][n] draft-tree node depths, or nullptr (chain)
  float* att_o;                           // [B][Hkv][att_nch][kMkAttRows][hd] chunk partials
  float* att_ml;                          // [B][Hkv][att_nch][kMkAttRows][2] (max, sum)
};
size_t forward_smem_bytes(int ntok, int stages, int hd);
int forward_max_stages(int ntok, int hd, size_t budget);
int forward_ctas_per_sm(int ntok, int stages, int hd);
bool forward_att_tc(int ntok, int stages, int hd);
int forward_acc_buffers(int ntok, bool att_tc);
// One layer's tensor-core attention (head dim 128, at most kMkAttRows query
// rows per KV head, at most 128 sequences) as two launches: the persistent
// kernel's attention phase (grid CTAs, one per SM), then its merge into o /
// o_lo (3 x grid smaller CTAs).  P as for the persistent kernel's attention,
// with stages = kStepAttStages.
constexpr int kStepAttStages = 3;
cudaError_t launch_attention_tc(const MkParams& P, int l, int grid, cudaStream_t stream);
cudaError_t launch_forward(const MkParams& P, int grid, int hd, cudaStream_t stream);

// ------------------------------------------------------------ small kernels
struct EmbedParams {
  const int32_t* tokens;  // [B][n]
  const uint16_t* embed;  // [V][d]
  const float* g0;        // gain of the first consumer norm
  float* h;
  uint16_t* hb;
  uint16_t* hb_lo;
  float* ssq;             // [d/128][ld]
  int ssq_ld;
  int32_t* len;           // [B] cache lengths (advanced by n)
  int32_t* pos_base;      // [B] out: length before this pass
  int32_t* seq_ok;        // [B] out
  int32_t* counters;      // zeroed here
  int n_counters;
  int32_t* status;
  const int32_t* kv_table;  // page table to validate, or nullptr
  int kv_max_pages, kv_n_pages;
  int B, n, d, V, cap;
};
cudaError_t launch_embed(const EmbedParams& p, cudaStream_t stream, bool pdl);

cudaError_t launch_init_weights(uint16_t* dst, long long rows, long long cols, int tid,
                                uint64_t seed, int block_rows, int row_stride_rows,
                                cudaStream_t stream);
cudaError_t launch_fill_f32(float* dst, long long n, float v, cudaStream_t stream);
cudaError_t launch_rope_table(float2* dst, int hd, double theta, cudaStream_t stream);
cudaError_t launch_wait_probe(const unsigned* ctr, unsigned target, unsigned long long limit_ns,
                              int32_t* status, cudaStream_t stream);

// ------------------------------------------------------------------ accept
constexpr int kAcceptMaxChunk = 4096;  // vocabulary ids per accept work unit
constexpr int kAcceptMaxRows = 128;    // gamma + 1 per sequence
constexpr int kAcceptGridRows = 1024;  // batch * (gamma + 1) of the grid schedule
constexpr int kNucleusMaxVocab = 1 << 21;  // vocabulary limit of top_p < 1
struct AcceptParams {
  const float* logits;   // [B][gamma+1][V]
  const float* q;        // [B][gamma][V]
  const int32_t* draft;  // [B][gamma]
  const float* u;        // [B][gamma+1]
  int32_t* out;          // [B][gamma+1]
  int32_t* n_acc;        // [B]
  int32_t* status;
  unsigned* bar;                 // grid-barrier arrivals, zeroed before launch
  float2* part_ms;               // [B][n][S] chunk (max, sum) or (value, id)
  unsigned long long* tot40;     // [B][n] nucleus mass (2^-40 fixed point)
  unsigned long long* hist;      // [B][n][4][256] radix-select histograms
  unsigned long long* sel;       // [B][n][4][2] (prefix, mass above) per digit
  unsigned long long* part_tot;  // [B][S][2] draw-weight sums (residual, p)
  int* part_last;                // [B][S][2] last id with positive weight
  int B, gamma, V, S, C;         // S chunks of C ids (C <= kAcceptMaxChunk)
  int S1, SL;                    // grid schedule: units per row of the chunk statistics
                                 // and of the nucleus select (<= S; set by the launcher)
  int grid;                      // 1: the cooperative grid schedule when it fits
  float T, top_p;
};
cudaError_t launch_accept(const AcceptParams& p, cudaStream_t stream);

struct SampleParams {
  const float* logits;  // [R][V]
  const float* u;       // [R]
  float* probs;         // [R][V] or nullptr
  int32_t* tokens;      // [R]
  int32_t* status;
  int R, V;
  float T, top_p;
};
cudaError_t launch_sample(const SampleParams& p, cudaStream_t stream);

// LM head with explicit stream-K scratch sized for rows <= 16: partials >=
// max_grid x 2 x 16 x 128 floats, counters >= ceil(vocab/128) ints (zero on
// entry).  SPEC_ESIZE when the model's vocabulary exceeds max_vocab or the
// launcher's grid cap exceeds max_grid.
}  // namespace spec
extern "C" int spec_internal_lm_head(const spec_model* m, const uint16_t* d_hidden, int rows,
                                     float* d_logits, float* partials, int32_t* counters,
                                     int32_t* status, int max_vocab, int max_grid, void* stream);
namespace spec {

cudaError_t launch_truncate(int32_t* len, const int32_t* n_acc, int B, int gamma, int32_t* status,
                            cudaStream_t stream, bool pdl);

// ------------------------------------------------------------- draft trees
constexpr int kTreeMaxNodes = 64;  // one 64-bit ancestor mask per node
struct TreeAcceptParams {
  const float* logits;     // [B][n][V] target logits per node
  const float* q;          // [B][n][V] each node's draft distribution (its children's)
  const int32_t* tokens;   // [B][n] node tokens (node 0: the root)
  const int32_t* parents;  // [B][n] parent index, -1 for node 0
  const float* u;          // [B][n]: u[c] coin of child c, u[0] the final draw
  int32_t* out;            // [B][n] accepted tokens, then the emitted token, -1 padding
  int32_t* path;           // [B][n] accepted nodes in depth order, -1 padding
  int32_t* n_acc;          // [B]
  int32_t* status;
  int B, n, V;
  float T, top_p;
};
cudaError_t launch_tree_accept(const TreeAcceptParams& p, cudaStream_t stream);

// logits[r][x] = -inf where bit x % 32 of allowed[r][x / 32] is clear
cudaError_t launch_mask_logits(float* logits, const uint32_t* allowed, int rows, int V, int32_t* status,
                               cudaStream_t stream);

struct TreeCommitParams {
  uint16_t* k;             // [L][B][Hkv][cap][hd]
  uint16_t* v;
  int32_t* len;            // [B], len = L0 + n on entry
  const int32_t* path;     // [B][n]
  const int32_t* n_acc;    // [B]
  int32_t* status;
  int L, B, Hkv, hd, cap, n;
};
cudaError_t launch_tree_commit(const TreeCommitParams& p, cudaStream_t stream);

}  // namespace spec
