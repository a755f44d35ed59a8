/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding
 * verification pass.
 *
 * The library runs one verification pass of lossless speculative decoding
 * on one GPU:
 *   1. spec_verify_forward: the target model's single forward over the
 *      gamma drafted tokens plus the bonus position (one weight read for all
 *      gamma+1 positions), producing fp32 logits for the gamma+1 positions.
 *   2. spec_accept: the acceptance rule -- temperature / top-p applied to the
 *      target rows, accept x_i iff u_i < min(1, p(x_i)/q(x_i)), resample from
 *      norm(max(0, p - q)) at the first rejection, or draw a bonus token from
 *      p at position gamma+1 when every draft survives.
 *   3. spec_kv_truncate: KV rollback by a length update (no memset).
 *
 * Sources (page title, section):
 *   [pigeon]   "Speculative decoding" (pigeon guide): How it works (steps 1-5),
 *              Why the output is exactly p, Speed, When it breaks.
 *   [lattice]  "Speculative decoding" (lattice-ai-eng inference notes): the
 *              rule, the worked example, the reference generation loop.
 *   [engine]   "Build a Speculative Decoding Engine to Cut LLM Latency by 3x":
 *              The Accept/Reject Mechanism, KV Cache Management for Dual
 *              Models, Rollback Protocol, Batch-Level Speculation,
 *              Speculation Depth Tuning and Tree Drafting.
 *   [aci]      "Speculative Decoding: Speeding Sequential Generation":
 *              Tree-Based Drafting, Constructing the Tree Attention Mask in
 *              Code, Expected Tokens per Verification Round: Chain vs. Tree.
 *   [kishorek] "Speculative Decoding: How to Make an LLM 3x Faster...":
 *              verifying a whole tree in one pass.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Every pointer named d_* is DEVICE memory owned by the caller (allocated
 *   with cudaMalloc / a framework allocator).  The library never allocates,
 *   frees or retains device memory.  `stream` is a cudaStream_t passed as
 *   void* (NULL = the legacy default stream).
 * - Calls are asynchronous on `stream`.  The return value reports argument
 *   validation and launch errors only (spec_status, 0 = OK, negative =
 *   error; nothing is enqueued on error).  Errors the device detects (a token
 *   id outside the vocabulary, a cache that would overflow its capacity,
 *   q(x) <= 0 for a drafted token, a bounded wait that ran out) set a status
 *   word in the workspace; kernels never trap.  Read and clear it with
 *   spec_device_status.
 * - Every call is usable inside CUDA stream capture (no host synchronisation,
 *   no allocation) except spec_device_status, which synchronises `stream`.
 * - Layouts are row-major.  bf16 is IEEE bfloat16 stored as uint16.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ----------------------------------------------------------------- status */
typedef enum {
  SPEC_OK = 0,
  SPEC_EINVAL = -1,   /* a NULL pointer, a negative size, T < 0, top_p outside (0,1] */
  SPEC_ESIZE = -2,    /* a size above a documented limit or a buffer too small */
  SPEC_ECUDA = -3,    /* a CUDA launch / runtime error (see spec_last_cuda_error) */
  SPEC_EDEVICE = -4,  /* returned by spec_device_status: the device set a status */
  SPEC_ETIMEOUT = -5, /* device status: a bounded wait gave up */
  SPEC_ENOTSUP = -6   /* the GPU is not sm_103 / the config is not supported */
} spec_status;

/* Device status bits (the value spec_device_status writes to *out). */
#define SPEC_DEV_BAD_TOKEN     0x1   /* an input / draft token id outside [0, V) */
#define SPEC_DEV_KV_OVERFLOW   0x2   /* len[b] + gamma + 1 > capacity, or truncate below 0 */
#define SPEC_DEV_Q_ZERO        0x4   /* q(x_i) <= 0 for a drafted token (treated as a rejection) */
#define SPEC_DEV_TIMEOUT       0x8   /* a bounded wait in a kernel gave up */
#define SPEC_DEV_BAD_NACC      0x10  /* truncate: n_accepted outside [0, gamma] */
#define SPEC_DEV_BAD_TREE      0x20  /* tree accept / commit: bad parents, path or n_accepted */
#define SPEC_DEV_EMPTY_MASK    0x40  /* mask_logits: a row's mask allows no token */
#define SPEC_DEV_BAD_PAGE      0x80  /* paged cache: a page id outside [0, n_pages) */

/* Text for a spec_status value (static storage). */
const char* spec_status_string(int status);
/* The CUDA error string of the last SPEC_ECUDA on this thread. */
const char* spec_last_cuda_error(void);

/* ------------------------------------------------------------------ model */
/* A Llama-style decoder ("8B-shaped": 32 layers, d 4096, 32 heads / 8 KV
 * heads of 128, SwiGLU ffn 14336, vocab 128256; "1B-shaped": 16, 2048,
 * 32/8 of 64, 8192, 32000).  Constraints: d_model = n_heads * head_dim,
 * n_heads % n_kv_heads == 0, head_dim in {64, 128}, d_model, n_heads*head_dim,
 * d_ffn multiples of 128 (d_ffn of 64 allowed), vocab >= 1.  n_layers = 0
 * gives an LM-head-only model (embedding + head). */
typedef struct {
  int n_layers;
  int d_model;
  int n_heads;
  int n_kv_heads;
  int d_ffn;
  int vocab;
  float rms_eps;     /* RMSNorm epsilon, e.g. 1e-5 */
  float rope_theta;  /* RoPE base, e.g. 500000 */
} spec_model_config;

typedef struct spec_model spec_model; /* opaque host-side handle */

/* Bytes of the device buffer that holds all weights of `cfg` (bf16 matrices
 * plus fp32 norm gains, each 256-byte aligned).  0 if cfg is invalid. */
size_t spec_model_weight_bytes(const spec_model_config* cfg);

/* Fill the caller's device buffer d_weights (>= spec_model_weight_bytes) with
 * seeded synthetic weights and return a handle in *out.
 * Every matrix element is bf16_round_nearest_even(0.02 * z) with z a standard
 * normal from Box-Muller (fp64) over Philox4x64-10 (Salmon et al. 2011):
 * logical tensor t, element e uses counter (e/4 + 1, t, 0, 0), key (seed, 0);
 * outputs (0,1) and (2,3) of a block are the Box-Muller pairs of elements
 * 4(e/4)+{0,1} and +{2,3}.  Tensor ids: 0 embedding [V][d], 1 LM head [V][d],
 * layer l: 2+7l+{0 W_q, 1 W_k, 2 W_v, 3 W_o, 4 W_gate, 5 W_up, 6 W_down}, all
 * [out][in].  RMSNorm gains are 1.0.  The generation is enqueued on `stream`.
 * Requires an sm_103 device (else SPEC_ENOTSUP).  The handle keeps the
 * pointer; the buffer must outlive the handle. */
int spec_model_create(const spec_model_config* cfg, uint64_t seed, void* d_weights,
                      size_t weight_bytes, void* stream, spec_model** out);

/* Free the host handle (never the caller's device buffer). NULL is a no-op. */
int spec_model_destroy(spec_model* model);

/* Where a logical weight lives, for tests that compare the generator with an
 * independent implementation.  which = 0..6 per layer as above (layer >= 0),
 * or layer = -1 with which 0 = embedding, 1 = LM head.  The physical storage
 * of W_gate/W_up is interleaved (blocks of 64 gate rows then 64 up rows), so
 * for them *row_stride_rows = 128 and *block_rows = 64 with *d_ptr at the
 * first row of the tensor's first block; for every other matrix the rows are
 * contiguous (*row_stride_rows = *block_rows = rows).  shape = {rows, cols}. */
int spec_model_tensor(const spec_model* model, int layer, int which, const void** d_ptr,
                      int64_t shape[2], int* block_rows, int* row_stride_rows);

/* ---------------------------------------------------------------- KV cache */
/* The target KV cache, caller-owned:
 *   k, v : bf16 [n_layers][batch][n_kv_heads][capacity][head_dim]
 *   len  : int32 [batch] device array, the valid length of each sequence.
 * A pass appends gamma+1 slots at len[b] .. len[b]+gamma and advances len;
 * spec_kv_truncate moves len back ([engine] KV Cache Management: "a pointer
 * update only"). */
typedef struct {
  void* k;
  void* v;
  int32_t* len;
  int batch;
  int capacity;
} spec_kv_cache;

/* Bytes of ONE of the k / v buffers. */
size_t spec_kv_bytes(const spec_model_config* cfg, int batch, int capacity);

/* ---------------------------------------------------------------- forward */
/* Workspace bytes for spec_verify_forward / spec_lm_head on `batch`
 * sequences of gamma+1 new tokens with a cache of `capacity` slots.  The
 * workspace also holds the device status word; one workspace serves one
 * stream at a time. */
size_t spec_workspace_bytes(const spec_model_config* cfg, int batch, int gamma, int capacity);

/* One verification forward ([pigeon] How it works, step 2; [lattice] the
 * single target call over the k drafted positions and the next-token slot).
 *   d_tokens  int32 [batch][gamma+1] = [t_last, x_1 .. x_gamma]: t_last is the
 *             previous pass's emitted token, not yet in the cache.
 *   kv        the cache; slots len[b] .. len[b]+gamma receive the new keys /
 *             values (RoPE positions len[b]+j) and len[b] += gamma+1.
 *   d_logits  fp32 [batch][gamma+1][vocab]; row j predicts the token after
 *             input j (rows 0..gamma-1 score x_1..x_gamma, row gamma is the
 *             bonus position).
 * Limits: batch*(gamma+1) <= 512, gamma+1 <= 128, capacity <= 32768 slots
 * (SPEC_ESIZE otherwise); prefill uses the same call
 * with gamma = prompt_len - 1 in chunks.  A token id outside [0, V) is read as
 * 0 and sets SPEC_DEV_BAD_TOKEN; a sequence whose len[b]+gamma+1 exceeds the
 * capacity sets SPEC_DEV_KV_OVERFLOW, its slots beyond the capacity are not
 * written and its logits are unspecified.
 * Schedule: a decode-shaped pass (batch*(gamma+1) <= 128, (gamma+1) x query
 * heads per KV head <= 64, <= 48 layers, d_model/128 a power of two) runs as
 * ONE persistent cooperative kernel (one CTA per SM, grid-wide barriers
 * between the pass's steps, weights streaming ahead across them); every
 * other pass (prefill chunks) runs as one kernel per step.  Setting the
 * environment variable SPEC_FORWARD_PERSISTENT=0 forces the per-step
 * schedule (read on every call).  Both give the same results up to fp32
 * summation order.  Attention of head dim 128 in decode shapes runs on the
 * tensor cores (S^T and O^T as tcgen05 MMAs) with its key blocks loaded by
 * TMA; SPEC_ATTENTION_TC=0 selects warp-level MMAs instead and
 * SPEC_ATTENTION_TMA=0 per-thread copies (both read on every call, for
 * comparison; the results agree up to fp32 summation order). */
int spec_verify_forward(const spec_model* model, const int32_t* d_tokens, int batch, int gamma,
                        const spec_kv_cache* kv, float* d_logits, void* d_ws, size_t ws_bytes,
                        void* stream);

/* LM head alone on given activations: d_logits[m][v] = sum_k hidden[m][k] *
 * W_head[v][k] (no norm).  d_hidden bf16 [rows][d_model], rows <= 512.
 * Workspace: spec_workspace_bytes(cfg, rows, 0, 1) suffices. */
int spec_lm_head(const spec_model* model, const uint16_t* d_hidden, int rows, float* d_logits,
                 void* d_ws, size_t ws_bytes, void* stream);

/* LM head for callers that cannot allocate device memory.  The pages have no
 * counterpart to this call; it exists for hosts that own every device
 * allocation and hand a plug-in only its input and output buffers, or that
 * run the call where no allocator may be used.  It computes exactly what
 * spec_lm_head computes (same kernel), but its scratch memory -- the stream-K
 * partial sums and tile counters spec_lm_head keeps in the caller's workspace
 * -- is a fixed 8.4 MiB device array inside the library, held by every GPU
 * that loads the library until the process exits.
 *   d_hidden  bf16 [rows][d_model], 16-byte aligned; rows <= 16 (else
 *             SPEC_ESIZE); a model vocabulary above 262144 gives SPEC_ESIZE.
 *   d_logits  fp32 [rows][vocab].
 * It allocates and frees nothing.  The first call on a device looks up the
 * array's device address on that device (the current device at the call)
 * and keeps it for the life of the process; make that first call before any
 * stream capture.  cudaDeviceReset() unloads the array with the rest of the
 * context, so after a reset of a device this entry point must not be called
 * on that device again in the same process (the kept address is stale).  All calls share the one
 * array and leave their contents in it: calls whose work overlaps on the GPU
 * (two streams, two host threads) race and produce wrong logits -- serialise
 * them.  The tile counters are cleared on `stream` at the start of every
 * call.  A device-side bounded-wait timeout is recorded in the library's own
 * scratch, not in a caller workspace, and is not reported: a caller of this
 * entry point has no way to learn that a call timed out (spec_lm_head, with
 * a workspace, reports it through spec_device_status). */
int spec_lm_head_noalloc(const spec_model* model, const uint16_t* d_hidden, int rows,
                         float* d_logits, void* stream);

/* ----------------------------------------------------------------- accept */
/* Workspace bytes for spec_accept / spec_draft_sample: the device status
 * word, a grid-barrier counter and the per-chunk partial statistics of the
 * accept grid (about 8.3 MiB for batch 64, gamma 7, vocab 128256).  The
 * workspace must be 16-byte aligned; one workspace serves one stream at a
 * time. */
size_t spec_accept_workspace_bytes(int batch, int gamma, int vocab);

/* The acceptance step ([pigeon] How it works, steps 3-5; [engine] The
 * Accept/Reject Mechanism); gamma + 1 <= 128 (else SPEC_ESIZE).  Batches of
 * up to 1024 rows (batch x (gamma+1)) run as one cooperative grid over
 * (sequence, row, vocabulary chunk) work units; larger batches run one CTA
 * per sequence (also forced by the environment variable SPEC_ACCEPT_GRID=0,
 * read per call).  Both give the same result up to fp32 summation order in
 * the softmax normaliser.
 *   d_target_logits fp32 [batch][gamma+1][vocab]
 *   d_draft_probs   fp32 [batch][gamma][vocab]: the distributions the drafts
 *                   were drawn from, after the same temperature / top-p
 *                   ([pigeon] When it breaks).  Unused when temperature = 0.
 *   d_draft_tokens  int32 [batch][gamma]
 *   d_uniforms      fp32 [batch][gamma+1] in [0,1): u_i (i < gamma) is the coin
 *                   of draft i, u_gamma drives the one residual / bonus draw.
 *                   Unused when temperature = 0.
 *   temperature     >= 0; 0 is greedy: accept while x_i = argmax (lowest id on
 *                   ties), emit the argmax at the first mismatch or the bonus.
 *   top_p           in (0, 1]; 1 disables the nucleus.  The nucleus keeps every
 *                   token whose probability is >= that of the token where the
 *                   descending cumulative mass first reaches top_p.  With
 *                   top_p < 1 the vocabulary is limited to 2^21 ids (else
 *                   SPEC_ESIZE; also for spec_draft_sample and spec_tree_accept).
 *   d_out_tokens    int32 [batch][gamma+1]: x_1..x_n, then the correction or
 *                   bonus token, then -1 padding.
 *   d_n_accepted    int32 [batch].
 * A draw is the inverse CDF in token-id order: the smallest id t with
 * cumulative weight > u * total.  A rejection whose residual mass is <= 1e-8
 * draws from p instead ([engine]'s numerical fallback). */
int spec_accept(const float* d_target_logits, const float* d_draft_probs,
                const int32_t* d_draft_tokens, const float* d_uniforms, int batch, int gamma,
                int vocab, float temperature, float top_p, int32_t* d_out_tokens,
                int32_t* d_n_accepted, void* d_ws, size_t ws_bytes, void* stream);

/* The draft side of "applied identically": for each of `rows` logits rows,
 * q = top-p(softmax(z / T)) written to d_probs (fp32 [rows][vocab], may be
 * NULL) and one token drawn from q with d_uniforms[r] by the same inverse CDF
 * (T = 0: the argmax; d_probs then one-hot).  Used to produce draft
 * distributions for spec_accept. */
int spec_draft_sample(const float* d_logits, int rows, int vocab, float temperature, float top_p,
                      const float* d_uniforms, float* d_probs, int32_t* d_tokens, void* d_ws,
                      size_t ws_bytes, void* stream);

/* ------------------------------------------------------ constrained rows */
/* Constrained generation ([engine] the question on JSON mode / grammar
 * constraints): the target and the draft apply the SAME allowed-token mask
 * before their probabilities are formed, the caller's constraint automaton
 * running in lockstep for both (a mask on one side only makes the acceptance
 * ratios wrong).  This call applies one mask per logits row in place:
 * d_logits[r][x] = -inf wherever bit (x % 32) of d_allowed[r][x / 32] is 0,
 * so the softmax gives those tokens probability 0 and the allowed tokens
 * keep their relative weights.  Apply it to the target rows before
 * spec_accept and to the draft rows before spec_draft_sample (or before
 * forming q): spec_accept, spec_draft_sample and spec_tree_accept handle
 * -inf logits.  Under greedy decoding the argmax is over the allowed tokens.
 *   d_logits   fp32 [rows][vocab], modified in place; rows <= 65535 (else
 *              SPEC_ESIZE).
 *   d_allowed  uint32 [rows][ceil(vocab / 32)]; bits at ids >= vocab are
 *              ignored.
 *   d_ws       any workspace of this library (its status word is used).
 * A row whose mask allows no token is left unchanged and sets
 * SPEC_DEV_EMPTY_MASK.  A drafted token outside the mask then has q(x) = 0
 * and is a rejection (SPEC_DEV_Q_ZERO). */
int spec_mask_logits(float* d_logits, const uint32_t* d_allowed, int rows, int vocab, void* d_ws,
                     void* stream);

/* --------------------------------------------------------------- rollback */
/* KV rollback after a pass that appended gamma+1 slots ([engine] Rollback
 * Protocol): len[b] -= gamma - n_accepted[b], so t_last and the accepted
 * drafts stay and the rejected drafts' slots are dropped.  Nothing is
 * cleared.  n_accepted outside [0, gamma] or a length that would go negative
 * leaves len[b] unchanged and sets a device status bit in d_ws (which may be
 * the forward's or the accept's workspace). */
int spec_kv_truncate(const spec_kv_cache* kv, const int32_t* d_n_accepted, int gamma, void* d_ws,
                     void* stream);

/* --------------------------------------------------------------- paged KV */
/* A paged target cache ([engine] Rollback Protocol: a paged KV cache with a
 * block pointer table; rollback updates the table and returns the pages of
 * rejected positions to the free list, nothing is zeroed).  Pages hold
 * SPEC_PAGE_SLOTS consecutive slots of one sequence for every KV head:
 *   k, v   bf16 [n_layers][n_pages][n_kv_heads][SPEC_PAGE_SLOTS][head_dim]
 *          (spec_paged_kv_bytes each), 16-byte aligned;
 *   len    int32 [batch] device, the valid length of each sequence;
 *   table  int32 [batch][max_pages] device: table[b][j] is the page holding
 *          slots j*SPEC_PAGE_SLOTS .. j*SPEC_PAGE_SLOTS + SPEC_PAGE_SLOTS-1
 *          of sequence b; only entries covering slots below len[b] + gamma
 *          + 1 are read by a pass.
 * The logical capacity of a sequence is max_pages * SPEC_PAGE_SLOTS <= 32768
 * slots.  A pass whose slots reach a page id outside [0, n_pages) sets
 * SPEC_DEV_BAD_PAGE and treats that sequence as overflowing (nothing written,
 * len not advanced). */
#define SPEC_PAGE_SLOTS 64
typedef struct {
  void* k;
  void* v;
  int32_t* len;
  const int32_t* table;
  int batch;
  int n_pages;
  int max_pages;
} spec_paged_kv_cache;

/* Bytes of the paged k array (and of v) for n_pages pages. */
size_t spec_paged_kv_bytes(const spec_model_config* cfg, int n_pages);

/* spec_verify_forward on a paged cache: the same pass (same kernels and
 * schedules, same results bit for bit as the contiguous cache holding the
 * same rows), every key / value row addressed through the page table.
 * Workspace: spec_workspace_bytes(cfg, batch, gamma, max_pages *
 * SPEC_PAGE_SLOTS). */
int spec_verify_forward_paged(const spec_model* model, const int32_t* d_tokens, int batch, int gamma,
                              const spec_paged_kv_cache* kv, float* d_logits, void* d_ws,
                              size_t ws_bytes, void* stream);

/* Rollback of a paged cache on the device: len[b] -= gamma - n_accepted[b]
 * (as spec_kv_truncate).  The pages wholly past the new length are then
 * returned by the host page pool (spec_page_pool_release). */
int spec_paged_kv_truncate(const spec_paged_kv_cache* kv, const int32_t* d_n_accepted, int gamma,
                           void* d_ws, void* stream);

/* Host page pool (no device access): a free list of n_pages page ids and a
 * host copy of the page table [batch][max_pages] (-1 = unmapped), to be
 * copied to the device table before a pass. */
typedef struct spec_page_pool spec_page_pool;
int spec_page_pool_create(int n_pages, int batch, int max_pages, spec_page_pool** out);
int spec_page_pool_destroy(spec_page_pool* pool);
/* Map every page sequence b needs for `slots` slots, taking pages from the
 * free list in order; SPEC_ESIZE (nothing taken) if the free list or
 * max_pages is too short. */
int spec_page_pool_reserve(spec_page_pool* pool, int b, int slots);
/* Return sequence b's pages past the first ceil(slots / SPEC_PAGE_SLOTS) to
 * the free list (after a rollback to `slots` slots; 0 frees the sequence). */
int spec_page_pool_release(spec_page_pool* pool, int b, int slots);
/* The host table [batch][max_pages] (valid until the pool is destroyed). */
const int32_t* spec_page_pool_table(const spec_page_pool* pool);
int spec_page_pool_free_pages(const spec_page_pool* pool);

/* ------------------------------------------------------------ draft trees */
/* Verification of a draft TREE instead of a chain ([aci] Tree-Based Drafting;
 * [engine] Speculation Depth Tuning and Tree Drafting): several candidates
 * per position, all scored by one target pass.  A tree of n_nodes <= 64
 * nodes (else SPEC_ESIZE) is given by parent pointers: node 0 is the root --
 * the previous pass's emitted token, not yet in the cache -- with parent -1,
 * and node i > 0 has a parent p(i) < i (parents are listed before their
 * children).  A chain of gamma drafts is the tree parents = [-1, 0, 1, ..,
 * gamma-1], and every tree call below then computes what the chain call
 * computes. */

/* Host-only (no device access): the attention mask and rotary positions of a
 * tree ([aci] Constructing the Tree Attention Mask in Code).  For each node i
 * out_anc[i] has bit j set iff node j is i itself or one of its ancestors
 * (node i sees the cached prefix and exactly those new slots) and
 * out_depth[i] is its depth (root 0), its rotary position offset.  Returns
 * SPEC_EINVAL for parents[0] != -1 or any parents[i] outside [0, i), and
 * SPEC_ESIZE for n_nodes > 64. */
int spec_tree_masks(const int32_t* parents, int n_nodes, uint64_t* out_anc, int32_t* out_depth);

/* One verification forward over a tree per sequence.
 *   d_tokens  int32 [batch][n_nodes] node tokens (node 0 the root).
 *   d_anc     uint64 [batch][n_nodes] ancestor masks (spec_tree_masks),
 *   d_depth   int32 [batch][n_nodes] depths; each sequence may have its own
 *             tree of the same node count.
 *   kv        node i's key / value goes to the flattened slot len[b] + i,
 *             rotated at position len[b] + depth(i); len[b] += n_nodes.
 *   d_logits  fp32 [batch][n_nodes][vocab]: row i scores the token after
 *             node i (its children's target distribution).
 * Workspace, limits, schedules and device errors as spec_verify_forward with
 * gamma = n_nodes - 1 (the persistent schedule applies when n_nodes x query
 * heads per KV head <= 64).  The masks and depths are not checked on the
 * device: a mask bit at or above n_nodes is ignored, and a node whose mask
 * lacks its own bit does not see itself. */
int spec_verify_forward_tree(const spec_model* model, const int32_t* d_tokens,
                             const uint64_t* d_anc, const int32_t* d_depth, int batch,
                             int n_nodes, const spec_kv_cache* kv, float* d_logits, void* d_ws,
                             size_t ws_bytes, void* stream);

/* Workspace bytes for spec_tree_accept: the status word (256 bytes; the walk
 * keeps each node's residual distribution in closed form, as a coefficient of
 * q and a normaliser, so it needs no vocabulary-sized scratch). */
size_t spec_tree_accept_workspace_bytes(int batch, int vocab);

/* The acceptance walk over each sequence's tree ([aci] Tree-Based Drafting:
 * the accept/reject test applied per node; [kishorek] accept the longest
 * valid root-to-node path), one CTA per sequence.  Starting at the root, at
 * the current node c with target distribution p' (softmax(z_c / T) after
 * top-p) the children are tried in index order: child j (token x_j) is
 * accepted iff u_j < min(1, p'(x_j) / q_c(x_j)); after each rejected child p'
 * becomes norm(max(0, p' - q_c)) (unchanged when that mass is <= 1e-8).  The
 * first accepted child becomes the current node; when no child is accepted
 * (or c is a leaf) one token is drawn from p' with u_0 by the inverse CDF in
 * id order and the walk ends.  Siblings are independent draws from their
 * parent's q, so the emitted tokens follow the target exactly as in the
 * chain rule, which is the case of one child per node.
 *   d_target_logits fp32 [batch][n_nodes][vocab] (spec_verify_forward_tree)
 *   d_draft_probs   fp32 [batch][n_nodes][vocab]: row c is the distribution
 *                   node c's children were drawn from (after the same T /
 *                   top-p); rows of leaves are not read.  Unused at T = 0.
 *   d_node_tokens   int32 [batch][n_nodes]; d_parents int32 [batch][n_nodes].
 *   d_uniforms      fp32 [batch][n_nodes] in [0,1): u_j (j >= 1) is the coin
 *                   of node j, u_0 drives the final draw.  Unused at T = 0.
 *   temperature     >= 0; 0 is greedy: move to the first child whose token is
 *                   the argmax (lowest id on ties), else emit the argmax.
 *   d_out_tokens    int32 [batch][n_nodes]: the accepted nodes' tokens, the
 *                   emitted token, then -1.
 *   d_out_path      int32 [batch][n_nodes]: the accepted nodes (root
 *                   excluded) in depth order, then -1.
 *   d_n_accepted    int32 [batch]: accepted nodes m (the round emits m + 1).
 * A sequence whose parents are not a valid tree sets SPEC_DEV_BAD_TREE and
 * gets m = 0 and no tokens (-1); a child token outside [0, V) or with
 * q_c(x) <= 0 is a rejection and sets SPEC_DEV_BAD_TOKEN / SPEC_DEV_Q_ZERO. */
int spec_tree_accept(const float* d_target_logits, const float* d_draft_probs,
                     const int32_t* d_node_tokens, const int32_t* d_parents,
                     const float* d_uniforms, int batch, int n_nodes, int vocab, float temperature,
                     float top_p, int32_t* d_out_tokens, int32_t* d_out_path,
                     int32_t* d_n_accepted, void* d_ws, size_t ws_bytes, void* stream);

/* The tree round's KV commit, run after spec_tree_accept (the tree
 * counterpart of spec_kv_truncate; [engine] Rollback Protocol): with
 * L0 = len[b] - n_nodes, the accepted path's keys / values move from the
 * flattened slots L0 + path[d-1] to L0 + d (d = 1 .. m, every layer and KV
 * head), and len[b] = L0 + 1 + m, so the root and the accepted path are
 * contiguous and the other nodes' slots are dropped.
 *   d_path, d_n_accepted  spec_tree_accept's outputs.
 *   kv->k, kv->v          16-byte aligned.
 * A path that is not strictly increasing within [1, n_nodes) or an m outside
 * [0, n_nodes) leaves the sequence unchanged and sets SPEC_DEV_BAD_TREE; a
 * length below n_nodes or above the capacity sets SPEC_DEV_KV_OVERFLOW.
 * d_ws is any workspace of this library (its status word is used). */
int spec_kv_tree_commit(const spec_model* model, const spec_kv_cache* kv, const int32_t* d_path,
                        const int32_t* d_n_accepted, int n_nodes, void* d_ws, void* stream);

/* ---------------------------------------------------------- dynamic gamma */
/* The speculation-depth controller ([engine] Speculation Depth Tuning and
 * Tree Drafting; Dynamic Gamma Controller).  Host only (no device access,
 * no stream): after each pass the caller records, per slot, the depth it
 * used and its n_accepted (spec_accept's output, copied to the host); each
 * slot keeps its last `window` passes and, once `min_records` are in,
 * chooses the depth in [gamma_min, gamma_max] that maximises expected
 * tokens per millisecond,
 *     E(alpha, g) / (g * draft_ms_per_token + target_ms_per_pass),
 *     E(alpha, g) = (1 - alpha^(g+1)) / (1 - alpha)   (g + 1 at alpha >= 1),
 * with alpha = accepted drafts / drafted tokens over the window
 * (alpha_prior while the window is empty).  Ties go to the smaller depth.
 * A slot is a sequence, or a group of sequences the caller pools (e.g. one
 * content type, [engine] the multi-tenant question).  The page's setting:
 * depths 2..8 starting at 4, window 20, decisions after 5 passes, 2.0 ms
 * per draft token, 20.0 ms per target pass (calibrate both), prior 0.80.
 * Not thread-safe per controller. */
typedef struct spec_gamma_ctl spec_gamma_ctl;

int spec_gamma_ctl_create(int slots, int gamma_min, int gamma_max, int gamma_init, int window,
                          int min_records, double draft_ms_per_token, double target_ms_per_pass,
                          double alpha_prior, spec_gamma_ctl** out);
int spec_gamma_ctl_destroy(spec_gamma_ctl* ctl);
/* Forget slot's passes (a new sequence in the slot); its depth returns to
 * gamma_init. */
int spec_gamma_ctl_reset(spec_gamma_ctl* ctl, int slot);
/* Record n passes: h_slot[i] used depth h_gamma_used[i] and accepted
 * h_n_accepted[i] drafts (host arrays of n entries; a slot may appear more
 * than once, in order).  h_gamma_next[i] receives that slot's depth for its
 * next pass.  An entry with a slot outside [0, slots) or n_accepted outside
 * [0, gamma_used] returns SPEC_EINVAL and records nothing. */
int spec_gamma_ctl_step(spec_gamma_ctl* ctl, int n, const int32_t* h_slot,
                        const int32_t* h_gamma_used, const int32_t* h_n_accepted,
                        int32_t* h_gamma_next);
/* A slot's current alpha estimate, depth and number of passes in its window
 * (any output pointer may be NULL). */
int spec_gamma_ctl_state(const spec_gamma_ctl* ctl, int slot, double* out_alpha,
                         int32_t* out_gamma, int32_t* out_records);
/* The depth rule alone, for a given alpha (clamped to 1). */
int spec_gamma_optimal(double alpha, int gamma_min, int gamma_max, double draft_ms_per_token,
                       double target_ms_per_pass, int32_t* out_gamma);

/* ----------------------------------------------------------------- status */
/* Synchronise `stream`, read the device status word of workspace d_ws into
 * *out (a SPEC_DEV_* bit set), clear it, and return SPEC_OK if it was 0,
 * SPEC_ETIMEOUT if the timeout bit was set, else SPEC_EDEVICE. */
int spec_device_status(void* d_ws, void* stream, int32_t* out);

/* Self-test of the bounded waits.  One thread of one CTA waits until the
 * uint32 counter at d_counter (device, 4-byte aligned, caller-owned) is >=
 * target, with the wait function every grid barrier of the persistent
 * forward uses, but bounded by limit_ms (0 < limit_ms <= 2000) instead of the
 * barrier's 2 s.  If the counter does not reach target in time the wait
 * gives up, sets SPEC_DEV_TIMEOUT in the status word of workspace d_ws (at
 * least 4 bytes, 4-byte aligned; any workspace of this library) and the
 * kernel returns: spec_device_status then reports SPEC_ETIMEOUT and the CUDA
 * context stays usable.  Errors: SPEC_EINVAL for NULL or misaligned pointers,
 * ws_bytes < 4 or limit_ms outside (0, 2000]; SPEC_ECUDA on a launch error. */
int spec_wait_selftest(const uint32_t* d_counter, uint32_t target, double limit_ms, void* d_ws,
                       size_t ws_bytes, void* stream);

/* ------------------------------------------------------------ diagnostics */
/* Per-kernel-kind timing for benchmarks.  When enabled on a model, every
 * subsequent forward records CUDA events around each launch of the GEMM,
 * attention and persistent forward kernels (this serialises the launches it
 * brackets).  spec_timing_read synchronises and returns, per kind (0 = GEMM,
 * 1 = attention, 2 = persistent forward), the summed milliseconds, launch
 * count and weight bytes streamed (kinds 0 and 2; 0 for kind 1) since the
 * last read. */
int spec_timing_enable(spec_model* model, int enable);
int spec_timing_read(spec_model* model, double ms[3], int64_t launches[3], double bytes[3]);

#ifdef __cplusplus
}
#endif
#endif /* SPEC_VERIFY_H */
