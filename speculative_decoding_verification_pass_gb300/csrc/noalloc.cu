// LM head whose scratch memory belongs to the library.
//
// Some callers cannot allocate device memory at all: a plugin running inside
// a host framework that owns every device allocation and hands out only
// input/output buffers, or code that must not call an allocator at the point
// where it runs.  spec_lm_head needs a caller-provided workspace for its
// stream-K partial sums and tile counters; this variant keeps that scratch in
// one file-scope device array instead, so the caller passes only the
// activations and the logits buffer.
//
// The array is a fixed 8.4 MiB of device memory that every GPU loading the
// library keeps until the process exits.  Every call shares it (and keeps
// the previous call's contents), so calls that overlap on the GPU -- on two
// streams at once, or on two threads -- race and give wrong results.
#include <mutex>

#include "internal.h"

namespace {

constexpr int kMaxRows = 16;             // token rows per call (one 16-row tile)
constexpr int kMaxVocab = 262144;        // output rows: 2048 tiles of 128
constexpr int kMaxGridCtas = 512;        // stream-K grid cap of the GEMM launcher
constexpr size_t kStatusBytes = 256;
constexpr size_t kCounterBytes = static_cast<size_t>(kMaxVocab / 128) * 4;
constexpr size_t kPartialBytes = static_cast<size_t>(kMaxGridCtas) * 2 * kMaxRows * 128 * 4;
constexpr size_t kScratchBytes = kStatusBytes + kCounterBytes + kPartialBytes;

static __device__ __align__(256) unsigned char g_lm_head_scratch[kScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The symbol's
// name is only a host-side handle; the address comes from the runtime, once
// per device, and is cached.
int scratch_for_current_device(unsigned char** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return SPEC_ECUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_scratch[dev]) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_lm_head_scratch);
    if (e != cudaSuccess || !p) return SPEC_ECUDA;
    g_scratch[dev] = p;
  }
  *out = static_cast<unsigned char*>(g_scratch[dev]);
  return SPEC_OK;
}

}  // namespace

extern "C" int spec_lm_head_noalloc(const spec_model* model, const uint16_t* d_hidden, int rows,
                                    float* d_logits, void* stream) {
  if (!model || !d_hidden || !d_logits || rows < 0) return SPEC_EINVAL;
  if (rows > kMaxRows) return SPEC_ESIZE;
  if (rows == 0) return SPEC_OK;
  unsigned char* s = nullptr;
  const int r = scratch_for_current_device(&s);
  if (r != SPEC_OK) return r;
  int32_t* status = reinterpret_cast<int32_t*>(s);
  int32_t* counters = reinterpret_cast<int32_t*>(s + kStatusBytes);
  float* partials = reinterpret_cast<float*>(s + kStatusBytes + kCounterBytes);
  // The tile counters must start at zero; the kernel leaves them at zero,
  // but a call that did not finish may not have, so clear them every time.
  if (cudaMemsetAsync(counters, 0, kCounterBytes, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return SPEC_ECUDA;
  // (the vocabulary and grid limits are checked against the model inside)
  return spec_internal_lm_head(model, d_hidden, rows, d_logits, partials, counters, status,
                               kMaxVocab, kMaxGridCtas, stream);
}
