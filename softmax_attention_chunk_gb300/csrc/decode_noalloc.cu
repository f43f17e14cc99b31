// Decode step that needs no caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they decode: code that runs
// inside another framework's memory pool with no allocator handle, plugins that may only
// touch the buffers they are given, or serving loops that forbid any allocation after start-up.
// For them this entry point keeps the per-split softmax partials of the decode step in a
// fixed array compiled into the library instead of a workspace argument.
//
// The array is a file-scope __device__ variable: each GPU that loads the library holds it
// (16 MiB) until the process exits.  Host code only sees a host-side stand-in for it, so its
// device address is looked up once per device with cudaGetSymbolAddress (on the first call
// made with that device current) and cached.  Every call on a device shares the one array.
#include "../../include/path_attn.h"
#include "internal.h"

#include <math.h>
#include <stdint.h>

#include <mutex>

using namespace pathattn;

namespace {

constexpr size_t kScratchBytes = (size_t)16 << 20;
static_assert((size_t)PATH_DECODE_NOALLOC_MAX_HEADS * kDecodeMaxSplits * (kHeadDim + 2) * sizeof(float) <=
                  kScratchBytes,
              "the no-allocation decode scratch must hold the partials of the largest allowed batch*heads");

static __device__ __align__(256) float g_decode_scratch[kScratchBytes / sizeof(float)];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_decode_scratch on the current device (looked up once per device).
int scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return PATH_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return PATH_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || !p) return PATH_ERR_CUDA;
    g_scratch_ptr[dev] = p;
  }
  *out = g_scratch_ptr[dev];
  return PATH_OK;
}

bool aligned16(const void* p) { return p && (reinterpret_cast<uintptr_t>(p) % 16) == 0; }

}  // namespace

extern "C" __attribute__((visibility("default"))) int path_decode_step_noalloc(
    const path_decode_desc_t* d, void* k_cache, void* v_cache, int t, const void* q_t,
    const void* k_t, const void* v_t, const void* w_t, const float* beta_t, void* o_t,
    void* stream) {
  // Same argument rules as path_decode_step, checked before any CUDA call.
  if (!d) return PATH_ERR_INVALID_ARG;
  if (d->batch <= 0 || d->heads <= 0 || d->capacity <= 0 || d->head_dim <= 0) return PATH_ERR_INVALID_ARG;
  if (d->cache_dtype != PATH_BF16 && d->cache_dtype != PATH_FP32) return PATH_ERR_INVALID_ARG;
  if (!isfinite(d->scale)) return PATH_ERR_INVALID_ARG;
  if (d->head_dim != kHeadDim) return PATH_ERR_UNSUPPORTED;
  if (t < 0) return PATH_ERR_INVALID_ARG;
  if ((long long)t + 1 > d->capacity) return PATH_ERR_CAPACITY;
  const void* ptrs[] = {k_cache, v_cache, q_t, k_t, v_t, w_t, beta_t, o_t};
  for (const void* p : ptrs)
    if (!aligned16(p)) return PATH_ERR_INVALID_ARG;
  // The built-in scratch holds the partials of at most PATH_DECODE_NOALLOC_MAX_HEADS heads.
  if ((long long)d->batch * d->heads > PATH_DECODE_NOALLOC_MAX_HEADS) return PATH_ERR_WORKSPACE;

  void* scratch = nullptr;
  const int rc = scratch_address(&scratch);
  if (rc != PATH_OK) return rc;
  // Every split writes its whole partial slot before the combine kernel reads it, so the
  // array needs no clearing between calls.
  return path_decode_step(d, k_cache, v_cache, t, q_t, k_t, v_t, w_t, beta_t, o_t, scratch,
                          kScratchBytes, stream);
}
