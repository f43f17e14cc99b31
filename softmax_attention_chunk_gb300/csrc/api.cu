// C ABI of the PaTH attention library: argument validation, workspace layout and kernel
// dispatch.  Declared in include/path_attn.h.
#include "../../include/path_attn.h"
#include "internal.h"

#include <math.h>
#include <stdint.h>
#include <stdlib.h>

using namespace pathattn;

namespace {

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// bf16 at head dim 64 with the default (or 64) chunk runs the tcgen05 kernels; fp32 and chunk 32
// run the SIMT kernels.
bool uses_tensor_cores(const path_attn_desc_t* d, int /*for_backward*/) {
  return d->dtype == PATH_BF16 && d->head_dim == kHeadDim && (d->chunk == 0 || d->chunk == 64);
}
// bf16 at head dim 128 with the default (or 64) chunk: the forward runs the head-dim-128 tcgen05
// kernels (64-row chunks, 128-row query tiles); the backward runs the SIMT kernels (32-row chunks).
bool uses_tc128(const path_attn_desc_t* d, int for_backward) {
  return !for_backward && d->dtype == PATH_BF16 && d->head_dim == kHeadDimWide && (d->chunk == 0 || d->chunk == 64);
}

// Validates a descriptor; on success fills g for the requested pass.
int check_desc(const path_attn_desc_t* d, int for_backward, Geom* g) {
  if (!d) return PATH_ERR_INVALID_ARG;
  if (d->batch <= 0 || d->heads <= 0 || d->seqlen <= 0 || d->head_dim <= 0) return PATH_ERR_INVALID_ARG;
  if (d->dtype != PATH_BF16 && d->dtype != PATH_FP32) return PATH_ERR_INVALID_ARG;
  if (!isfinite(d->scale)) return PATH_ERR_INVALID_ARG;
  if (d->head_dim != kHeadDim && d->head_dim != kHeadDimWide) return PATH_ERR_UNSUPPORTED;
  const long long BH = (long long)d->batch * d->heads;
  if (BH > 65535) return PATH_ERR_UNSUPPORTED;
  if (d->chunk != 0 && d->chunk != 32 && d->chunk != 64) return PATH_ERR_UNSUPPORTED;
  // head dim 128: the SIMT kernels' shared memory holds 32-row chunks only (bf16 forwards run the
  // tensor-core kernels on 64-row chunks; their backward takes 32-row chunks whatever the descriptor)
  if (d->head_dim == kHeadDimWide && d->chunk == 64 && d->dtype != PATH_BF16) return PATH_ERR_UNSUPPORTED;
  int B = for_backward ? 32 : (d->chunk ? d->chunk : (d->head_dim == kHeadDimWide ? 32 : 64));
  // The tensor-core paths scan 64-row key chunks and 128-row query tiles.
  const bool tc = uses_tensor_cores(d, for_backward) || uses_tc128(d, for_backward);
  if (tc) B = 64;
  long long nc = (d->seqlen + B - 1) / B;
  if (tc) nc = (d->seqlen + 127) / 128 * 2;
  if (nc * (B / 32) > 65535 || nc * B > (1LL << 30)) return PATH_ERR_UNSUPPORTED;
  if (g) {
    g->BH = (int)BH;
    g->L = d->seqlen;
    g->B = B;
    g->nc = (int)nc;
    g->Lp = (int)(nc * B);
    g->scale = d->scale;
    g->D = d->head_dim;
  }
  return PATH_OK;
}

TcWs tc_layout(const path_attn_desc_t* d, bool for_backward) {
  return tc_ws_layout(d->batch * d->heads, d->seqlen, d->scale, for_backward);
}

// Forward workspace size of the path this descriptor takes.
size_t fwd_ws_total(const path_attn_desc_t* d, const Geom& g) {
  if (uses_tc128(d, 0)) return fwd_ws_layout(g, 2).total;
  return uses_tensor_cores(d, 0) ? tc_layout(d, false).total : fwd_ws_layout(g, 4).total;
}

#define CHECK_PTR(p)                         \
  do {                                       \
    if (!(p)) return PATH_ERR_INVALID_ARG;   \
    if (!aligned((p), 16)) return PATH_ERR_INVALID_ARG; \
  } while (0)

int cuda_status(cudaError_t e) { return e == cudaSuccess ? PATH_OK : PATH_ERR_CUDA; }

// Test hook of the failure path: PATH_ATTN_DEBUG_STALL_NS=<n> (n > 0) in the environment makes
// the forward's PREPARE phase on the tensor-core path give up a wait after n ns in every CTA (see
// launch_ut_prep64).  Read at every call; unset (the normal case) it is 0.
uint32_t debug_stall_ns() {
  const char* v = getenv("PATH_ATTN_DEBUG_STALL_NS");
  if (!v || !*v) return 0;
  const long long n = atoll(v);
  return n <= 0 ? 0u : (n > 1000000000LL ? 1000000000u : (uint32_t)n);
}

// Reads the int error word at dev_word after the work queued on st; PATH_ERR_INTERNAL if it is set.
int read_error_word(const void* dev_word, int* code, cudaStream_t st) {
  int h = 0;
  cudaError_t e = cudaMemcpyAsync(&h, dev_word, sizeof(int), cudaMemcpyDeviceToHost, st);
  if (e == cudaSuccess) e = cudaStreamSynchronize(st);
  if (e != cudaSuccess) return PATH_ERR_CUDA;
  if (code) *code = h;
  return h == 0 ? PATH_OK : PATH_ERR_INTERNAL;
}

}  // namespace

#define PATH_API __attribute__((visibility("default")))
extern "C" {

PATH_API const char* path_status_string(int status) {
  switch (status) {
    case PATH_OK: return "PATH_OK";
    case PATH_ERR_INVALID_ARG: return "PATH_ERR_INVALID_ARG: invalid argument (null/misaligned pointer, bad size or enum)";
    case PATH_ERR_UNSUPPORTED: return "PATH_ERR_UNSUPPORTED: valid but unsupported configuration";
    case PATH_ERR_WORKSPACE: return "PATH_ERR_WORKSPACE: workspace too small";
    case PATH_ERR_CAPACITY: return "PATH_ERR_CAPACITY: decode position exceeds cache capacity";
    case PATH_ERR_CUDA: return "PATH_ERR_CUDA: CUDA launch or runtime error";
    case PATH_ERR_INTERNAL: return "PATH_ERR_INTERNAL: internal error";
    default: return "unknown path_status_t";
  }
}

PATH_API int path_attn_chunk(const path_attn_desc_t* desc, int for_backward) {
  Geom g;
  const int rc = check_desc(desc, for_backward, &g);
  return rc == PATH_OK ? g.B : -rc;
}

PATH_API size_t path_attn_workspace_size(const path_attn_desc_t* desc, int for_backward) {
  Geom g;
  if (check_desc(desc, for_backward, &g) != PATH_OK) return 0;
  if (for_backward) return uses_tensor_cores(desc, 1) ? tc_layout(desc, true).total : bwd_ws_layout(g).total;
  return fwd_ws_total(desc, g);
}

PATH_API int path_attn_fwd_phases(int phases, const path_attn_desc_t* desc, const void* q,
                                  const void* k, const void* v, const void* w, const float* beta,
                                  const float* log_f, void* o, float* lse, void* ws,
                                  size_t ws_bytes, void* stream) {
  Geom g;
  int rc = check_desc(desc, 0, &g);
  if (rc != PATH_OK) return rc;
  if ((phases & PATH_FWD_ALL) == 0 || (phases & ~(PATH_FWD_ALL | PATH_FWD_STORE_Z))) return PATH_ERR_INVALID_ARG;
  CHECK_PTR(q); CHECK_PTR(k); CHECK_PTR(v); CHECK_PTR(w); CHECK_PTR(beta); CHECK_PTR(o); CHECK_PTR(lse);
  if (log_f && !aligned(log_f, 16)) return PATH_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return PATH_ERR_INVALID_ARG;
  if (ws_bytes < fwd_ws_total(desc, g)) return PATH_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  const bool bf = desc->dtype == PATH_BF16;
  char* wsb = (char*)ws;
  if (uses_tensor_cores(desc, 0)) {
    const TcWs tw = tc_layout(desc, false);
    void* zstore = nullptr;
    if (phases & PATH_FWD_STORE_Z) {  // the backward-sized layout holds the Z store
      const TcWs twb = tc_layout(desc, true);
      if (ws_bytes < twb.total) return PATH_ERR_WORKSPACE;
      zstore = wsb + twb.zs;
    }
    if (phases & PATH_FWD_PREPARE) {
      rc = cuda_status(cudaMemsetAsync(wsb + tw.p64.err, 0, sizeof(int), st));
      if (rc == PATH_OK)
        rc = cuda_status(launch_ut_prep64(tw.g64, q, k, v, w, beta, log_f, wsb, tw.p64, true, st, false,
                                          debug_stall_ns()));
      if (rc != PATH_OK) return rc;
    }
    if (phases & PATH_FWD_SCAN) {
      rc = cuda_status(launch_scan_tc(tw.g64, v, log_f, wsb, tw.p64, o, lse, zstore, st));
      if (rc != PATH_OK) return rc;
    }
    return PATH_OK;
  }
  if (uses_tc128(desc, 0)) {  // (no Z store: the head-dim-128 backward recomputes its own operands)
    const FwdWs lay = fwd_ws_layout(g, 2);
    if (phases & PATH_FWD_PREPARE) {
      rc = cuda_status(cudaMemsetAsync(wsb + lay.err, 0, sizeof(int), st));
      if (rc == PATH_OK) rc = cuda_status(launch_ut_prep128(g, q, k, v, w, beta, log_f, wsb, lay, st));
      if (rc != PATH_OK) return rc;
    }
    if (phases & PATH_FWD_SCAN) {
      rc = cuda_status(launch_scan128_tc(g, v, log_f, wsb, lay, o, lse, st));
      if (rc != PATH_OK) return rc;
    }
    return PATH_OK;
  }
  const FwdWs lay = fwd_ws_layout(g, 4);
  if (phases & PATH_FWD_PREPARE) {
    rc = cuda_status(launch_prep_simt(bf, g, q, k, v, w, beta, log_f, wsb, lay, true, st));
    if (rc != PATH_OK) return rc;
  }
  if (phases & PATH_FWD_SCAN) {
    rc = cuda_status(launch_main_simt(bf, g, v, log_f, wsb, lay, o, lse, st));
    if (rc != PATH_OK) return rc;
  }
  return PATH_OK;
}

PATH_API int path_attn_fwd(const path_attn_desc_t* desc, const void* q, const void* k, const void* v,
                           const void* w, const float* beta, const float* log_f, void* o, float* lse,
                           void* ws, size_t ws_bytes, void* stream) {
  return path_attn_fwd_phases(PATH_FWD_ALL, desc, q, k, v, w, beta, log_f, o, lse, ws, ws_bytes, stream);
}

PATH_API int path_attn_bwd_phases(int phases, const path_attn_desc_t* desc, const void* q,
                                  const void* k, const void* v, const void* w, const float* beta,
                                  const float* log_f, const void* o, const float* lse,
                                  const void* dO, void* dq, void* dk, void* dv, void* dw,
                                  float* dbeta, float* dlog_f, void* ws, size_t ws_bytes,
                                  void* stream) {
  Geom g;
  int rc = check_desc(desc, 1, &g);
  if (rc != PATH_OK) return rc;
  if ((phases & PATH_BWD_ALL) == 0 || (phases & ~(PATH_BWD_ALL | PATH_BWD_REUSE_FWD | PATH_BWD_Z_FROM_FWD)))
    return PATH_ERR_INVALID_ARG;
  CHECK_PTR(q); CHECK_PTR(k); CHECK_PTR(v); CHECK_PTR(w); CHECK_PTR(beta); CHECK_PTR(o);
  CHECK_PTR(lse); CHECK_PTR(dO); CHECK_PTR(dq); CHECK_PTR(dk); CHECK_PTR(dv); CHECK_PTR(dw);
  CHECK_PTR(dbeta);
  if (dlog_f && !log_f) return PATH_ERR_INVALID_ARG;
  if (log_f && !aligned(log_f, 16)) return PATH_ERR_INVALID_ARG;
  if (dlog_f && !aligned(dlog_f, 16)) return PATH_ERR_INVALID_ARG;
  if (!ws || !aligned(ws, 256)) return PATH_ERR_INVALID_ARG;
  if (uses_tensor_cores(desc, 1)) {
    // PaTH-FoX: the tensor-core backward takes the forget gate (dlog f needs a nonzero scale: the
    // logit gradient is recovered from the scaled one)
    if (log_f && desc->scale == 0.f) return PATH_ERR_UNSUPPORTED;
    const TcWs tw = tc_layout(desc, true);
    if (ws_bytes < tw.total) return PATH_ERR_WORKSPACE;
    return cuda_status(launch_bwd_tc(tw, q, k, v, w, beta, o, lse, dO, dq, dk, dv, dw, dbeta, (char*)ws, phases,
                                     (cudaStream_t)stream, log_f, dlog_f));
  }
  const BwdWs lay = bwd_ws_layout(g);
  if (ws_bytes < lay.total) return PATH_ERR_WORKSPACE;
  return cuda_status(launch_bwd_simt(desc->dtype == PATH_BF16, g, q, k, v, w, beta, o, lse, dO, dq,
                                     dk, dv, dw, dbeta, (char*)ws, lay, phases & PATH_BWD_ALL,
                                     (cudaStream_t)stream, log_f, dlog_f));
}

PATH_API int path_attn_bwd(const path_attn_desc_t* desc, const void* q, const void* k, const void* v,
                           const void* w, const float* beta, const float* log_f, const void* o,
                           const float* lse, const void* dO, void* dq, void* dk, void* dv, void* dw,
                           float* dbeta, float* dlog_f, void* ws, size_t ws_bytes, void* stream) {
  return path_attn_bwd_phases(PATH_BWD_ALL, desc, q, k, v, w, beta, log_f, o, lse, dO, dq, dk, dv, dw,
                              dbeta, dlog_f, ws, ws_bytes, stream);
}

PATH_API size_t path_decode_workspace_size(const path_decode_desc_t* d) {
  if (!d || d->batch <= 0 || d->heads <= 0 || d->capacity <= 0) return 0;
  if (d->head_dim != kHeadDim && d->head_dim != kHeadDimWide) return 0;
  if (d->cache_dtype != PATH_BF16 && d->cache_dtype != PATH_FP32) return 0;
  const long long BH = (long long)d->batch * d->heads;
  if (BH > 65535) return 0;
  return decode_ws_bytes((int)BH, d->head_dim);
}

PATH_API int path_decode_step(const path_decode_desc_t* d, void* k_cache, void* v_cache, int t,
                     const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                     const float* beta_t, void* o_t, void* ws, size_t ws_bytes, void* stream) {
  if (!d) return PATH_ERR_INVALID_ARG;
  if (d->batch <= 0 || d->heads <= 0 || d->capacity <= 0 || d->head_dim <= 0) return PATH_ERR_INVALID_ARG;
  if (d->cache_dtype != PATH_BF16 && d->cache_dtype != PATH_FP32) return PATH_ERR_INVALID_ARG;
  if (!isfinite(d->scale)) return PATH_ERR_INVALID_ARG;
  if (d->head_dim != kHeadDim && d->head_dim != kHeadDimWide) return PATH_ERR_UNSUPPORTED;
  const long long BH = (long long)d->batch * d->heads;
  if (BH > 65535) return PATH_ERR_UNSUPPORTED;
  if (t < 0) return PATH_ERR_INVALID_ARG;
  if ((long long)t + 1 > d->capacity) return PATH_ERR_CAPACITY;
  CHECK_PTR(k_cache); CHECK_PTR(v_cache); CHECK_PTR(q_t); CHECK_PTR(k_t); CHECK_PTR(v_t);
  CHECK_PTR(w_t); CHECK_PTR(beta_t); CHECK_PTR(o_t);
  if (!ws || !aligned(ws, 256)) return PATH_ERR_INVALID_ARG;
  if (ws_bytes < decode_ws_bytes((int)BH, d->head_dim)) return PATH_ERR_WORKSPACE;
  return cuda_status(launch_decode(d->cache_dtype == PATH_BF16, (int)BH, d->capacity, t, d->scale,
                                   k_cache, v_cache, q_t, k_t, v_t, w_t, beta_t, o_t, (float*)ws,
                                   (cudaStream_t)stream, nullptr, nullptr, d->head_dim));
}

// Geometry of the prompt of a prefill hand-off: 64-row chunks over prompt_len rows (32-row chunks
// at head dim 128).
static Geom prefill_geom(const path_decode_desc_t* d, int prompt_len) {
  Geom g;
  g.BH = d->batch * d->heads;
  g.L = prompt_len;
  g.D = d->head_dim;
  g.B = g.D == kHeadDimWide ? 32 : 64;
  g.nc = (prompt_len + g.B - 1) / g.B;
  g.Lp = g.nc * g.B;
  g.scale = d->scale;
  return g;
}

static int check_decode_desc(const path_decode_desc_t* d) {
  if (!d) return PATH_ERR_INVALID_ARG;
  if (d->batch <= 0 || d->heads <= 0 || d->capacity <= 0 || d->head_dim <= 0) return PATH_ERR_INVALID_ARG;
  if (d->cache_dtype != PATH_BF16 && d->cache_dtype != PATH_FP32) return PATH_ERR_INVALID_ARG;
  if (!isfinite(d->scale)) return PATH_ERR_INVALID_ARG;
  if (d->head_dim != kHeadDim && d->head_dim != kHeadDimWide) return PATH_ERR_UNSUPPORTED;
  if ((long long)d->batch * d->heads > 65535) return PATH_ERR_UNSUPPORTED;
  return PATH_OK;
}

PATH_API size_t path_decode_prefill_workspace_size(const path_decode_desc_t* d, int prompt_len) {
  if (check_decode_desc(d) != PATH_OK || prompt_len < 0 || prompt_len > d->capacity) return 0;
  return prefill_ws_bytes(prefill_geom(d, prompt_len), d->cache_dtype == PATH_BF16);
}

PATH_API int path_decode_prefill(const path_decode_desc_t* d, void* k_cache, void* v_cache, int prompt_len,
                                 const void* k, const void* v, const void* w, const float* beta,
                                 const float* log_f, float* a_cache, void* ws, size_t ws_bytes, void* stream) {
  int rc = check_decode_desc(d);
  if (rc != PATH_OK) return rc;
  if (prompt_len < 0) return PATH_ERR_INVALID_ARG;
  if (prompt_len > d->capacity) return PATH_ERR_CAPACITY;
  CHECK_PTR(k_cache); CHECK_PTR(v_cache); CHECK_PTR(k); CHECK_PTR(v); CHECK_PTR(w); CHECK_PTR(beta);
  if ((!log_f) != (!a_cache)) return PATH_ERR_INVALID_ARG;
  if (log_f) { CHECK_PTR(log_f); CHECK_PTR(a_cache); }
  if (!ws || !aligned(ws, 256)) return PATH_ERR_INVALID_ARG;
  const Geom g = prefill_geom(d, prompt_len);
  const bool bf = d->cache_dtype == PATH_BF16;
  if (ws_bytes < prefill_ws_bytes(g, bf)) return PATH_ERR_WORKSPACE;
  if (prompt_len == 0) return PATH_OK;
  return cuda_status(launch_prefill(bf, g, d->capacity, k, v, w, beta, k_cache, v_cache, (char*)ws,
                                    (cudaStream_t)stream, log_f, a_cache));
}

PATH_API int path_decode_step_fox(const path_decode_desc_t* d, void* k_cache, void* v_cache, float* a_cache, int t,
                                  const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                                  const float* beta_t, const float* log_f_t, void* o_t, void* ws, size_t ws_bytes,
                                  void* stream) {
  int rc = check_decode_desc(d);
  if (rc != PATH_OK) return rc;
  if (t < 0) return PATH_ERR_INVALID_ARG;
  if ((long long)t + 1 > d->capacity) return PATH_ERR_CAPACITY;
  CHECK_PTR(k_cache); CHECK_PTR(v_cache); CHECK_PTR(a_cache); CHECK_PTR(q_t); CHECK_PTR(k_t); CHECK_PTR(v_t);
  CHECK_PTR(w_t); CHECK_PTR(beta_t); CHECK_PTR(log_f_t); CHECK_PTR(o_t);
  const int BH = d->batch * d->heads;
  if (!ws || !aligned(ws, 256)) return PATH_ERR_INVALID_ARG;
  if (ws_bytes < decode_ws_bytes(BH, d->head_dim)) return PATH_ERR_WORKSPACE;
  return cuda_status(launch_decode(d->cache_dtype == PATH_BF16, BH, d->capacity, t, d->scale, k_cache, v_cache,
                                   q_t, k_t, v_t, w_t, beta_t, o_t, (float*)ws, (cudaStream_t)stream, a_cache,
                                   log_f_t, d->head_dim));
}

PATH_API int path_attn_workspace_status(const path_attn_desc_t* desc, int for_backward, const void* ws,
                                        size_t ws_bytes, int* code, void* stream) {
  Geom g;
  int rc = check_desc(desc, for_backward ? 1 : 0, &g);
  if (rc != PATH_OK) return rc;
  if (!ws || !aligned(ws, 256)) return PATH_ERR_INVALID_ARG;
  if (code) *code = 0;
  if (uses_tc128(desc, for_backward)) {
    const FwdWs lay = fwd_ws_layout(g, 2);
    if (ws_bytes < lay.total) return PATH_ERR_WORKSPACE;
    return read_error_word((const char*)ws + lay.err, code, (cudaStream_t)stream);
  }
  if (!uses_tensor_cores(desc, for_backward)) return PATH_OK;  // no bounded waits on the fp32 path
  const TcWs tw = tc_layout(desc, for_backward != 0);
  if (ws_bytes < tw.total) return PATH_ERR_WORKSPACE;
  return read_error_word((const char*)ws + tw.p64.err, code, (cudaStream_t)stream);
}

PATH_API int path_decode_prefill_status(const path_decode_desc_t* d, int prompt_len, const void* ws,
                                        size_t ws_bytes, int* code, void* stream) {
  int rc = check_decode_desc(d);
  if (rc != PATH_OK) return rc;
  if (prompt_len < 0) return PATH_ERR_INVALID_ARG;
  if (prompt_len > d->capacity) return PATH_ERR_CAPACITY;
  if (!ws || !aligned(ws, 256)) return PATH_ERR_INVALID_ARG;
  if (code) *code = 0;
  const Geom g = prefill_geom(d, prompt_len);
  const bool bf = d->cache_dtype == PATH_BF16;
  if (ws_bytes < prefill_ws_bytes(g, bf)) return PATH_ERR_WORKSPACE;
  const size_t off = prefill_err_offset(g, bf);
  if (prompt_len == 0 || off == (size_t)-1) return PATH_OK;  // nothing ran / no bounded waits
  return read_error_word((const char*)ws + off, code, (cudaStream_t)stream);
}

}  // extern "C"
