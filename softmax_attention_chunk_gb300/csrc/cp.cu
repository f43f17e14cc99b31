// Context-parallel (sequence-sharded) forward of PaTH attention: the per-shard transports and the
// merge of one remote key block into a shard's softmax state.
//
// The PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.8, last paragraph (the paper's
// Sec. 3.5), sketch sequence parallelism: pass the transported keys and values and the block
// transforms between devices and accumulate right to left.  With the sequence cut into consecutive
// shards, for a query i of shard r and a key j of an earlier shard r':
//   logit(i, j) = scale k~_j^T (M_{r'+1} ... M_{r-1}) z^_i  (+ forget bias)
// with k~_j = H_{e(r')} ... H_{j+1} k_j the key moved to the end of its shard, z^_i =
// H_{s(r)} ... H_i q_i the query moved to the start of its shard and M_s = H_{s(s)} ... H_{e(s)}
// the product over shard s (H_t = I - beta_t w_t w_t^T).  Blockwise (§2.6-§2.7), from the UT
// preparation's K->, Q<- (each row moved to its chunk's end / start) and chunk transforms
// F_c = H_{s(c)} ... H_{e(c)}:
//   k~ rows of chunk c = K->_c S_c^T,  S_{nc-1} = I,  S_{c-1} = S_c F_c^T   (walk right to left)
//   z^ rows of chunk c = Q<-_c P_c,    P_0 = I,       P_{c+1} = F_c^T P_c   (walk left to right)
//   M^T = S_{-1}                                                          (end of the first walk)
// A key block at the end of shard r' reaches the end of shard r by k^ <- M_r^T k^, i.e. the rows
// K^ <- K^ M_r.  Forget gate (§2.5): bias(i, j) = a_i + b_j with a_i = sum_{t = s(r)..i} log f_t
// (shard-local inclusive prefix) and b_j = (T_{r'} - a_j) + the totals T of the shards passed.
// The walks are the hand-off's tensor-core chunk walk (walk_tc.cu: one CTA per head, the running
// product and F split into bf16 high and low parts); the merge is the forward scan's block mode
// (fwd_tc.cu).
#include "../../include/path_attn.h"
#include "internal.h"
#include "dev_common.cuh"
#include "walk_common.cuh"

#include <math.h>
#include <stdint.h>

namespace pathattn {

cudaError_t launch_scan_block(const Geom& g, int Lb, const void* zq, const void* kb, const void* vb,
                              const float* aq, const float* bk, char* ws, const FwdWs& lay, cudaStream_t st);

namespace {

constexpr int D = kHeadDim;
constexpr int CB = 64;  // chunk rows of the tcgen05 preparation
constexpr int LD = D + 1;
constexpr int NB = D / 4;
constexpr int WT = 256;  // threads of the walk and pass kernels

// Forget gate of a shard, one CTA per head: a = inclusive prefix sums of log f, T = the total,
// b = T - a (fp32; segment sums, then a block scan of the segment totals).
__global__ void __launch_bounds__(WT) cp_fox_kernel(int L, const float* __restrict__ logf, float* __restrict__ a,
                                                    float* __restrict__ b, float* __restrict__ tot) {
  __shared__ float seg_tot[WT];
  const int tid = threadIdx.x, bh = blockIdx.x;
  const int seg = (L + WT - 1) / WT, j0 = min(L, tid * seg), j1 = min(L, j0 + seg);
  const float* src = logf + (size_t)bh * L;
  float s = 0.f;
  for (int j = j0; j < j1; ++j) s += src[j];
  seg_tot[tid] = s;
  __syncthreads();
  for (int o = 1; o < WT; o <<= 1) {  // inclusive scan of the segment totals
    const float x = tid >= o ? seg_tot[tid - o] : 0.f;
    __syncthreads();
    seg_tot[tid] += x;
    __syncthreads();
  }
  const float total = seg_tot[WT - 1];
  float run = tid > 0 ? seg_tot[tid - 1] : 0.f;
  for (int j = j0; j < j1; ++j) {
    run += src[j];
    a[(size_t)bh * L + j] = run;
    b[(size_t)bh * L + j] = total - run;
  }
  if (tid == 0) tot[bh] = total;
}

// One hop of a key block through a shard: rows K^ <- K^ M (t = M^T, so K^ t^T), 64 rows of one
// head per CTA, in place; the keys' forget bias gains the shard's total.
__global__ void __launch_bounds__(WT) cp_pass_kernel(int Lb, float* __restrict__ kh, const float* __restrict__ t,
                                                     float* __restrict__ bk, const float* __restrict__ tot) {
  __shared__ float sr[CB * LD], stt[D * LD];
  const int tid = threadIdx.x, c = blockIdx.x, bh = blockIdx.y;
  float* rows = kh + ((size_t)bh * Lb + (size_t)c * CB) * D;
  for (int e = tid; e < D * D; e += WT) stt[(e / D) * LD + e % D] = t[(size_t)bh * D * D + e];
  for (int e = tid; e < CB * D; e += WT) sr[(e / D) * LD + e % D] = rows[e];
  __syncthreads();
  for (int blk = tid; blk < (CB / 4) * NB; blk += WT) {
    const int r0 = 4 * (blk / NB), n0 = 4 * (blk % NB);
    float acc[4][4];
    mm_abt<D, LD>(sr, stt, r0, n0, acc);
#pragma unroll
    for (int i = 0; i < 4; ++i)
      *reinterpret_cast<float4*>(rows + (r0 + i) * D + n0) = make_float4(acc[i][0], acc[i][1], acc[i][2], acc[i][3]);
  }
  if (bk && tid < CB) bk[(size_t)bh * Lb + (size_t)c * CB + tid] += tot[bh];
}

// The block's keys rounded to bf16 (the MMA operand of the scan's block mode).
__global__ void cp_block_operands_kernel(size_t n, const float* __restrict__ kh, __nv_bfloat16* __restrict__ kb) {
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i < n) kb[i] = __float2bfloat16_rn(kh[i]);
}

// Shard geometry: 64-row chunks, L a multiple of 128 (the scan's query tiles).
bool cp_geom(const path_attn_desc_t* d, Geom* g) {
  if (!d || d->batch <= 0 || d->heads <= 0 || d->seqlen <= 0) return false;
  *g = tc_geom(d->batch * d->heads, d->seqlen, d->scale, CB);
  g->D = D;
  return true;
}

int check_cp_desc(const path_attn_desc_t* d) {
  if (!d) return PATH_ERR_INVALID_ARG;
  if (d->batch <= 0 || d->heads <= 0 || d->seqlen <= 0 || d->head_dim <= 0) return PATH_ERR_INVALID_ARG;
  if (d->dtype != PATH_BF16 && d->dtype != PATH_FP32) return PATH_ERR_INVALID_ARG;
  if (!isfinite(d->scale)) return PATH_ERR_INVALID_ARG;
  if (d->dtype != PATH_BF16 || d->head_dim != D || (d->chunk != 0 && d->chunk != 64)) return PATH_ERR_UNSUPPORTED;
  if ((long long)d->batch * d->heads > 65535) return PATH_ERR_UNSUPPORTED;
  if (d->seqlen % 128 != 0 || d->seqlen > (1 << 24)) return PATH_ERR_UNSUPPORTED;
  return PATH_OK;
}

bool al(const void* p, uintptr_t a) { return p && (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct CpPrepWs {
  FwdWs lay;  // the tcgen05 preparation's outputs (bf16 Q<-, K->; the F slot unused; split F at f32)
  size_t f32, total;
};
CpPrepWs cp_prep_ws(const Geom& g) {
  CpPrepWs w;
  w.lay = fwd_ws_layout(g, 2);
  w.f32 = align_up(w.lay.total, 256);
  w.total = w.f32 + (size_t)g.BH * g.nc * D * D * 4;
  return w;
}

size_t cp_block_ws(const Geom& g, int Lb) { return align_up((size_t)g.BH * Lb * D * 2, 256); }

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? PATH_OK : PATH_ERR_CUDA; }

}  // namespace
}  // namespace pathattn

using namespace pathattn;

#define PATH_API __attribute__((visibility("default")))
extern "C" {

PATH_API size_t path_cp_prepare_workspace_size(const path_attn_desc_t* desc) {
  Geom g;
  if (check_cp_desc(desc) != PATH_OK || !cp_geom(desc, &g)) return 0;
  return cp_prep_ws(g).total;
}

PATH_API int path_cp_shard_prepare(const path_attn_desc_t* desc, const void* q, const void* k, const void* w,
                                   const float* beta, const float* log_f, float* k_end, void* q_start,
                                   float* t_shard, float* a_q, float* b_k, float* f_tot, void* ws, size_t ws_bytes,
                                   void* stream) {
  int rc = check_cp_desc(desc);
  if (rc != PATH_OK) return rc;
  const void* ptrs[] = {q, k, w, beta, k_end, q_start, t_shard};
  for (const void* p : ptrs)
    if (!al(p, 16)) return PATH_ERR_INVALID_ARG;
  const bool fox = log_f != nullptr;
  if (fox != (a_q != nullptr) || fox != (b_k != nullptr) || fox != (f_tot != nullptr)) return PATH_ERR_INVALID_ARG;
  if (fox && (!al(log_f, 16) || !al(a_q, 16) || !al(b_k, 16) || !al(f_tot, 16))) return PATH_ERR_INVALID_ARG;
  if (!al(ws, 256)) return PATH_ERR_INVALID_ARG;
  Geom g;
  cp_geom(desc, &g);
  const CpPrepWs pw = cp_prep_ws(g);
  if (ws_bytes < pw.total) return PATH_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  char* wsb = (char*)ws;
  FwdWs lay = pw.lay;
  lay.f = pw.f32;  // split F
  int* err = (int*)(wsb + lay.err);
  if ((rc = cuda_rc(cudaMemsetAsync(err, 0, sizeof(int), st))) != PATH_OK) return rc;
  // K->, Q<- (bf16) and the split chunk transforms of every chunk (the values are not needed: k
  // stands in for them)
  if ((rc = cuda_rc(launch_ut_prep64(g, q, k, k, w, beta, nullptr, wsb, lay, false, st, true))) != PATH_OK) return rc;
  if ((rc = cuda_rc(launch_walk_tc_pair(g, wsb + lay.kr, wsb + lay.ql, wsb + pw.f32, k_end, q_start, g.L, t_shard, err,
                                        st))) != PATH_OK)
    return rc;
  if (fox) {
    cp_fox_kernel<<<(unsigned)g.BH, WT, 0, st>>>(g.L, log_f, a_q, b_k, f_tot);
    if ((rc = cuda_rc(cudaGetLastError())) != PATH_OK) return rc;
  }
  return PATH_OK;
}

PATH_API size_t path_cp_block_workspace_size(const path_attn_desc_t* desc, int block_len) {
  Geom g;
  if (check_cp_desc(desc) != PATH_OK || !cp_geom(desc, &g) || block_len <= 0 || block_len % 128 != 0 ||
      block_len > (1 << 24))
    return 0;
  return cp_block_ws(g, block_len);
}

PATH_API int path_cp_attend_block(const path_attn_desc_t* desc, int block_len, const void* q_start,
                                  const float* k_block, const void* v_block, const float* a_q, const float* b_k,
                                  void* fwd_ws, size_t fwd_ws_bytes, void* blk_ws, size_t blk_ws_bytes, void* stream) {
  int rc = check_cp_desc(desc);
  if (rc != PATH_OK) return rc;
  if (block_len <= 0 || block_len > (1 << 24)) return PATH_ERR_INVALID_ARG;
  if (block_len % 128 != 0) return PATH_ERR_UNSUPPORTED;
  const void* ptrs[] = {q_start, k_block, v_block};
  for (const void* p : ptrs)
    if (!al(p, 16)) return PATH_ERR_INVALID_ARG;
  if ((a_q != nullptr) != (b_k != nullptr)) return PATH_ERR_INVALID_ARG;
  if (a_q && (!al(a_q, 16) || !al(b_k, 16))) return PATH_ERR_INVALID_ARG;
  if (!al(fwd_ws, 256) || !al(blk_ws, 256)) return PATH_ERR_INVALID_ARG;
  Geom g;
  cp_geom(desc, &g);
  const TcWs tw = tc_ws_layout(g.BH, g.L, g.scale, false);
  if (fwd_ws_bytes < tw.total || blk_ws_bytes < cp_block_ws(g, block_len)) return PATH_ERR_WORKSPACE;
  cudaStream_t st = (cudaStream_t)stream;
  char* bw = (char*)blk_ws;
  __nv_bfloat16* kb = (__nv_bfloat16*)bw;
  const size_t n = (size_t)g.BH * block_len * D;
  cp_block_operands_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(n, k_block, kb);
  if ((rc = cuda_rc(cudaGetLastError())) != PATH_OK) return rc;
  return cuda_rc(launch_scan_block(tw.g64, block_len, q_start, kb, v_block, a_q, b_k, (char*)fwd_ws, tw.p64, st));
}

PATH_API int path_cp_pass_block(const path_attn_desc_t* desc, int block_len, float* k_block, float* b_k,
                                const float* t_shard, const float* f_tot, void* stream) {
  int rc = check_cp_desc(desc);
  if (rc != PATH_OK) return rc;
  if (block_len <= 0 || block_len > (1 << 24)) return PATH_ERR_INVALID_ARG;
  if (block_len % 128 != 0) return PATH_ERR_UNSUPPORTED;
  if (!al(k_block, 16) || !al(t_shard, 16)) return PATH_ERR_INVALID_ARG;
  if ((b_k != nullptr) != (f_tot != nullptr)) return PATH_ERR_INVALID_ARG;
  if (b_k && (!al(b_k, 16) || !al(f_tot, 16))) return PATH_ERR_INVALID_ARG;
  const int BH = desc->batch * desc->heads;
  cp_pass_kernel<<<dim3((unsigned)(block_len / CB), (unsigned)BH), WT, 0, (cudaStream_t)stream>>>(block_len, k_block,
                                                                                              t_shard, b_k, f_tot);
  return cuda_rc(cudaGetLastError());
}

}  // extern "C"
