// Prefill -> decode hand-off.
//
// The decode step of the PaTH reading notes (cc.laoqi.cc/papers/2505.16381, §2.8, Eq. (1))
// expects every cached key already transported to the newest position: after a prompt of L
// tokens, row j of the key cache must hold
//   k~_j = H_{L-1} ... H_{j+1} k_j,           H_t = I - beta_t w_t w_t^T,
// and the last paragraph of §2.8 says the block suffix products do this.  Blockwise (§2.6-§2.7),
// for the 64-row chunk c that holds j:
//   K->_c row j = H_{e(c)} ... H_{j+1} k_j     (the key moved to the end of its own chunk)
//   F_c = I - W_c^T U_c^T W_c = H_{s(c)} ... H_{e(c)}, so H_{e(c)} ... H_{s(c)} = F_c^T,
// hence k~_j = F_{nc-1}^T ... F_{c+1}^T K->_c row j.  With the suffix products
//   S_{nc-1} = I,   S_{c-1} = S_c F_c^T,
// the cache rows of chunk c are K->_c S_c^T.  At head dim 64, for a bf16 cache, K-> (bf16) and F
// (split into bf16 high and low tiles, from split-precision products: the long suffix chain must
// not accumulate bf16 rounding) come from the tcgen05 UT preparation (ut_tc.cu, without its query
// side) on 64-row chunks, and the walk runs on the tensor cores with S split the same way
// (walk_tc.cu).  For an fp32 cache, and at head dim 128 for both cache types, both come from the
// fp32 SIMT preparation (simt_fwd.cu), at head dim 128 on 32-row chunks, and one CTA per head
// walks the chunks right to left on the CUDA cores, keeping S (d x d) in shared memory, in fp32:
// per chunk CB d^2 + d^3 multiply-adds.
#include "internal.h"
#include "dev_common.cuh"
#include "walk_common.cuh"

#include <type_traits>

namespace pathattn {
namespace {

constexpr int PT = 256;      // threads: each owns one or more 4 x 4 blocks of a product

// Shared memory of the walk at head dim D (chunk rows CB <= D), rows padded to LD = D + 1 floats:
// S_c, then K->_c or F_c, then S_c F_c^T before it replaces S.
template <int D>
constexpr size_t prefill_smem_bytes() { return (size_t)3 * D * (D + 1) * sizeof(float); }

template <typename T, typename KR, int D, int CB>
__global__ void __launch_bounds__(PT) prefill_transport_kernel(int L, int Lp, int nc, int cap,
                                                               const KR* __restrict__ kr,
                                                               const float* __restrict__ f,
                                                               T* __restrict__ k_cache) {
  constexpr int LD = D + 1;
  constexpr int NB = D / 4;  // 4-column blocks of an output row
  extern __shared__ float smem_f[];
  float* ss = smem_f;            // S_c
  float* sa = ss + D * LD;       // K->_c, then F_c
  float* st = sa + D * LD;       // S_c F_c^T
  const int tid = threadIdx.x, bh = blockIdx.x;
  for (int e = tid; e < D * D; e += PT) ss[(e / D) * LD + e % D] = (e / D == e % D) ? 1.f : 0.f;
  for (int c = nc - 1; c >= 0; --c) {
    const int rows = min(CB, L - c * CB);
    const KR* src = kr + ((size_t)bh * Lp + (size_t)c * CB) * D;
    if (tid == 0 && c > 0) {  // F_c (used after the first product) and the next step's K-> into L2
      l2_prefetch(f + ((size_t)bh * nc + c) * D * D, D * D * sizeof(float));
      l2_prefetch(kr + ((size_t)bh * Lp + (size_t)(c - 1) * CB) * D, CB * D * sizeof(KR));
    }
    for (int e = tid; e < CB * D; e += PT) sa[(e / D) * LD + e % D] = e / D < rows ? to_f(src[e]) : 0.f;
    __syncthreads();
    for (int blk = tid; blk < (CB / 4) * NB; blk += PT) {  // K->_c S_c^T
      const int r0 = 4 * (blk / NB), n0 = 4 * (blk % NB);
      float acc[4][4];
      mm_abt<D, LD>(sa, ss, r0, n0, acc);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        if (r0 + i < rows) {
          T* dst = k_cache + ((size_t)bh * cap + (size_t)c * CB + r0 + i) * D + n0;
#pragma unroll
          for (int j = 0; j < 4; ++j) dst[j] = from_f<T>(acc[i][j]);
        }
      }
    }
    if (c == 0) break;
    __syncthreads();  // every thread has read K->_c
    const float* fc = f + ((size_t)bh * nc + c) * D * D;
    for (int e = tid; e < D * D; e += PT) sa[(e / D) * LD + e % D] = fc[e];
    __syncthreads();
    for (int blk = tid; blk < NB * NB; blk += PT) {  // S_c F_c^T
      const int r0 = 4 * (blk / NB), n0 = 4 * (blk % NB);
      float acc[4][4];
      mm_abt<D, LD>(ss, sa, r0, n0, acc);
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) st[(r0 + i) * LD + n0 + j] = acc[i][j];
    }
    __syncthreads();
    for (int e = tid; e < D * D; e += PT) ss[(e / D) * LD + e % D] = st[(e / D) * LD + e % D];
    __syncthreads();
  }
}

// Workspace of the hand-off: the forward layout of the chosen preparation (bf16 tcgen05 or fp32
// SIMT), plus the split F array of the bf16 path (two bf16 tiles, 16 KB per chunk).
struct PrefillWs {
  FwdWs lay;
  size_t f32, total;
};
// The tcgen05 preparation (bf16 cache, head dim 64) writes bf16 K-> and a separate split F; the
// SIMT preparation writes both in fp32.
bool prefill_tc(const Geom& g, bool is_bf16) { return is_bf16 && g.D == kHeadDim; }
PrefillWs prefill_ws(const Geom& g, bool is_bf16) {
  PrefillWs w;
  const bool tcp = prefill_tc(g, is_bf16);
  w.lay = fwd_ws_layout(g, tcp ? 2 : 4);
  w.f32 = align_up(w.lay.total, 256);
  w.total = tcp ? w.f32 + (size_t)g.BH * g.nc * g.D * g.D * 4 : w.lay.total;
  return w;
}

// Inclusive prefix sums of log f per head into the forget-gate prefix cache: one CTA of 256
// threads per head, each thread summing a contiguous segment, then a block scan of the segment
// totals (fp32; the decode step extends the same running sum).
__global__ void __launch_bounds__(PT) prefill_logf_prefix_kernel(int L, int cap, const float* __restrict__ logf,
                                                                 float* __restrict__ ac) {
  __shared__ float tot[PT];
  const int tid = threadIdx.x, bh = blockIdx.x;
  const int seg = (L + PT - 1) / PT, j0 = tid * seg, j1 = min(L, j0 + seg);
  const float* src = logf + (size_t)bh * L;
  float s = 0.f;
  for (int j = j0; j < j1; ++j) s += src[j];
  tot[tid] = s;
  __syncthreads();
  for (int o = 1; o < PT; o <<= 1) {  // inclusive Hillis-Steele scan of the segment totals
    const float x = tid >= o ? tot[tid - o] : 0.f;
    __syncthreads();
    tot[tid] += x;
    __syncthreads();
  }
  float run = tid > 0 ? tot[tid - 1] : 0.f;
  float* dst = ac + (size_t)bh * cap;
  for (int j = j0; j < j1; ++j) {
    run += src[j];
    dst[j] = run;
  }
}

template <typename T, typename KR, int D, int CB>
cudaError_t transport(const Geom& g, int cap, const KR* kr, const float* f, void* k_cache, cudaStream_t st) {
  const size_t smem = prefill_smem_bytes<D>();
  auto kern = prefill_transport_kernel<T, KR, D, CB>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)g.BH, PT, smem, st>>>(g.L, g.Lp, g.nc, cap, kr, f, (T*)k_cache);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_ws_bytes(const Geom& g, bool is_bf16) { return prefill_ws(g, is_bf16).total; }

size_t prefill_err_offset(const Geom& g, bool is_bf16) {
  return (is_bf16 && g.D == kHeadDim) ? prefill_ws(g, is_bf16).lay.err : (size_t)-1;
}

cudaError_t launch_prefill(bool is_bf16, const Geom& g, int cap, const void* k, const void* v, const void* w,
                           const float* beta, void* k_cache, void* v_cache, char* ws, cudaStream_t st,
                           const float* logf, float* a_cache) {
  if ((!logf) != (!a_cache)) return cudaErrorInvalidValue;
  if (!((g.D == kHeadDim && g.B == 64) || (g.D == kHeadDimWide && g.B == 32))) return cudaErrorInvalidValue;
  const PrefillWs pw = prefill_ws(g, is_bf16);
  cudaError_t e;
  bool values_done = false;
  // K-> and F of every chunk (the query input is unused here: k stands in for it)
  if (g.D == kHeadDimWide) {
    if ((e = launch_prep_simt(is_bf16, g, k, k, v, w, beta, nullptr, ws, pw.lay, false, st)) != cudaSuccess) return e;
    const float* kr = (const float*)(ws + pw.lay.kr);
    const float* f = (const float*)(ws + pw.lay.f);
    e = is_bf16 ? transport<__nv_bfloat16, float, kHeadDimWide, 32>(g, cap, kr, f, k_cache, st)
                : transport<float, float, kHeadDimWide, 32>(g, cap, kr, f, k_cache, st);
  } else if (is_bf16) {
    FwdWs lay = pw.lay;
    lay.f = pw.f32;  // split F
    if ((e = cudaMemsetAsync(ws + lay.err, 0, sizeof(int), st)) != cudaSuccess) return e;
    // K->, the split F and the values (copied to the cache by the preparation on the way)
    if ((e = launch_ut_prep64(g, k, k, v, w, beta, nullptr, ws, lay, false, st, true, 0, false, v_cache, cap)) !=
        cudaSuccess)
      return e;
    e = launch_walk_tc(g, false, false, ws + lay.kr, ws + pw.f32, k_cache, (size_t)cap, nullptr, (int*)(ws + lay.err),
                       st);
    values_done = true;
  } else {
    if ((e = launch_prep_simt(false, g, k, k, v, w, beta, nullptr, ws, pw.lay, false, st)) != cudaSuccess) return e;
    e = transport<float, float, kHeadDim, 64>(g, cap, (const float*)(ws + pw.lay.kr), (const float*)(ws + pw.lay.f),
                                              k_cache, st);
  }
  if (e != cudaSuccess) return e;
  if (logf) {
    prefill_logf_prefix_kernel<<<(unsigned)g.BH, PT, 0, st>>>(g.L, cap, logf, a_cache);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (values_done) return cudaSuccess;
  // values are appended unchanged: rows 0..L-1 of every (batch, head) slab of the cache
  const size_t row = (size_t)g.D * (is_bf16 ? 2 : 4);
  return cudaMemcpy2DAsync(v_cache, (size_t)cap * row, v, (size_t)g.L * row, (size_t)g.L * row, (size_t)g.BH,
                           cudaMemcpyDeviceToDevice, st);
}

}  // namespace pathattn
