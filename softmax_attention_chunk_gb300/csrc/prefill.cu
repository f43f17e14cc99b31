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
// the cache rows of chunk c are K->_c S_c^T.  For a bf16 cache, K-> (bf16) and F (fp32, from
// split-precision bf16 products: the long suffix chain must not accumulate bf16 rounding) come
// from the tcgen05 UT preparation (ut_tc.cu); for an fp32 cache both come from the fp32 SIMT
// preparation (simt_fwd.cu).  One CTA per head then walks the chunks right to left, keeping S in
// shared memory, in fp32: 2 * 64^3 multiply-adds per chunk.
#include "internal.h"
#include "dev_common.cuh"

#include <type_traits>

namespace pathattn {
namespace {

constexpr int D = kHeadDim;
constexpr int CB = 64;       // chunk rows
constexpr int LD = D + 1;    // padded row stride of the shared-memory matrices
constexpr int PT = 256;      // threads: each owns a 4 x 4 block of a 64 x 64 product

struct PrefillSmem {
  float s[D * LD];   // S_c
  float a[CB * LD];  // K->_c, then F_c
  float t[D * LD];   // S_c F_c^T before it replaces S
};

// Asynchronous copy of `bytes` (a multiple of 16, 16-byte aligned) from global memory into L2.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

// out[r][n] = sum_m A[r][m] * B[n][m] for the thread's 4 x 4 block (A B^T).
__device__ __forceinline__ void mm_abt(const float* A, const float* Bm, int r0, int n0, float (&acc)[4][4]) {
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[i][j] = 0.f;
#pragma unroll 4
  for (int m = 0; m < D; ++m) {
    float a[4], b[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) a[i] = A[(r0 + i) * LD + m];
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = Bm[(n0 + j) * LD + m];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
}

template <typename T, typename KR>
__global__ void __launch_bounds__(PT) prefill_transport_kernel(int L, int Lp, int nc, int cap,
                                                               const KR* __restrict__ kr,
                                                               const float* __restrict__ f,
                                                               T* __restrict__ k_cache) {
  extern __shared__ float smem_f[];
  PrefillSmem& s = *reinterpret_cast<PrefillSmem*>(smem_f);
  const int tid = threadIdx.x, bh = blockIdx.x;
  const int r0 = 4 * (tid / 16), n0 = 4 * (tid % 16);
  for (int e = tid; e < D * D; e += PT) s.s[(e / D) * LD + e % D] = (e / D == e % D) ? 1.f : 0.f;
  for (int c = nc - 1; c >= 0; --c) {
    const int rows = min(CB, L - c * CB);
    const KR* src = kr + ((size_t)bh * Lp + (size_t)c * CB) * D;
    if (tid == 0 && c > 0) {  // F_c (used after the first product) and the next step's K-> into L2
      l2_prefetch(f + ((size_t)bh * nc + c) * D * D, D * D * sizeof(float));
      l2_prefetch(kr + ((size_t)bh * Lp + (size_t)(c - 1) * CB) * D, CB * D * sizeof(KR));
    }
    for (int e = tid; e < CB * D; e += PT) s.a[(e / D) * LD + e % D] = e / D < rows ? to_f(src[e]) : 0.f;
    __syncthreads();
    float acc[4][4];
    mm_abt(s.a, s.s, r0, n0, acc);  // K->_c S_c^T
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      if (r0 + i < rows) {
        T* dst = k_cache + ((size_t)bh * cap + (size_t)c * CB + r0 + i) * D + n0;
#pragma unroll
        for (int j = 0; j < 4; ++j) dst[j] = from_f<T>(acc[i][j]);
      }
    }
    if (c == 0) break;
    __syncthreads();  // every thread has read K->_c
    const float* fc = f + ((size_t)bh * nc + c) * D * D;
    for (int e = tid; e < D * D; e += PT) s.a[(e / D) * LD + e % D] = fc[e];
    __syncthreads();
    mm_abt(s.s, s.a, r0, n0, acc);  // S_c F_c^T
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < 4; ++j) s.t[(r0 + i) * LD + n0 + j] = acc[i][j];
    __syncthreads();
    for (int e = tid; e < D * D; e += PT) s.s[(e / D) * LD + e % D] = s.t[(e / D) * LD + e % D];
    __syncthreads();
  }
}

// Workspace of the hand-off: the forward layout of the chosen preparation (bf16 tcgen05 or fp32
// SIMT), plus the fp32 F array of the bf16 path.
struct PrefillWs {
  FwdWs lay;
  size_t f32, total;
};
PrefillWs prefill_ws(const Geom& g, bool is_bf16) {
  PrefillWs w;
  w.lay = fwd_ws_layout(g, is_bf16 ? 2 : 4);
  w.f32 = align_up(w.lay.total, 256);
  w.total = is_bf16 ? w.f32 + (size_t)g.BH * g.nc * D * D * 4 : w.lay.total;
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

template <typename T, typename KR>
cudaError_t transport(const Geom& g, int cap, const KR* kr, const float* f, void* k_cache, cudaStream_t st) {
  const size_t smem = sizeof(PrefillSmem);
  cudaError_t e = cudaFuncSetAttribute(prefill_transport_kernel<T, KR>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem);
  if (e != cudaSuccess) return e;
  prefill_transport_kernel<T, KR><<<(unsigned)g.BH, PT, smem, st>>>(g.L, g.Lp, g.nc, cap, kr, f, (T*)k_cache);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_ws_bytes(const Geom& g, bool is_bf16) { return prefill_ws(g, is_bf16).total; }

cudaError_t launch_prefill(bool is_bf16, const Geom& g, int cap, const void* k, const void* v, const void* w,
                           const float* beta, void* k_cache, void* v_cache, char* ws, cudaStream_t st,
                           const float* logf, float* a_cache) {
  if (g.B != CB || (!logf) != (!a_cache)) return cudaErrorInvalidValue;
  const PrefillWs pw = prefill_ws(g, is_bf16);
  cudaError_t e;
  // K-> and F of every chunk (the query input is unused here: k stands in for it)
  if (is_bf16) {
    FwdWs lay = pw.lay;
    lay.f = pw.f32;  // F in fp32
    if ((e = cudaMemsetAsync(ws + lay.err, 0, sizeof(int), st)) != cudaSuccess) return e;
    if ((e = launch_ut_prep64(g, k, k, v, w, beta, nullptr, ws, lay, false, st, true)) != cudaSuccess) return e;
    e = transport<__nv_bfloat16>(g, cap, (const __nv_bfloat16*)(ws + lay.kr), (const float*)(ws + pw.f32), k_cache, st);
  } else {
    if ((e = launch_prep_simt(false, g, k, k, v, w, beta, nullptr, ws, pw.lay, false, st)) != cudaSuccess) return e;
    e = transport<float>(g, cap, (const float*)(ws + pw.lay.kr), (const float*)(ws + pw.lay.f), k_cache, st);
  }
  if (e != cudaSuccess) return e;
  if (logf) {
    prefill_logf_prefix_kernel<<<(unsigned)g.BH, PT, 0, st>>>(g.L, cap, logf, a_cache);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  // values are appended unchanged: rows 0..L-1 of every (batch, head) slab of the cache
  const size_t row = (size_t)D * (is_bf16 ? 2 : 4);
  return cudaMemcpy2DAsync(v_cache, (size_t)cap * row, v, (size_t)g.L * row, (size_t)g.L * row, (size_t)g.BH,
                           cudaMemcpyDeviceToDevice, st);
}

}  // namespace pathattn
