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
// the cache rows of chunk c are K->_c S_c^T.  K-> and F come from the fp32 UT preparation
// (simt_fwd.cu); here one CTA per head walks the chunks right to left, keeping S in shared
// memory, all in fp32: 2 * 64^3 multiply-adds per chunk.
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

template <typename T>
__global__ void __launch_bounds__(PT) prefill_transport_kernel(int L, int Lp, int nc, int cap,
                                                               const float* __restrict__ kr,
                                                               const float* __restrict__ f,
                                                               T* __restrict__ k_cache) {
  extern __shared__ float smem_f[];
  PrefillSmem& s = *reinterpret_cast<PrefillSmem*>(smem_f);
  const int tid = threadIdx.x, bh = blockIdx.x;
  const int r0 = 4 * (tid / 16), n0 = 4 * (tid % 16);
  for (int e = tid; e < D * D; e += PT) s.s[(e / D) * LD + e % D] = (e / D == e % D) ? 1.f : 0.f;
  for (int c = nc - 1; c >= 0; --c) {
    const int rows = min(CB, L - c * CB);
    const float* src = kr + ((size_t)bh * Lp + (size_t)c * CB) * D;
    for (int e = tid; e < CB * D; e += PT) s.a[(e / D) * LD + e % D] = e / D < rows ? src[e] : 0.f;
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

template <typename T>
cudaError_t prefill_t(const Geom& g, int cap, const void* k, const void* v, const void* w, const float* beta,
                      void* k_cache, void* v_cache, char* ws, const FwdWs& lay, cudaStream_t st) {
  // K-> and F of every chunk in fp32 (the query input is unused here: k stands in for it)
  cudaError_t e = launch_prep_simt(std::is_same<T, __nv_bfloat16>::value, g, k, k, v, w, beta, nullptr, ws,
                                   lay, false, st);
  if (e != cudaSuccess) return e;
  const size_t smem = sizeof(PrefillSmem);
  e = cudaFuncSetAttribute(prefill_transport_kernel<T>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  prefill_transport_kernel<T><<<(unsigned)g.BH, PT, smem, st>>>(
      g.L, g.Lp, g.nc, cap, (const float*)(ws + lay.kr), (const float*)(ws + lay.f), (T*)k_cache);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // values are appended unchanged: rows 0..L-1 of every (batch, head) slab of the cache
  const size_t row = (size_t)D * sizeof(T);
  return cudaMemcpy2DAsync(v_cache, (size_t)cap * row, v, (size_t)g.L * row, (size_t)g.L * row, (size_t)g.BH,
                           cudaMemcpyDeviceToDevice, st);
}

}  // namespace

cudaError_t launch_prefill(bool is_bf16, const Geom& g, int cap, const void* k, const void* v, const void* w,
                           const float* beta, void* k_cache, void* v_cache, char* ws, const FwdWs& lay,
                           cudaStream_t st) {
  if (g.B != CB) return cudaErrorInvalidValue;
  return is_bf16 ? prefill_t<__nv_bfloat16>(g, cap, k, v, w, beta, k_cache, v_cache, ws, lay, st)
                 : prefill_t<float>(g, cap, k, v, w, beta, k_cache, v_cache, ws, lay, st);
}

}  // namespace pathattn
