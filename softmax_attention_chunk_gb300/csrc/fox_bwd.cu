// PaTH-FoX backward: the forget-gate parts that are plain scans over the sequence.
//
// With the forget gate (PaTH reading notes cc.laoqi.cc/papers/2505.16381, §2.5) the logit of the
// pair (i, j) gains sum_{s=j+1..i} log f_s = A_i - A_j, A_i = sum_{s<=i} log f_s.  With
// dS'_ij = P_ij (dP_ij - D_i) the gradient of a logit,
//   dL/dA_m = rowsum_m(dS') - colsum_m(dS'),
//   dL/dlog f_s = sum_{m>=s} dL/dA_m = -sum_{m>=s} (colsum_m - rowsum_m).
// In exact arithmetic every row of dS' sums to zero (sum_j P_ij dP_ij = dO_i . o_i = D_i), but D_i
// is formed from the rounded output, so the computed rows do not, and dropping them would
// accumulate along the suffix sum: both terms are kept.  The backward scans add
// colsum_m - rowsum_m into cs; these kernels form A before them and dlog f after them, one CTA per
// head: each thread sums a contiguous segment, a block scan joins the segments.
#include "internal.h"
#include "dev_common.cuh"

namespace pathattn {
namespace {

constexpr int ST = 256;

// Inclusive block scan of one value per thread (Hillis-Steele over shared memory).
__device__ __forceinline__ float block_inclusive_scan(float v, float* tot) {
  const int tid = threadIdx.x;
  tot[tid] = v;
  __syncthreads();
  for (int o = 1; o < ST; o <<= 1) {
    const float x = tid >= o ? tot[tid - o] : 0.f;
    __syncthreads();
    tot[tid] += x;
    __syncthreads();
  }
  return tot[tid];
}

__global__ void __launch_bounds__(ST) fox_prefix_kernel(int L, int Lp, const float* __restrict__ logf,
                                                        float* __restrict__ A) {
  __shared__ float tot[ST];
  const int tid = threadIdx.x, bh = blockIdx.x;
  const int seg = (Lp + ST - 1) / ST, j0 = tid * seg, j1 = min(Lp, j0 + seg);
  const float* src = logf + (size_t)bh * L;
  float s = 0.f;
  for (int j = j0; j < j1; ++j) s += j < L ? src[j] : 0.f;
  float run = block_inclusive_scan(s, tot) - s;  // exclusive prefix of this segment
  float* dst = A + (size_t)bh * Lp;
  for (int j = j0; j < j1; ++j) {
    run += j < L ? src[j] : 0.f;
    dst[j] = run;
  }
}

__global__ void __launch_bounds__(ST) fox_dlogf_kernel(int L, int Lp, const float* __restrict__ cs,
                                                       float* __restrict__ dlogf) {
  __shared__ float tot[ST];
  const int tid = threadIdx.x, bh = blockIdx.x;
  // thread t sums segment ST-1-t of the reversed sequence, so the scan runs from the end
  const int seg = (L + ST - 1) / ST, j1 = L - tid * seg, j0 = max(0, j1 - seg);
  const float* src = cs + (size_t)bh * Lp;
  float s = 0.f;
  for (int j = j0; j < j1; ++j) s += src[j];
  float run = block_inclusive_scan(s, tot) - s;  // sum of cs over the rows after this segment
  float* dst = dlogf + (size_t)bh * L;
  for (int j = j1 - 1; j >= j0; --j) {
    run += src[j];
    dst[j] = -run;
  }
}

}  // namespace

cudaError_t launch_fox_prefix(const Geom& g, const float* logf, float* A, cudaStream_t st) {
  fox_prefix_kernel<<<(unsigned)g.BH, ST, 0, st>>>(g.L, g.Lp, logf, A);
  return cudaGetLastError();
}

cudaError_t launch_fox_dlogf(const Geom& g, const float* cs, float* dlogf, cudaStream_t st) {
  fox_dlogf_kernel<<<(unsigned)g.BH, ST, 0, st>>>(g.L, g.Lp, cs, dlogf);
  return cudaGetLastError();
}

}  // namespace pathattn
