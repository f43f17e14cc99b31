// Helpers of the per-head chunk walks (prefill hand-off, context-parallel shard transports):
// L2 prefetch and a 4 x 4 register block of a product of two shared-memory fp32 matrices.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pathattn {

// Asynchronous copy of `bytes` (a multiple of 16, 16-byte aligned) from global memory into L2.
__device__ __forceinline__ void l2_prefetch(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(reinterpret_cast<uint64_t>(p)), "r"(bytes)
               : "memory");
}

// out[r][n] = sum_m A[r][m] * B[n][m] for one 4 x 4 block (A B^T), both operands with row stride
// LD and D columns.
template <int D, int LD>
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

}  // namespace pathattn
