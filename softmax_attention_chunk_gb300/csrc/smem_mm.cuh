// Block-level product of small fp32 matrices held in shared memory, used by the CUDA-core per-chunk
// UT kernels (32x32, 32x64, 64x64 operands) and the CUDA-core backward scan (32- or 64-row chunks
// against head-dim-wide operands up to 128 x 128).  C = op(A) op(B) with
//   op(A)(i,k) = TA ? A[k*lda + i] : A[i*lda + k]    (M x K)
//   op(B)(k,j) = TB ? B[j*ldb + k] : B[k*ldb + j]    (K x N)
// and every result element handed to epi(i, j, value).  The operands' zeros encode the
// triangular masks of the UT algebra, so products run over the full K range.
//
// TC = true runs 16x8x8 TF32 warp MMAs (fp32 accumulate; operands rounded to TF32, relative
// 2^-11), the bf16 path's choice: these products are too small and too dependent for tcgen05's
// 64/128-row tiles and TMEM round trips (the head-dim-128 backward keeps them here because its
// accumulators exceed the SM's TMEM).  TC = false is a plain fp32 loop (fp32 mode).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace pathattn {

__device__ __forceinline__ uint32_t to_tf32(float x) {
  uint32_t r;
  asm("cvt.rna.tf32.f32 %0, %1;" : "=r"(r) : "f"(x));
  return r;
}

__device__ __forceinline__ void mma_m16n8k8_tf32(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
  asm volatile(
      "mma.sync.aligned.m16n8k8.row.col.f32.tf32.tf32.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
      "{%0,%1,%2,%3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

template <int M, int N, int K, bool TA, bool TB, bool TC, typename Epi>
__device__ __forceinline__ void smem_mm(const float* A, int lda, const float* B, int ldb, Epi epi) {
  auto LA = [&](int i, int k) { return TA ? A[k * lda + i] : A[i * lda + k]; };
  auto LB = [&](int k, int j) { return TB ? B[j * ldb + k] : B[k * ldb + j]; };
  const int tid = threadIdx.x;
  if constexpr (TC) {
    static_assert(M % 16 == 0 && N % 8 == 0 && K % 16 == 0, "tile shape");
    const int warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int nwarps = blockDim.x >> 5;
    // Products with at least eight 16 x 16 tiles give each warp 16 x 16 tiles: one A fragment
    // serves two MMAs, and two N halves x two K parities make four independent chains.
    constexpr bool WIDE = N % 16 == 0 && (M / 16) * (N / 16) >= 8;
    if constexpr (WIDE) {
      constexpr int TN = N / 16, NTW = (M / 16) * TN;
      for (int tile = warp; tile < NTW; tile += nwarps) {
        const int i0 = (tile / TN) * 16, j0 = (tile % TN) * 16;
        float c0[4] = {0.f, 0.f, 0.f, 0.f}, c1[4] = {0.f, 0.f, 0.f, 0.f};
        float d0[4] = {0.f, 0.f, 0.f, 0.f}, d1[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
        for (int k0 = 0; k0 < K; k0 += 16) {
          const uint32_t a[4] = {to_tf32(LA(i0 + g, k0 + t)), to_tf32(LA(i0 + g + 8, k0 + t)),
                                 to_tf32(LA(i0 + g, k0 + t + 4)), to_tf32(LA(i0 + g + 8, k0 + t + 4))};
          const uint32_t b0[2] = {to_tf32(LB(k0 + t, j0 + g)), to_tf32(LB(k0 + t + 4, j0 + g))};
          const uint32_t b1[2] = {to_tf32(LB(k0 + t, j0 + 8 + g)), to_tf32(LB(k0 + t + 4, j0 + 8 + g))};
          const uint32_t a2[4] = {to_tf32(LA(i0 + g, k0 + 8 + t)), to_tf32(LA(i0 + g + 8, k0 + 8 + t)),
                                  to_tf32(LA(i0 + g, k0 + 12 + t)), to_tf32(LA(i0 + g + 8, k0 + 12 + t))};
          const uint32_t e0[2] = {to_tf32(LB(k0 + 8 + t, j0 + g)), to_tf32(LB(k0 + 12 + t, j0 + g))};
          const uint32_t e1[2] = {to_tf32(LB(k0 + 8 + t, j0 + 8 + g)), to_tf32(LB(k0 + 12 + t, j0 + 8 + g))};
          mma_m16n8k8_tf32(c0, a, b0);
          mma_m16n8k8_tf32(c1, a, b1);
          mma_m16n8k8_tf32(d0, a2, e0);
          mma_m16n8k8_tf32(d1, a2, e1);
        }
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          c0[e] += d0[e];
          c1[e] += d1[e];
        }
        epi(i0 + g, j0 + 2 * t, c0[0]);
        epi(i0 + g, j0 + 2 * t + 1, c0[1]);
        epi(i0 + g + 8, j0 + 2 * t, c0[2]);
        epi(i0 + g + 8, j0 + 2 * t + 1, c0[3]);
        epi(i0 + g, j0 + 8 + 2 * t, c1[0]);
        epi(i0 + g, j0 + 8 + 2 * t + 1, c1[1]);
        epi(i0 + g + 8, j0 + 8 + 2 * t, c1[2]);
        epi(i0 + g + 8, j0 + 8 + 2 * t + 1, c1[3]);
      }
      return;
    }
    constexpr int TN = N / 8, NT = (M / 16) * TN;
    for (int tile = warp; tile < NT; tile += nwarps) {
      const int i0 = (tile / TN) * 16, j0 = (tile % TN) * 8;
      // two accumulators over alternate 8-wide K slices: two independent MMA chains
      float c[4] = {0.f, 0.f, 0.f, 0.f}, c2[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 2
      for (int k0 = 0; k0 < K; k0 += 16) {
        const uint32_t a[4] = {to_tf32(LA(i0 + g, k0 + t)), to_tf32(LA(i0 + g + 8, k0 + t)),
                               to_tf32(LA(i0 + g, k0 + t + 4)), to_tf32(LA(i0 + g + 8, k0 + t + 4))};
        const uint32_t b[2] = {to_tf32(LB(k0 + t, j0 + g)), to_tf32(LB(k0 + t + 4, j0 + g))};
        const uint32_t a2[4] = {to_tf32(LA(i0 + g, k0 + 8 + t)), to_tf32(LA(i0 + g + 8, k0 + 8 + t)),
                                to_tf32(LA(i0 + g, k0 + 12 + t)), to_tf32(LA(i0 + g + 8, k0 + 12 + t))};
        const uint32_t b2[2] = {to_tf32(LB(k0 + 8 + t, j0 + g)), to_tf32(LB(k0 + 12 + t, j0 + g))};
        mma_m16n8k8_tf32(c, a, b);
        mma_m16n8k8_tf32(c2, a2, b2);
      }
#pragma unroll
      for (int e = 0; e < 4; ++e) c[e] += c2[e];
      epi(i0 + g, j0 + 2 * t, c[0]);
      epi(i0 + g, j0 + 2 * t + 1, c[1]);
      epi(i0 + g + 8, j0 + 2 * t, c[2]);
      epi(i0 + g + 8, j0 + 2 * t + 1, c[3]);
    }
  } else {
    for (int idx = tid; idx < M * N; idx += blockDim.x) {
      const int i = idx / N, j = idx % N;
      float acc = 0.f;
#pragma unroll 8
      for (int k = 0; k < K; ++k) acc += LA(i, k) * LB(k, j);
      epi(i, j, acc);
    }
  }
}

}  // namespace pathattn
