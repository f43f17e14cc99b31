// Helpers of the tcgen05 per-chunk UT kernels (chunk 64): rows of 64x64 bf16 tiles in the
// 128-byte swizzled layout, M=64 N=64 K=64 MMAs on such tiles, and M=64 accumulator rows.
#pragma once

#include "internal.h"
#include "tc_common.cuh"

namespace pathattn {
namespace tc {

// Writes 64 fp32 values as one bf16 row of a 128-byte swizzled 64x64 tile.
__device__ __forceinline__ void put_row(uint8_t* tile, int r, const float* x) {
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    uint4 pk;
    pk.x = pack_bf16(x[8 * q], x[8 * q + 1]);
    pk.y = pack_bf16(x[8 * q + 2], x[8 * q + 3]);
    pk.z = pack_bf16(x[8 * q + 4], x[8 * q + 5]);
    pk.w = pack_bf16(x[8 * q + 6], x[8 * q + 7]);
    *reinterpret_cast<uint4*>(row + ((q ^ (r & 7)) * 16)) = pk;
  }
}
// Reads one row of a swizzled bf16 tile as 64 floats.
__device__ __forceinline__ void get_row(const uint8_t* tile, int r, float* x) {
  const uint8_t* row = tile + r * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const uint4 pk = *reinterpret_cast<const uint4*>(row + ((q ^ (r & 7)) * 16));
    const uint32_t wv[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      x[8 * q + 2 * h] = __uint_as_float(wv[h] << 16);
      x[8 * q + 2 * h + 1] = __uint_as_float(wv[h] & 0xffff0000u);
    }
  }
}
// One M=64 N=64 K=64 MMA: D (+)= A B with A, B given by their tile base addresses and major-ness.
__device__ __forceinline__ void mma64(uint32_t d, uint32_t a, int a_mn, uint32_t b, int b_mn, uint32_t acc,
                                      int neg_a = 0) {
  const uint32_t idesc = idesc_bf16(64, 64, a_mn, b_mn) | ((uint32_t)neg_a << 13);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    const uint32_t ao = a_mn ? 2048u * kk : 32u * kk;
    const uint32_t bo = b_mn ? 2048u * kk : 32u * kk;
    mma_ss(d, sdesc_sw128(a + ao, 1024, a_mn ? 0 : 16), sdesc_sw128(b + bo, 1024, b_mn ? 0 : 16), idesc,
           (acc || kk > 0) ? 1u : 0u);
  }
}
// Loads this thread's 64-column row of an M=64 accumulator at TMEM column col.
__device__ __forceinline__ void ld_row(uint32_t tb, uint32_t lane_off, uint32_t col, float* x) {
  uint32_t a[32], b[32];
  tmem_ld32(tb + lane_off + col, a);
  tmem_ld32(tb + lane_off + col + 32, b);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) {
    x[j] = __uint_as_float(a[j]);
    x[32 + j] = __uint_as_float(b[j]);
  }
}

// Half rows: 32 columns (half h) of row r of a swizzled bf16 tile.
__device__ __forceinline__ void put_half(uint8_t* tile, int r, int h, const float* x) {
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    uint4 pk;
    pk.x = pack_bf16(x[8 * q], x[8 * q + 1]);
    pk.y = pack_bf16(x[8 * q + 2], x[8 * q + 3]);
    pk.z = pack_bf16(x[8 * q + 4], x[8 * q + 5]);
    pk.w = pack_bf16(x[8 * q + 6], x[8 * q + 7]);
    *reinterpret_cast<uint4*>(row + (((4 * h + q) ^ (r & 7)) * 16)) = pk;
  }
}
__device__ __forceinline__ void get_half(const uint8_t* tile, int r, int h, float* x) {
  const uint8_t* row = tile + r * 128;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 pk = *reinterpret_cast<const uint4*>(row + (((4 * h + q) ^ (r & 7)) * 16));
    const uint32_t wv[4] = {pk.x, pk.y, pk.z, pk.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      x[8 * q + 2 * e] = __uint_as_float(wv[e] << 16);
      x[8 * q + 2 * e + 1] = __uint_as_float(wv[e] & 0xffff0000u);
    }
  }
}
// This thread's half row of an M=64 accumulator at TMEM column col: row 16 * warp + lane % 16,
// columns col + 32 * (lane / 16) .. + 31.
__device__ __forceinline__ void ld_half(uint32_t tb, uint32_t lane_off, uint32_t col, float* x) {
  uint32_t a[32];
  tmem_ld16x2(tb + lane_off + col, a);
  tmem_ld_wait();
#pragma unroll
  for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(a[j]);
}

}  // namespace tc
}  // namespace pathattn
