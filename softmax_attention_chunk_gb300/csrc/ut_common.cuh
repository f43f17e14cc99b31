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
// fp32 64x64 matrix over two adjacent tile slots, element (r, m) at r * 64 + (m ^ 4 (r mod 8)):
// rows of a warp's 16-byte stores fall on different banks, 4-column groups stay contiguous.
__device__ __forceinline__ int f32_idx(int r, int m) { return r * 64 + (m ^ ((r & 7) << 2)); }

// Coalesced conversion of fp32 rows [64 columns] into a swizzled bf16 tile by the threads of
// NW warps: warp w takes rows w * (64 / NW) ..; each warp-wide 16-byte load covers two whole rows
// (lane l: row + l / 16, columns 4 (l % 16) .. + 3), all loads are issued before the first
// store, and each thread stores its four values as one 8-byte piece of the tile row.  Rows >= nvalid
// are stored as zero.  load() and store() are separate so that a caller can wait in between.
template <int NW>
struct RowsToTile {
  static constexpr int kLoads = 32 / NW;  // loads per thread (two rows each)
  float4 v[kLoads];
  __device__ __forceinline__ void load(const float* src, int nvalid, int w, int lane) {
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
      const int r = w * (64 / NW) + 2 * k + (lane >> 4);
      v[k] = r < nvalid ? reinterpret_cast<const float4*>(src + (size_t)r * 64)[lane & 15]
                        : make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  __device__ __forceinline__ void store(uint8_t* tile, int w, int lane) const {
#pragma unroll
    for (int k = 0; k < kLoads; ++k) {
      const int r = w * (64 / NW) + 2 * k + (lane >> 4), col = 4 * (lane & 15);
      *reinterpret_cast<uint2*>(tile + sw128_offset(r, col)) =
          make_uint2(pack_bf16(v[k].x, v[k].y), pack_bf16(v[k].z, v[k].w));
    }
  }
};

// 32 fp32 values as bf16 to global memory (64 bytes, 16-byte aligned).
__device__ __forceinline__ void store_bf16_half(__nv_bfloat16* dst, const float* x) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 4; ++q)
    d4[q] = make_uint4(pack_bf16(x[8 * q], x[8 * q + 1]), pack_bf16(x[8 * q + 2], x[8 * q + 3]),
                       pack_bf16(x[8 * q + 4], x[8 * q + 5]), pack_bf16(x[8 * q + 6], x[8 * q + 7]));
}
// 32 fp32 values from global memory (128 bytes, 16-byte aligned).
__device__ __forceinline__ void load_f32_half(const float* src, float* x) {
  const float4* s4 = reinterpret_cast<const float4*>(src);
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 v = s4[q];
    x[4 * q] = v.x;
    x[4 * q + 1] = v.y;
    x[4 * q + 2] = v.z;
    x[4 * q + 3] = v.w;
  }
}

// Named barrier 2 over the 128 threads of a per-chunk UT kernel (the block-inversion routine
// below synchronises through it).
__device__ __forceinline__ void ut_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

// The block inversion of the UT transform: U = (I + L)^{-1} diag(beta) for one 64-row chunk, by
// two-level block inversion over the row halves t (0-31) and b (32-63):
//   (I + L)^{-1} = [[Y_tt, 0], [-Y_bb L_bt Y_tt, Y_bb]],  Y_tt = (I + L_tt)^{-1}, Y_bb = (I + L_bb)^{-1}.
// Phase 1: warp 0 solves the columns of Y_tt, warp 1 those of Y_bb (one column per thread, 32 rows
// by forward substitution, four partial sums per row).  Phase 2: all 128 threads form T = L_bt Y_tt
// (into the unused upper-right block of sl), then Y_bt = -Y_bb T, each thread a 2 x 4 block.
// sl: the fp32 L of the chunk (f32_idx layout over two tile slots, strictly lower; overwritten).
// ut_solve_blocked_t writes U transposed: U^T (and, LO, U_lo^T with U = U_hi + U_lo, both bf16)
// as swizzled bf16 tiles, so that a thread, which holds one column of a diagonal block, writes it
// as one contiguous tile row (four 16-byte stores instead of 32 scalar ones); Y is kept transposed
// in sl the same way (row j of a diagonal block = column j of Y), and phase 2 reads
//   T = L_bt Y_tt:   T[i][j] = sum_m L[32+i][m] Yt[j][m]   (rows of L against rows of Yt; each
//                    thread's columns interleaved, cg + 8 j, so that the eight Yt rows of a warp's
//                    load sit on eight different swizzle positions)
//   Y_bt = -Y_bb T:  Y_bt[i][j] = -sum_m Yt_bb[m][i] T[m][j]
// writing U^T rows j, columns 32 + i as bf16 pairs.  The MMAs read U^T with the opposite operand
// major-ness.  Called by threads 0-127 together; ends with the tiles written by generic stores
// (the caller fences them for the tensor core).
template <bool LO>
__device__ __forceinline__ void ut_solve_blocked_t(float* sl, const float* beta, uint8_t* ut, uint8_t* ut_lo,
                                                   int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  // ---- phase 1: diagonal 32 x 32 blocks ----
  float y[32];
  if (warp < 2) {
    const float* sh = sl + 65 * 32 * warp;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      float acc[16];
      if (b == 1) {
        uint64_t s2[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) s2[rr] = 0ull;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
          const uint64_t y01 = f2(y[m], y[m + 1]), y23 = f2(y[m + 2], y[m + 3]);
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            const ulonglong2 lv = *reinterpret_cast<const ulonglong2*>(sh + f32_idx(16 + rr, m));
            s2[rr] = f2_fma(lv.x, y01, s2[rr]);
            s2[rr] = f2_fma(lv.y, y23, s2[rr]);
          }
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          float lo, hi;
          f2_split(s2[rr], lo, hi);
          acc[rr] = lo + hi;
        }
      } else {
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) acc[rr] = 0.f;
      }
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) {
        const int r = 16 * b + rr;
        float a0 = acc[rr], a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int m = 16 * b; m < r; m += 4) {
          const float4 lv = *reinterpret_cast<const float4*>(sh + f32_idx(r, m));
          a0 = fmaf(lv.x, y[m], a0);
          if (m + 1 < r) a1 = fmaf(lv.y, y[m + 1], a1);
          if (m + 2 < r) a2 = fmaf(lv.z, y[m + 2], a2);
          if (m + 3 < r) a3 = fmaf(lv.w, y[m + 3], a3);
        }
        y[r] = (lane == r ? 1.f : 0.f) - ((a0 + a1) + (a2 + a3));
      }
    }
  }
  ut_sync();  // every read of L_tt / L_bb is done
  if (warp < 2) {
    const int o = 32 * warp, col = o + lane;
    const float bc = beta[col];
    // Yt row col (the column of Y), columns o .. o+31
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4*>(sl + f32_idx(col, o + 4 * q)) = make_float4(y[4 * q], y[4 * q + 1], y[4 * q + 2], y[4 * q + 3]);
    float uv[32];
#pragma unroll
    for (int r = 0; r < 32; ++r) uv[r] = y[r] * bc;
    put_half(ut, col, warp, uv);  // U^T row col, columns o .. o+31
    if constexpr (LO) {
#pragma unroll
      for (int r = 0; r < 32; ++r) uv[r] -= __bfloat162float(__float2bfloat16_rn(uv[r]));
      put_half(ut_lo, col, warp, uv);
    }
    if (warp == 1) {  // U^T rows 32-63, columns 0-31 (the zero upper-right block of U)
#pragma unroll
      for (int r = 0; r < 32; ++r) uv[r] = 0.f;
      put_half(ut, col, 0, uv);
      if constexpr (LO) put_half(ut_lo, col, 0, uv);
    }
  }
  ut_sync();
  // ---- phase 2: rows 2 rg, 2 rg + 1 and columns 4 cg .. 4 cg + 3 of a 32 x 32 product ----
  const int rg = tid >> 3, cg = tid & 7;
  float acc[2][4];
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[e][j] = 0.f;
  // T = L_bt Y_tt: rows 32 + 2 rg + e of L against rows cg + 8 j of Yt_tt (the eight rows a warp
  // reads in one load sit on eight different swizzle positions)
#pragma unroll
  for (int m = 0; m < 32; m += 4) {
    const float4 a0 = *reinterpret_cast<const float4*>(sl + f32_idx(32 + 2 * rg, m));
    const float4 a1 = *reinterpret_cast<const float4*>(sl + f32_idx(32 + 2 * rg + 1, m));
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float4 bv = *reinterpret_cast<const float4*>(sl + f32_idx(cg + 8 * j, m));
      acc[0][j] = fmaf(a0.x, bv.x, fmaf(a0.y, bv.y, fmaf(a0.z, bv.z, fmaf(a0.w, bv.w, acc[0][j]))));
      acc[1][j] = fmaf(a1.x, bv.x, fmaf(a1.y, bv.y, fmaf(a1.z, bv.z, fmaf(a1.w, bv.w, acc[1][j]))));
    }
  }
  // T into the unused upper-right block of sl (rows 0-31, columns 32-63)
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int j = 0; j < 4; ++j) sl[f32_idx(2 * rg + e, 32 + cg + 8 * j)] = acc[e][j];
  ut_sync();
  // Y_bt = -Y_bb T: Yt_bb rows m (columns 32 + 2 rg, + 1) times T rows m (columns 4 cg ..)
#pragma unroll
  for (int e = 0; e < 2; ++e)
#pragma unroll
    for (int j = 0; j < 4; ++j) acc[e][j] = 0.f;
#pragma unroll 8
  for (int m = 0; m < 32; ++m) {
    const float2 av = *reinterpret_cast<const float2*>(sl + f32_idx(32 + m, 32 + 2 * rg));
    const float4 bv = *reinterpret_cast<const float4*>(sl + f32_idx(m, 32 + 4 * cg));
    acc[0][0] = fmaf(av.x, bv.x, acc[0][0]);
    acc[0][1] = fmaf(av.x, bv.y, acc[0][1]);
    acc[0][2] = fmaf(av.x, bv.z, acc[0][2]);
    acc[0][3] = fmaf(av.x, bv.w, acc[0][3]);
    acc[1][0] = fmaf(av.y, bv.x, acc[1][0]);
    acc[1][1] = fmaf(av.y, bv.y, acc[1][1]);
    acc[1][2] = fmaf(av.y, bv.z, acc[1][2]);
    acc[1][3] = fmaf(av.y, bv.w, acc[1][3]);
  }
  // U[32 + i][j] = Y_bt[i][j] beta_j  ->  U^T row j, columns 32 + 2 rg, + 1 (a bf16 pair)
  const float4 bq = *reinterpret_cast<const float4*>(beta + 4 * cg);
  const float bv[4] = {bq.x, bq.y, bq.z, bq.w};
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    const float u0 = -acc[0][j] * bv[j], u1 = -acc[1][j] * bv[j];
    const int row = 4 * cg + j, colp = 32 + 2 * rg;
    *reinterpret_cast<uint32_t*>(ut + sw128_offset(row, colp)) = pack_bf16(u0, u1);
    if constexpr (LO) {
      const float l0 = u0 - __bfloat162float(__float2bfloat16_rn(u0));
      const float l1 = u1 - __bfloat162float(__float2bfloat16_rn(u1));
      *reinterpret_cast<uint32_t*>(ut_lo + sw128_offset(row, colp)) = pack_bf16(l0, l1);
    }
  }
}

// Named barrier 3 over threads 0-63 (warps 0-1).
__device__ __forceinline__ void ut_sync64() { asm volatile("bar.sync 3, 64;" ::: "memory"); }
// The same block inversion in two parts, U and Y stored untransposed, for a caller whose warps 2-3
// have their own work during the diagonal solves but are free for the off-diagonal products:
//   ut_inv_diag64 (warps 0-1, named barrier 3): Y_tt, Y_bb into sl and the tiles yt (Y) and u
//     (U = Y diag(beta)), the zero upper-right blocks included;
//   ut_inv_offdiag128 (all 128 threads, after a barrier that makes ut_inv_diag64's stores
//     visible): T = L_bt Y_tt, then Y_bt = -Y_bb T into yt and u; rows 2 rg, 2 rg + 1 and columns
//     4 cg .. 4 cg + 3 of each 32 x 32 product per thread.
__device__ __forceinline__ void ut_inv_diag64(float* sl, const float* beta, uint8_t* u, uint8_t* yt, int tid) {
  const int warp = tid >> 5, lane = tid & 31;
  float y[32];
  {
    const float* sh = sl + 65 * 32 * warp;
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      float acc[16];
      if (b == 1) {
        uint64_t s2[16];
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) s2[rr] = 0ull;
#pragma unroll
        for (int m = 0; m < 16; m += 4) {
          const uint64_t y01 = f2(y[m], y[m + 1]), y23 = f2(y[m + 2], y[m + 3]);
#pragma unroll
          for (int rr = 0; rr < 16; ++rr) {
            const ulonglong2 lv = *reinterpret_cast<const ulonglong2*>(sh + f32_idx(16 + rr, m));
            s2[rr] = f2_fma(lv.x, y01, s2[rr]);
            s2[rr] = f2_fma(lv.y, y23, s2[rr]);
          }
        }
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) {
          float lo, hi;
          f2_split(s2[rr], lo, hi);
          acc[rr] = lo + hi;
        }
      } else {
#pragma unroll
        for (int rr = 0; rr < 16; ++rr) acc[rr] = 0.f;
      }
#pragma unroll
      for (int rr = 0; rr < 16; ++rr) {
        const int r = 16 * b + rr;
        float a0 = acc[rr], a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
        for (int m = 16 * b; m < r; m += 4) {
          const float4 lv = *reinterpret_cast<const float4*>(sh + f32_idx(r, m));
          a0 = fmaf(lv.x, y[m], a0);
          if (m + 1 < r) a1 = fmaf(lv.y, y[m + 1], a1);
          if (m + 2 < r) a2 = fmaf(lv.z, y[m + 2], a2);
          if (m + 3 < r) a3 = fmaf(lv.w, y[m + 3], a3);
        }
        y[r] = (lane == r ? 1.f : 0.f) - ((a0 + a1) + (a2 + a3));
      }
    }
  }
  ut_sync64();  // every read of L_tt / L_bb is done
  const int o = 32 * warp, col = o + lane;
  const float bc = beta[col];
#pragma unroll
  for (int r = 0; r < 32; ++r) {
    sl[65 * o + f32_idx(r, lane)] = y[r];
    *reinterpret_cast<__nv_bfloat16*>(yt + sw128_offset(o + r, col)) = __float2bfloat16_rn(y[r]);
    *reinterpret_cast<__nv_bfloat16*>(u + sw128_offset(o + r, col)) = __float2bfloat16_rn(y[r] * bc);
  }
  if (warp == 1) {  // the upper-right blocks of Y and U are zero
#pragma unroll
    for (int r = 0; r < 32; ++r) {
      *reinterpret_cast<__nv_bfloat16*>(yt + sw128_offset(r, col)) = __float2bfloat16_rn(0.f);
      *reinterpret_cast<__nv_bfloat16*>(u + sw128_offset(r, col)) = __float2bfloat16_rn(0.f);
    }
  }
}

__device__ __forceinline__ void ut_inv_offdiag128(float* sl, const float* beta, uint8_t* u, uint8_t* yt, int tid) {
  const int rg = tid >> 3, cg = tid & 7;
  float acc[2][4];
  auto product = [&](int a_row0, int a_col0, int b_row0, int b_col0) {
#pragma unroll
    for (int e = 0; e < 2; ++e)
#pragma unroll
      for (int j = 0; j < 4; ++j) acc[e][j] = 0.f;
#pragma unroll
    for (int m = 0; m < 32; m += 4) {
      const float4 a0 = *reinterpret_cast<const float4*>(sl + f32_idx(a_row0 + 2 * rg, a_col0 + m));
      const float4 a1 = *reinterpret_cast<const float4*>(sl + f32_idx(a_row0 + 2 * rg + 1, a_col0 + m));
      const float av0[4] = {a0.x, a0.y, a0.z, a0.w}, av1[4] = {a1.x, a1.y, a1.z, a1.w};
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const float4 bv = *reinterpret_cast<const float4*>(sl + f32_idx(b_row0 + m + kk, b_col0 + 4 * cg));
        acc[0][0] = fmaf(av0[kk], bv.x, acc[0][0]);
        acc[0][1] = fmaf(av0[kk], bv.y, acc[0][1]);
        acc[0][2] = fmaf(av0[kk], bv.z, acc[0][2]);
        acc[0][3] = fmaf(av0[kk], bv.w, acc[0][3]);
        acc[1][0] = fmaf(av1[kk], bv.x, acc[1][0]);
        acc[1][1] = fmaf(av1[kk], bv.y, acc[1][1]);
        acc[1][2] = fmaf(av1[kk], bv.z, acc[1][2]);
        acc[1][3] = fmaf(av1[kk], bv.w, acc[1][3]);
      }
    }
  };
  product(32, 0, 0, 0);  // T = L_bt Y_tt, into the unused upper-right block of sl
#pragma unroll
  for (int e = 0; e < 2; ++e)
    *reinterpret_cast<float4*>(sl + f32_idx(2 * rg + e, 32 + 4 * cg)) =
        make_float4(acc[e][0], acc[e][1], acc[e][2], acc[e][3]);
  ut_sync();
  product(32, 32, 0, 32);  // Y_bb T
  const float4 bq = *reinterpret_cast<const float4*>(beta + 4 * cg);
  const float bv[4] = {bq.x, bq.y, bq.z, bq.w};
#pragma unroll
  for (int e = 0; e < 2; ++e) {
    const int r = 32 + 2 * rg + e;
#pragma unroll
    for (int j = 0; j < 4; j += 2) {  // bf16 pairs of columns 4 cg + j, + 1
      const int cj = 4 * cg + j;
      *reinterpret_cast<uint32_t*>(yt + sw128_offset(r, cj)) = pack_bf16(-acc[e][j], -acc[e][j + 1]);
      *reinterpret_cast<uint32_t*>(u + sw128_offset(r, cj)) = pack_bf16(-acc[e][j] * bv[j], -acc[e][j + 1] * bv[j + 1]);
    }
  }
}


}  // namespace tc
}  // namespace pathattn
