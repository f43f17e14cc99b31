// tcgen05 forward scan of PaTH attention at head dim 128 (bf16 operands, fp32 accumulation in TMEM).
//
// Method: the right-to-left chunk scan of the PaTH reading notes (cc.laoqi.cc/papers/2505.16381),
// §2.7, as at head dim 64: for a query tile, Z starts at the boundary-adjusted queries Q<-; for
// each earlier key chunk c (right to left) the scores are Z K->_c^T, the online softmax
// accumulates P V_c, and Z <- Z F_c^T carries the queries across chunk c (F_c is 128 x 128).
//
// GB300 mapping (one CTA = one 128-row query tile = two 64-row UT chunks; one CTA per SM: its
// TMEM plan needs more than half of the 512 columns):
//   * every head-dim-wide operand is split into column halves x = a, b (0-63, 64-127), each a
//     128-byte swizzled atom; a stage holds, per half, K->_c (64 rows) stacked over F_c (128 rows)
//     and the half of V_c;
//   * warp 9 issues the MMAs with the A operands in TMEM: one N=192 MMA per 16-wide slice of the
//     head dim gives S = Z K->_c^T and Z' = Z F_c^T together (K = 128: eight slices, the first four
//     from half a, the last four from half b), and O += P V_c runs as two N=64 MMAs (V halves read
//     MN-major);
//   * warp 8 streams the stages with TMA (a 3-stage ring) and the Q<- tile, whose buffer is the
//     third stage's (the ring's third load waits until the softmax threads have moved Q<- to TMEM);
//   * warps 0-7 run the softmax, two threads per query row (TMEM lane): the thread of column half h
//     takes S columns 32h..32h+31, Z' and O columns 64h..64h+63 and the matching Z and P words.
//     Each step it first turns its half of Z' into bf16 Z (TMEM to registers to TMEM), then reads
//     its half of S and runs the online softmax (lazy rescaling of O above a threshold of 8 in
//     log2 units, as at head dim 64).
// TMEM: S 0-63, Z' 64-191 (the N=192 accumulator), O 192-319, Z 320-383 (bf16 pairs), P 384-415.
#include "internal.h"
#include "dev_common.cuh"
#include "tc_common.cuh"
#include "scan_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace pathattn {

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();  // fwd_tc.cu

namespace {
using namespace tc;

constexpr int BQ = 128;
constexpr int BK = 64;
constexpr int D = kHeadDimWide;
constexpr int NSTAGE = 3;
constexpr int NSOFT = 256;  // softmax threads: two per query row
constexpr int NTHREADS = NSOFT + 64;
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S = 0, COL_ZP = 64, COL_O = 192, COL_Z = 320, COL_P = 384;
constexpr uint32_t KF_BYTES = 192 * 128;  // one half of a stage: K->_c (8 KB) over F_c (16 KB)
constexpr float kTau = 8.f;               // lazy-rescale threshold (log2 units)

struct __align__(1024) Scan128Smem {
  uint8_t kf[NSTAGE][2][KF_BYTES];  // per stage and column half: K->_c rows 0-63, F_c rows 64-191;
                                    // stage 2 first holds the Q<- tile (two 16 KB halves)
  uint8_t v[NSTAGE][2][BK * 128];   // V_c column halves
  float xm[2][BQ];                  // per-half row maxima / sums exchanged between the halves
  float frs[NSTAGE][BK];            // PaTH-FoX: the chunk's suffix sums of log f
  uint64_t full[NSTAGE], empty[NSTAGE];
  uint64_t z_init, z0_free, z_ready, s_full, p_ready, pv_done, o_done;
  uint32_t tmem_base;
};

struct Scan128Params {
  int L, Lp, nc, BH, ntiles;
  float scl;  // scale * log2(e)
  const float* dm;  // diagonal-chunk softmax state from the preparation
  const float* dl;
  const float* dacc;  // [BH][Lp][128]
  const float* fa;
  const float* fr;
  const float* ft;
  __nv_bfloat16* o;
  float* lse;
  int* err;
};


template <bool FOX>
__global__ void __launch_bounds__(NTHREADS, 1)
    fwd_scan128_tc_kernel(const __grid_constant__ CUtensorMap tm_ql, const __grid_constant__ CUtensorMap tm_kr,
                          const __grid_constant__ CUtensorMap tm_f, const __grid_constant__ CUtensorMap tm_v,
                          const Scan128Params p) {
  extern __shared__ uint8_t smem_raw[];
  Scan128Smem& s = *reinterpret_cast<Scan128Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int err0 = threadIdx.x == 0 ? peek_err(p.err) : 0;  // consumed at the setup barrier
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bh, T;
  tile_of_block((int)blockIdx.x, p.ntiles, p.BH, bh, T);
  const bool has_partial = (2 * T + 1) * BK < p.L;
  const int nsteps = (has_partial ? 1 : 0) + 2 * T;
  auto step_chunk = [&](int n) { return has_partial ? 2 * T - n : 2 * T - 1 - n; };

  if (tid == 0) {
    for (int k = 0; k < NSTAGE; ++k) {
      mbar_init(&s.full[k], 1);
      mbar_init(&s.empty[k], 1);
    }
    mbar_init(&s.z_init, 1);
    mbar_init(&s.z0_free, NSOFT);
    mbar_init(&s.z_ready, NSOFT);
    mbar_init(&s.s_full, 1);
    mbar_init(&s.p_ready, NSOFT);
    mbar_init(&s.pv_done, 1);
    mbar_init(&s.o_done, 1);
    fence_barrier_init();
  }
  if (warp == 9) tmem_alloc(&s.tmem_base, TMEM_COLS);
  tc_fence_before();
  // a wait of an earlier CTA of the launch has given up: end at once (the pipeline is broken)
  const bool launch_err = __syncthreads_or(err0 != 0) != 0;
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  if (launch_err) {
    if (warp == 9) tmem_dealloc(tb, TMEM_COLS);
    return;
  }

  if (warp == 8) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && nsteps > 0) {
      prefetch_tmap(&tm_ql);
      prefetch_tmap(&tm_kr);
      prefetch_tmap(&tm_f);
      prefetch_tmap(&tm_v);
      // Q<- of the tile (both column halves) into the third stage's buffer
      mbar_arrive_expect_tx(&s.z_init, 2 * BQ * 128);
      tma_load_2d(s.kf[NSTAGE - 1][0], &tm_ql, 0, bh * p.Lp + T * BQ, &s.z_init);
      tma_load_2d(s.kf[NSTAGE - 1][1], &tm_ql, 64, bh * p.Lp + T * BQ, &s.z_init);
      for (int n = 0; n < nsteps; ++n) {
        const int st = n % NSTAGE;
        if (n >= NSTAGE && !mbar_wait(&s.empty[st], ((n / NSTAGE) - 1) & 1, p.err, 1)) break;
        if (n == NSTAGE - 1) {  // the softmax threads have moved Q<- into TMEM
          if (!mbar_wait(&s.z0_free, 0, p.err, 12)) break;
          fence_proxy_async_smem();
        }
        const int c = step_chunk(n);
        mbar_arrive_expect_tx(&s.full[st], 2 * KF_BYTES + 2 * BK * 128 + (FOX ? BK * 4 : 0));
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          tma_load_2d(s.kf[st][x], &tm_kr, 64 * x, bh * p.Lp + c * BK, &s.full[st]);
          tma_load_2d(s.kf[st][x] + BK * 128, &tm_f, 64 * x, (bh * p.nc + c) * D, &s.full[st]);
          tma_load_2d(s.v[st][x], &tm_v, 64 * x, bh * p.L + c * BK, &s.full[st]);
        }
        if constexpr (FOX) bulk_load(s.frs[st], p.fr + (size_t)bh * p.Lp + (size_t)c * BK, BK * 4, &s.full[st]);
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    // order: S(n), Z'(n) once Z(n) is in TMEM and S(n-1), Z'(n-1) have been read; then
    // O += P(n-1) V(n-1) once P(n-1) is written.
    if (lane == 0 && nsteps > 0) {
      // S and Z' from one N=192 MMA per 16-wide slice of the head dim (B = [K->_c; F_c] of that
      // half); O += P V_c as two N=64 MMAs, one per V half (MN-major)
      const uint32_t idesc_sz = idesc_bf16(128, 192, 0, 0);
      const uint32_t idesc_pv = idesc_bf16(128, 64, 0, 1);
      bool ok = true;
      auto issue_pv = [&](int m) {
        const int st = m % NSTAGE;
#pragma unroll
        for (int x = 0; x < 2; ++x) {
          const uint32_t vb = smem_u32(s.v[st][x]);
#pragma unroll
          for (int k = 0; k < 4; ++k)
            mma_ts(tb + COL_O + 64 * x, tb + COL_P + 8 * k, sdesc_sw128(vb + 2048u * k, 1024, 0), idesc_pv, 1);
        }
        mma_commit(&s.empty[st]);
        mma_commit(&s.pv_done);
      };
      for (int n = 0; ok && n < nsteps; ++n) {
        const int st = n % NSTAGE;
        if (!mbar_wait(&s.full[st], (n / NSTAGE) & 1, p.err, 3)) { ok = false; break; }
        if (!mbar_wait(&s.z_ready, n & 1, p.err, 4)) { ok = false; break; }
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t bd = sdesc_sw128(smem_u32(s.kf[st][kk >> 2]) + 32u * (kk & 3), 1024, 16);
          mma_ts(tb + COL_S, tb + COL_Z + 8 * kk, bd, idesc_sz, kk > 0 ? 1u : 0u);
        }
        mma_commit(&s.s_full);
        if (n > 0) {
          if (!mbar_wait(&s.p_ready, (n - 1) & 1, p.err, 5)) { ok = false; break; }
          tc_fence_after();
          issue_pv(n - 1);
        }
      }
      if (ok && mbar_wait(&s.p_ready, (nsteps - 1) & 1, p.err, 5)) {
        tc_fence_after();
        issue_pv(nsteps - 1);
        mma_commit(&s.o_done);
      }
    }
  } else {
    // ---------------- softmax / transport: thread (r, h) owns S columns 32h.., Z' and O columns 64h.. ----------------
    const int q4 = warp & 3, h = warp >> 2;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t c_s = tb + lane_off + COL_S + 32 * h, c_zp = tb + lane_off + COL_ZP + 64 * h;
    const uint32_t c_o = tb + lane_off + COL_O + 64 * h, c_p = tb + lane_off + COL_P + 16 * h;
    const uint32_t c_z = tb + lane_off + COL_Z + 32 * h;
    const int grow = T * BQ + r;
    const size_t wrow = (size_t)bh * p.Lp + (size_t)T * BQ + r;
    float m = p.dm[wrow], l = h == 0 ? p.dl[wrow] : 0.f;  // l: this half's share of the row sum
    uint32_t x[32];
    bool ok = true;
    if (nsteps > 0) {
#pragma unroll
      for (int u = 0; u < 2; ++u) {  // O = the diagonal chunk's accumulator
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __float_as_uint(p.dacc[wrow * D + 64 * h + 32 * u + j]);
        tmem_st32(c_o + 32 * u, x);
      }
      // Z_0 = Q<- of the tile: column half h of row r, shared memory (swizzled) -> TMEM
      ok = mbar_wait(&s.z_init, 0, p.err, 2);  // (on a timeout the tile below is garbage; err is set)
      const uint8_t* zrow = s.kf[NSTAGE - 1][h] + r * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(zrow + ((q ^ (r & 7)) * 16));
        x[4 * q] = v.x;
        x[4 * q + 1] = v.y;
        x[4 * q + 2] = v.z;
        x[4 * q + 3] = v.w;
      }
      tmem_st32(c_z, x);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.z0_free);  // its buffer may take the third stage
      mbar_arrive(&s.z_ready);
    }
    const float arow = FOX ? p.fa[wrow] : 0.f;
    float R = 0.f;
    // Every softmax thread runs every step (the per-step barrier needs all of them); after a
    // wait has timed out (error recorded) the remaining waits are skipped.
    for (int n = 0; n < nsteps; ++n) {
      ok = ok && mbar_wait(&s.s_full, n & 1, p.err, 6);
      tc_fence_after();
      const int c = step_chunk(n);
      const bool active = !(has_partial && n == 0 && r < 64);
      // transport first: Z <- bf16(Z F_c^T) into TMEM, so that the next MMAs can start (rows not
      // transported at the partial step keep Z_0)
      if (n + 1 < nsteps && active) {
        uint32_t zb[32];
        tmem_ld32(c_zp, x);
        tmem_ld32(c_zp + 32, zb);
        tmem_ld_wait();
        uint32_t z32[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          z32[j] = pack_bf16(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
          z32[16 + j] = pack_bf16(__uint_as_float(zb[2 * j]), __uint_as_float(zb[2 * j + 1]));
        }
        tmem_st32(c_z, z32);
      }
      tmem_ld32(c_s, x);
      tmem_ld_wait();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.z_ready);  // Z(n+1) written, S(n) and Z'(n) read
      // this half's maximum of the log2-domain scores x = scl s (+ forget-gate terms); without a
      // forget gate x is a plain multiple of the raw score, so its maximum comes from the raw
      // maximum (minimum for a negative scale) and x itself is folded into the exponent below
      float mxh;
      uint64_t v2[FOX ? 16 : 1];  // FoX: the biased log2-domain scores, key pairs (kept packed)
      if constexpr (FOX) {
        // the keys' suffix sums came with the chunk's stage (its barrier completed before S was
        // issued; the stage is refilled only after this step's P V)
        ok = ok && mbar_wait(&s.full[n % NSTAGE], (n / NSTAGE) & 1, p.err, 11);
        const float rb = (arow + R) * kLog2e;
        const uint64_t rb2 = f2(rb, rb), l2e2 = f2(kLog2e, kLog2e), sc2 = f2(p.scl, p.scl);
        const ulonglong2* f4 = reinterpret_cast<const ulonglong2*>(s.frs[n % NSTAGE] + 32 * h);
        float e0 = -INFINITY, e1 = -INFINITY;
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const ulonglong2 fv = f4[q];
          v2[2 * q] = f2_fma(f2(__uint_as_float(x[4 * q]), __uint_as_float(x[4 * q + 1])), sc2,
                             f2_fma(fv.x, l2e2, rb2));
          v2[2 * q + 1] = f2_fma(f2(__uint_as_float(x[4 * q + 2]), __uint_as_float(x[4 * q + 3])), sc2,
                                 f2_fma(fv.y, l2e2, rb2));
          float a0, a1, a2, a3;
          f2_split(v2[2 * q], a0, a1);
          f2_split(v2[2 * q + 1], a2, a3);
          e0 = max3(e0, a0, a1);
          e1 = max3(e1, a2, a3);
        }
        mxh = fmaxf(e0, e1);
      } else {
        float e0, e1;
        if (p.scl >= 0.f) {
          e0 = e1 = -INFINITY;
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            e0 = max3(e0, __uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
            e1 = max3(e1, __uint_as_float(x[2 * j + 2]), __uint_as_float(x[2 * j + 3]));
          }
          mxh = fmaxf(e0, e1) * p.scl;
        } else {
          e0 = e1 = INFINITY;
#pragma unroll
          for (int j = 0; j < 16; j += 2) {
            e0 = min3(e0, __uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
            e1 = min3(e1, __uint_as_float(x[2 * j + 2]), __uint_as_float(x[2 * j + 3]));
          }
          mxh = fminf(e0, e1) * p.scl;
        }
      }
      if (!active) mxh = -INFINITY;
      if (softmax_any(mxh > m + kTau)) {
        // some row needs a larger reference: the halves agree on the row maximum first
        s.xm[h][r] = mxh;
        softmax_sync();
        const float mnew = fmaxf(m, fmaxf(s.xm[0][r], s.xm[1][r]));
        softmax_sync();
        // the TMEM loads and stores of O are warp-wide instructions: a warp with any row to
        // rescale rescales all 32 of its rows, by 1 where the reference stays
        const bool resc = mnew > m + kTau;
        if (__any_sync(0xffffffffu, resc)) {
          // O holds P(n-1) V(n-1) only once that MMA has completed
          if (n > 0) ok = ok && mbar_wait(&s.pv_done, (n - 1) & 1, p.err, 8);
          tc_fence_after();
          const float corr = resc ? fast_exp2(m - mnew) : 1.f;
          if (resc) {
            m = mnew;
            l *= corr;
          }
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            uint32_t ob[32];
            tmem_ld32(c_o + 32 * u, ob);
            tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) ob[j] = __float_as_uint(__uint_as_float(ob[j]) * corr);
            tmem_st32(c_o + 32 * u, ob);
          }
        }
      }
      // probabilities, packed bf16 pairs (key 2j in the low half); exponents and row sums by
      // paired fp32 instructions
      uint32_t pk[16];
      if (active) {
        uint64_t acc[2] = {0ull, 0ull};
        const uint64_t nm = f2(-m, -m), sc = f2(p.scl, p.scl);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float a0, a1;
          if constexpr (FOX) {
            f2_split(f2_add(v2[j], nm), a0, a1);
          } else {
            f2_split(f2_fma(f2(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1])), sc, nm), a0, a1);
          }
          const float p0 = fast_exp2(a0), p1 = fast_exp2(a1);
          acc[j & 1] = f2_add(acc[j & 1], f2(p0, p1));
          pk[j] = pack_bf16(p0, p1);
        }
        float s0, s1, s2, s3;
        f2_split(acc[0], s0, s1);
        f2_split(acc[1], s2, s3);
        l += (s0 + s1) + (s2 + s3);
        if (FOX) R += p.ft[(size_t)bh * p.nc + c];
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = 0u;
      }
      // P(n-1) has been consumed by its MMAs before P(n) replaces it
      if (n > 0) ok = ok && mbar_wait(&s.pv_done, (n - 1) & 1, p.err, 9);
      tmem_st16(c_p, pk);
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_ready);
    }
    // ---------------- epilogue ----------------
    if (nsteps > 0) {
      if (ok) ok = mbar_wait(&s.o_done, 0, p.err, 7);
      tc_fence_after();
    }
    s.xm[h][r] = l;
    softmax_sync();
    const float lt = s.xm[0][r] + s.xm[1][r];
    const float inv = 1.f / lt;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      if (nsteps > 0) {
        tmem_ld32(c_o + 32 * u, x);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __float_as_uint(p.dacc[wrow * D + 64 * h + 32 * u + j]);
      }
      if (grow < p.L) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)bh * p.L + grow) * D + 64 * h + 32 * u);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 pkv;
          pkv.x = pack_bf16(__uint_as_float(x[8 * q]) * inv, __uint_as_float(x[8 * q + 1]) * inv);
          pkv.y = pack_bf16(__uint_as_float(x[8 * q + 2]) * inv, __uint_as_float(x[8 * q + 3]) * inv);
          pkv.z = pack_bf16(__uint_as_float(x[8 * q + 4]) * inv, __uint_as_float(x[8 * q + 5]) * inv);
          pkv.w = pack_bf16(__uint_as_float(x[8 * q + 6]) * inv, __uint_as_float(x[8 * q + 7]) * inv);
          dst[q] = pkv;
        }
      }
    }
    if (h == 0 && grow < p.L) p.lse[(size_t)bh * p.L + grow] = (m + log2f(lt)) * kLn2;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tb, TMEM_COLS);
  }
}

}  // namespace
}  // namespace pathattn

namespace pathattn {

// 2-D map over a [rows][128] bf16 matrix seen in 128-byte swizzled boxes of box_rows x 64 (one
// column half; x = 0 or 64).
bool make_map_rows128(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [heads][L][128] bf16 tensor seen in 64-row x 64-column boxes of one head (x = 0 or 64); rows
// >= L read as zero.
bool make_map_head_rows128(CUtensorMap* m, const void* base, uint64_t L, uint64_t heads) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {128, L, heads};
  cuuint64_t strides[2] = {256, L * 256};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_scan128_tc(const Geom& g, const void* v, const float* logf, char* ws, const FwdWs& lay, void* o,
                              float* lse, cudaStream_t st) {
  if (g.B != BK || g.D != D || (g.nc & 1) || g.Lp != g.nc * BK) return cudaErrorInvalidValue;
  CUtensorMap m_ql, m_kr, m_f, m_v;
  const uint64_t prow = (uint64_t)g.BH * g.Lp;
  if (!make_map_rows128(&m_ql, ws + lay.ql, prow, BQ) || !make_map_rows128(&m_kr, ws + lay.kr, prow, BK) ||
      !make_map_rows128(&m_f, ws + lay.f, (uint64_t)g.BH * g.nc * D, D) ||
      !make_map_rows128(&m_v, v, (uint64_t)g.BH * g.L, BK))
    return cudaErrorInvalidValue;
  Scan128Params p;
  p.L = g.L;
  p.Lp = g.Lp;
  p.nc = g.nc;
  p.BH = g.BH;
  p.ntiles = g.nc / 2;
  p.scl = g.scale * kLog2e;
  p.dm = (const float*)(ws + lay.dm);
  p.dl = (const float*)(ws + lay.dl);
  p.dacc = (const float*)(ws + lay.dacc);
  p.fa = (const float*)(ws + lay.fa);
  p.fr = (const float*)(ws + lay.fr);
  p.ft = (const float*)(ws + lay.ft);
  p.o = (__nv_bfloat16*)o;
  p.lse = lse;
  p.err = (int*)(ws + lay.err);
  const size_t smem = sizeof(Scan128Smem) + 1024;
  auto kern = logf ? fwd_scan128_tc_kernel<true> : fwd_scan128_tc_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long ntiles = (long)p.ntiles * g.BH;
  kern<<<(unsigned)ntiles, NTHREADS, smem, st>>>(m_ql, m_kr, m_f, m_v, p);
  return cudaGetLastError();
}

}  // namespace pathattn
