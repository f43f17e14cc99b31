// Tensor-core backward of PaTH attention (bf16 operands, fp32 accumulation).
//
// The pages give no backward; this is the exact derivative of the blockwise forward of the
// PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.6–§2.7, on 128-row query tiles and
// 64-row key chunks.  For query tile T the forward visits key chunks c_0 > c_1 > ... with the
// transported queries Z_0 = Q<-_T, Z_{n+1} = Z_n F_{c_n}^T.  The backward
//   1. (zchain) recomputes and stores every Z_n of every tile (bf16, swizzled 128x64 images);
//   2. (scan) walks the steps in reverse (ascending c) with G_{nsteps} = 0:
//        P = exp(scale Z_n K->_c^T - lse), dP = dO V_c^T, dS = scale P (dP - D)
//        dV_c += P^T dO,  dK->_c += dS^T Z_n,  dF_c += G_{n+1}^T Z_n,
//        G_n = dS K->_c + G_{n+1} F_c,     dQ<-_T = G_0,
//      the chunk sums dV, dK->, dF being added across tiles with TMA tensor fp32 reductions;
//   3. (finish) the per-chunk UT backward (ut_bwd_tc.cu) adds the diagonal chunk and takes
//      dQ<-, dK->, dF back to q, k, w, beta.
#include "internal.h"
#include "dev_common.cuh"
#include "tc_common.cuh"
#include "ut_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace pathattn {

bool make_map_rows64(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows);  // fwd_tc.cu
bool make_map_f32_rows64(CUtensorMap* m, const void* base, uint64_t rows);                 // fwd_tc.cu

namespace {
using namespace tc;

constexpr int BQ = 128;
constexpr int BK = 64;
constexpr int D = kHeadDim;
constexpr uint32_t ZTILE = BQ * 128;  // bytes of one 128x64 bf16 tile

__device__ __forceinline__ void wg_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ int step_chunk(bool has_partial, int T, int n) {
  return has_partial ? 2 * T - n : 2 * T - 1 - n;
}

// ============================ Z chain ============================
constexpr int ZC_NSTAGE = 3;
struct __align__(1024) ZcSmem {
  uint8_t z[2][ZTILE];
  uint8_t f[ZC_NSTAGE][BK * 128];
  uint64_t full[ZC_NSTAGE], empty[ZC_NSTAGE];
  uint64_t z_init, z_ready, zp_full;
  uint32_t tmem_base;
};

struct ZcParams {
  int L, Lp, nc, BH, ntiles;
  uint8_t* zs;
  int* err;
};

__global__ void __launch_bounds__(160) zchain_tc_kernel(const __grid_constant__ CUtensorMap tm_ql,
                                                        const __grid_constant__ CUtensorMap tm_f,
                                                        const ZcParams p) {
  extern __shared__ uint8_t smem_raw[];
  ZcSmem& s = *reinterpret_cast<ZcSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int err0 = threadIdx.x == 0 ? peek_err(p.err) : 0;  // consumed at the setup barrier
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bh, T;
  tile_of_block((int)blockIdx.x, p.ntiles, p.BH, bh, T);
  const bool has_partial = (2 * T + 1) * BK < p.L;
  const int nsteps = (has_partial ? 1 : 0) + 2 * T;
  uint8_t* zbase = p.zs + ((size_t)bh * p.ntiles * p.ntiles + (size_t)T * T) * ZTILE;
  if (nsteps == 0) return;

  if (tid == 0) {
    for (int k = 0; k < ZC_NSTAGE; ++k) {
      mbar_init(&s.full[k], 1);
      mbar_init(&s.empty[k], 1);
    }
    mbar_init(&s.z_init, 1);
    mbar_init(&s.z_ready, 1);
    mbar_init(&s.zp_full, 1);
    fence_barrier_init();
  }
  if (warp == 4) tmem_alloc(&s.tmem_base, 64);
  tc_fence_before();
  // a wait of an earlier CTA of the launch has given up: end at once (the pipeline is broken)
  const bool launch_err = __syncthreads_or(err0 != 0) != 0;
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  if (launch_err) {
    if (warp == 4) tmem_dealloc(tb, 64);
    return;
  }

  if (warp == 4) {
    if (lane == 0) {
      mbar_arrive_expect_tx(&s.z_init, ZTILE);
      tma_load_2d(s.z[0], &tm_ql, 0, bh * p.Lp + T * BQ, &s.z_init);
      const int nmma = nsteps - 1;
      for (int m = 0; m < nmma && m < ZC_NSTAGE; ++m) {
        mbar_arrive_expect_tx(&s.full[m], BK * 128);
        tma_load_2d(s.f[m], &tm_f, 0, (bh * p.nc + step_chunk(has_partial, T, m)) * D, &s.full[m]);
      }
      const uint32_t idesc = idesc_bf16(128, 64, 0, 0);
      for (int n = 0; n < nmma; ++n) {
        const int st = n % ZC_NSTAGE;
        if (!mbar_wait(&s.full[st], (n / ZC_NSTAGE) & 1, p.err, 11)) break;
        if (!mbar_wait(&s.z_ready, n & 1, p.err, 12)) break;
        tc_fence_after();
        const uint32_t za = smem_u32(s.z[n & 1]), fa = smem_u32(s.f[st]);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tb, sdesc_sw128(za + 32 * k, 1024, 16), sdesc_sw128(fa + 32 * k, 1024, 16), idesc, k > 0);
        mma_commit(&s.empty[st]);
        mma_commit(&s.zp_full);
        const int m = n + ZC_NSTAGE;
        if (m < nmma) {
          if (!mbar_wait(&s.empty[st], (n / ZC_NSTAGE) & 1, p.err, 13)) break;
          mbar_arrive_expect_tx(&s.full[st], BK * 128);
          tma_load_2d(s.f[st], &tm_f, 0, (bh * p.nc + step_chunk(has_partial, T, m)) * D, &s.full[st]);
        }
      }
    }
  } else {
    const int r = tid;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    // every thread runs every step (wg_sync needs all of them); after a timed-out wait (error
    // recorded) the remaining waits are skipped
    bool ok = mbar_wait(&s.z_init, 0, p.err, 14);
    for (int n = 0; n < nsteps; ++n) {
      uint8_t* cur = s.z[n & 1];
      fence_proxy_async_smem();
      wg_sync();
      if (r == 0) {
        bulk_store(zbase + (size_t)n * ZTILE, cur, ZTILE);
        bulk_commit();
        if (n + 1 < nsteps) mbar_arrive(&s.z_ready);
      }
      if (n + 1 == nsteps) break;
      ok = ok && mbar_wait(&s.zp_full, n & 1, p.err, 15);
      tc_fence_after();
      uint8_t* nxt = s.z[(n + 1) & 1];
      if (r == 0) bulk_wait_read0();  // the store of step n-1 read `nxt`
      wg_sync();
      const bool active = !(has_partial && n == 0 && r < 64);
      uint32_t a[32], b[32];
      tmem_ld32(tb + lane_off, a);
      tmem_ld32(tb + lane_off + 32, b);
      tmem_ld_wait();
      uint8_t* row = nxt + r * 128;
      if (active) {
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const uint32_t* src = (q < 4) ? (a + 8 * q) : (b + 8 * (q - 4));
          uint4 pk;
          pk.x = pack_bf16(__uint_as_float(src[0]), __uint_as_float(src[1]));
          pk.y = pack_bf16(__uint_as_float(src[2]), __uint_as_float(src[3]));
          pk.z = pack_bf16(__uint_as_float(src[4]), __uint_as_float(src[5]));
          pk.w = pack_bf16(__uint_as_float(src[6]), __uint_as_float(src[7]));
          *reinterpret_cast<uint4*>(row + ((q ^ (r & 7)) * 16)) = pk;
        }
      } else {
        const uint4* src = reinterpret_cast<const uint4*>(cur + r * 128);
#pragma unroll
        for (int q = 0; q < 8; ++q) reinterpret_cast<uint4*>(row)[q] = src[q];
      }
      tc_fence_before();
    }
    if (r == 0) bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 4) {
    tc_fence_after();
    tmem_dealloc(tb, 64);
  }
}

// ============================ adjoint scan ============================
// Per step k (chunk c, transported queries Z_n, n = nsteps - 1 - k) the MMA issuer runs
//   S_{k+1} = Z K->^T, dP_{k+1} = dO V^T          (one step ahead: as soon as the softmax side has
//                                                  taken S_k, dP_k into registers)
//   G_n = [dS | G_{n+1}] [K->_c ; F_c]            (one K=128 chain, A from TMEM)
//   [dK->_c ; dF_c] = [dS^T ; G_{n+1}^T] Z_n      (one M=128 MMA: the dS and G tiles are adjacent
//                                                  in shared memory and form one MN-major operand)
//   dV_c = P^T dO
// dO (constant per tile), dS and G_{n+1} are also kept in TMEM as bf16 pairs, so that dP and G
// read only their B tiles from shared memory; shared-memory bandwidth, not the tensor pipe,
// bounds these N=64 products.
constexpr int BS_KSTAGE = 3;   // [K->_c ; F_c] ring (held until the G chain of the step completes)
constexpr int BS_VSTAGE = 2;   // V_c ring (released once dP of the step completes)
constexpr int BS_ZSTAGE = 3;   // Z_n ring (streamed from HBM)
constexpr uint32_t BOX = 64 * 128;  // one 64-row x 32-column fp32 box (128-byte swizzled rows)
// TMEM columns: S (also G_0 of a partial step), dP, G_n, [dK->; dF], dV (two buffers), dO (bf16
// pairs), dS | G_{n+1} (bf16 pairs, the A operand of the G chain)
constexpr uint32_t TM_S = 0, TM_DP = 64, TM_G = 128, TM_DKF = 192, TM_DV = 256, TM_DO = 384, TM_DSG = 416;
constexpr uint32_t TM_G2 = TM_S;  // the last step issues no next S

struct __align__(1024) BsStage {
  uint8_t kr[BK * 128];    // K->_c  } adjacent: the B operand [K->_c ; F_c] of the G chain
  uint8_t f[BK * 128];     // F_c    }
};
struct __align__(1024) BsSmem {
  uint8_t ps[ZTILE];       // P  (bf16, rows x keys)
  uint8_t ds[ZTILE];       // dS (bf16, rows x keys), scale included
  uint8_t gs[ZTILE];       // G_{n+1} (bf16, rows x d); follows ds (stacked operand)
  uint8_t dO[ZTILE];
  uint8_t z[BS_ZSTAGE][ZTILE];  // Z_n
  BsStage st[BS_KSTAGE];
  uint8_t v[BS_VSTAGE][BK * 128];  // V_c
  // dK->, dF, dV of a step as fp32 boxes (column halves 0-31 / 32-63) for the tensor reductions
  uint8_t stg[6][BOX];       // 0,1: dK->   2,3: dF   4,5: dV
  uint64_t full[BS_KSTAGE], empty[BS_KSTAGE], vfull[BS_VSTAGE], vempty[BS_VSTAGE], zfull[BS_ZSTAGE],
      zempty[BS_ZSTAGE];
  uint64_t do_full, sp_full, sp_free, ps_ready, g_full, gs_ready, acc_full, dkf_free, dv_free[2];
  uint32_t tmem_base;
  alignas(16) float fxa[BS_KSTAGE][BK];  // PaTH-FoX: prefix sums A_j of the stage's key chunk
};

struct BsParams {
  int L, Lp, nc, BH, ntiles;
  float scale, scl;
  const float* lse;
  const float* Dv;
  const uint8_t* zs;
  float* dql;   // [BH][Lp][64]  dQ<- (written)
  float* dkr;   // [BH][Lp][64]  dK-> (accumulated)
  float* dv;    // [BH][Lp][64]  dV   (accumulated)
  float* df;    // [BH][nc][64][64] dF (accumulated)
  int* err;
  const float* fxa;  // PaTH-FoX: A_i = sum_{s<=i} log f_s        [BH][Lp]
  float* fxcs;       // PaTH-FoX: column sums of dS' (accumulated) [BH][Lp]
};

// 32 fp32 values as row r of a 128-byte swizzled fp32 box.
__device__ __forceinline__ void store_box_row(uint8_t* box, int r, const uint32_t* x) {
  uint8_t* row = box + r * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<uint4*>(row + ((q ^ (r & 7)) * 16)) = make_uint4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
}
__device__ __forceinline__ void grad_sync() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
__device__ __forceinline__ void soft_sync() { asm volatile("bar.sync 3, 256;" ::: "memory"); }
// 16 fp32 values as columns 16q .. 16q+15 of row r of a 128-byte swizzled fp32 box.
__device__ __forceinline__ void store_box_quarter(uint8_t* box, int r, int q, const uint32_t* x) {
  uint8_t* row = box + r * 128;
#pragma unroll
  for (int j = 0; j < 4; ++j)
    *reinterpret_cast<uint4*>(row + (((4 * q + j) ^ (r & 7)) * 16)) =
        make_uint4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
}

// 32 bf16 pairs (column 2j in the low half) as row r of a 128-byte swizzled bf16 tile.
__device__ __forceinline__ void put_row_packed(uint8_t* tile, int r, const uint32_t* pk) {
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int q = 0; q < 8; ++q)
    *reinterpret_cast<uint4*>(row + ((q ^ (r & 7)) * 16)) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}
// 16 bf16 pairs as columns 32h .. 32h+31 of row r of a 128-byte swizzled bf16 tile.
__device__ __forceinline__ void put_half_packed(uint8_t* tile, int r, int h, const uint32_t* pk) {
  uint8_t* row = tile + r * 128;
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(row + (((4 * h + q) ^ (r & 7)) * 16)) = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
}
// 64 fp32 values as 32 bf16 pairs (column 2j in the low half), the TMEM A-operand layout.
__device__ __forceinline__ void pack_row_pairs(const float* x, uint32_t (&pk)[32]) {
#pragma unroll
  for (int j = 0; j < 32; ++j) pk[j] = pack_bf16(x[2 * j], x[2 * j + 1]);
}

// Warp roles: 0-3 and 11-14 softmax side (P, dS of a step; two threads per query row, column
// halves 0-31 / 32-63; then the dV reductions of the previous step), 4 TMA/bulk producer (lane 0:
// K->, F; lane 8: V; lane 16: Z), 5 MMA issuer A (S, dP, the G chain), 6-9 gradient side (G_n
// conversion, dQ<- output, dK->/dF reductions), 10 MMA issuer B ([dK->; dF], dV).  Two issuers because a tcgen05.mma costs tens of cycles to
// issue from one thread and these products are small (N = 64).
constexpr int BS_THREADS = 480;
constexpr int BS_NSOFT = 256;

// Column sums over the warp's 32 rows of the 32 values each lane holds (its row's columns):
// a reduce-scatter butterfly; on return v[0] of lane l is the sum of column l.
__device__ __forceinline__ void warp_column_sums(float (&v)[32], int lane) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) {
    const bool up = (lane & o) != 0;
#pragma unroll
    for (int j = 0; j < o; ++j) {
      const float send = up ? v[j] : v[j + o];
      const float keep = up ? v[j + o] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
    }
  }
}

// FOX (PaTH-FoX, notes §2.5): the logit of (i, j) gains A_i - A_j; the column sums of the
// step's dS' = P (dP - D) are added into fxcs for dlog f.
template <bool FOX>
__global__ void __launch_bounds__(BS_THREADS, 1) bwd_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_do,
                                                            const __grid_constant__ CUtensorMap tm_kr,
                                                            const __grid_constant__ CUtensorMap tm_v,
                                                            const __grid_constant__ CUtensorMap tm_f,
                                                            const __grid_constant__ CUtensorMap tm_rdk,
                                                            const __grid_constant__ CUtensorMap tm_rdv,
                                                            const __grid_constant__ CUtensorMap tm_rdf,
                                                            const BsParams p) {
  extern __shared__ uint8_t smem_raw[];
  BsSmem& s = *reinterpret_cast<BsSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int err0 = threadIdx.x == 0 ? peek_err(p.err) : 0;  // consumed at the setup barrier
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bh, T;
  tile_of_block((int)blockIdx.x, p.ntiles, p.BH, bh, T);
  const bool has_partial = (2 * T + 1) * BK < p.L;
  const int nsteps = (has_partial ? 1 : 0) + 2 * T;
  const uint8_t* zbase = p.zs + ((size_t)bh * p.ntiles * p.ntiles + (size_t)T * T) * ZTILE;

  if (nsteps == 0) {  // no earlier chunk: dQ<- of the tile is zero
    for (int idx = tid; idx < BQ * D; idx += blockDim.x)
      p.dql[((size_t)bh * p.Lp + (size_t)T * BQ) * D + idx] = 0.f;
    return;
  }
  if (tid == 0) {
    for (int k = 0; k < BS_KSTAGE; ++k) {
      mbar_init(&s.full[k], 1);
      mbar_init(&s.empty[k], 1);
    }
    for (int k = 0; k < BS_VSTAGE; ++k) {
      mbar_init(&s.vfull[k], 1);
      mbar_init(&s.vempty[k], 1);
    }
    for (int k = 0; k < BS_ZSTAGE; ++k) {
      mbar_init(&s.zfull[k], 1);
      mbar_init(&s.zempty[k], 2);  // both issuers read Z
    }
    mbar_init(&s.do_full, 1);
    mbar_init(&s.sp_full, 1);
    mbar_init(&s.sp_free, BS_NSOFT);
    mbar_init(&s.ps_ready, BS_NSOFT);
    mbar_init(&s.g_full, 2);       // G_n (issuer A) and [dK->; dF] (issuer B) complete
    mbar_init(&s.gs_ready, 128);
    mbar_init(&s.acc_full, 1);     // issuer B's MMAs of the step complete
    mbar_init(&s.dkf_free, 128);   // the gradient side has read [dK->; dF] of the step
    mbar_init(&s.dv_free[0], BS_NSOFT);  // the softmax side has read dV, one barrier per dV buffer (a
    mbar_init(&s.dv_free[1], BS_NSOFT);  // single one could complete step k-1 before issuer B waits for k-2)
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(&s.tmem_base, 512);
  tc_fence_before();
  // a wait of an earlier CTA of the launch has given up: end at once (the pipeline is broken)
  const bool launch_err = __syncthreads_or(err0 != 0) != 0;
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  if (launch_err) {
    if (warp == 5) tmem_dealloc(tb, 512);
    return;
  }

  if (warp == 4) {
    // ---------------- producers ----------------
    if (lane == 0) {  // [K->_c ; F_c] (and dO once)
      mbar_arrive_expect_tx(&s.do_full, ZTILE);
      tma_load_2d(s.dO, &tm_do, 0, bh * p.L + T * BQ, &s.do_full);
      for (int k = 0; k < nsteps; ++k) {
        const int si = k % BS_KSTAGE;
        if (k >= BS_KSTAGE && !mbar_wait(&s.empty[si], ((k / BS_KSTAGE) - 1) & 1, p.err, 21)) break;
        const int c = step_chunk(has_partial, T, nsteps - 1 - k);
        BsStage& S = s.st[si];
        mbar_arrive_expect_tx(&s.full[si], 2 * BK * 128 + (FOX ? BK * 4 : 0));
        tma_load_2d(S.kr, &tm_kr, 0, bh * p.Lp + c * BK, &s.full[si]);
        tma_load_2d(S.f, &tm_f, 0, (bh * p.nc + c) * D, &s.full[si]);
        if constexpr (FOX) bulk_load(s.fxa[si], p.fxa + (size_t)bh * p.Lp + (size_t)c * BK, BK * 4, &s.full[si]);
      }
    } else if (lane == 8) {  // V_c
      for (int k = 0; k < nsteps; ++k) {
        const int vi = k % BS_VSTAGE;
        if (k >= BS_VSTAGE && !mbar_wait(&s.vempty[vi], ((k / BS_VSTAGE) - 1) & 1, p.err, 19)) break;
        const int c = step_chunk(has_partial, T, nsteps - 1 - k);
        mbar_arrive_expect_tx(&s.vfull[vi], BK * 128);
        tma_load_2d(s.v[vi], &tm_v, 0, bh * p.L + c * BK, &s.vfull[vi]);
      }
    } else if (lane == 16) {  // Z_n
      for (int k = 0; k < nsteps; ++k) {
        const int zi = k % BS_ZSTAGE;
        if (k >= BS_ZSTAGE && !mbar_wait(&s.zempty[zi], ((k / BS_ZSTAGE) - 1) & 1, p.err, 20)) break;
        mbar_arrive_expect_tx(&s.zfull[zi], ZTILE);
        bulk_load(s.z[zi], zbase + (size_t)(nsteps - 1 - k) * ZTILE, ZTILE, &s.zfull[zi]);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer A: S, dP (one step ahead) and the G chain ----------------
    if (lane == 0) {
      const uint32_t i_rk = idesc_bf16(128, 64, 0, 0);   // [128 x 64] = A(K-major / TMEM) B(K-major)^T
      const uint32_t i_rm = idesc_bf16(128, 64, 0, 1);   // [128 x 64] = A(TMEM) B(MN-major)
      auto issue_sdp = [&](int k) {  // S and dP of step k
        const BsStage& S = s.st[k % BS_KSTAGE];
        const uint32_t a_z = smem_u32(s.z[k % BS_ZSTAGE]), a_kr = smem_u32(S.kr), a_v = smem_u32(s.v[k % BS_VSTAGE]);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ss(tb + TM_S, sdesc_sw128(a_z + 32 * kk, 1024, 16), sdesc_sw128(a_kr + 32 * kk, 1024, 16), i_rk, kk > 0);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(tb + TM_DP, tb + TM_DO + 8 * kk, sdesc_sw128(a_v + 32 * kk, 1024, 16), i_rk, kk > 0);
        mma_commit(&s.sp_full);
        mma_commit(&s.vempty[k % BS_VSTAGE]);
      };
      // phase 0 of gs_ready: dO is in TMEM and G_{nsteps} = 0 is in place
      bool ok = mbar_wait(&s.gs_ready, 0, p.err, 22) && mbar_wait(&s.full[0], 0, p.err, 23) &&
                mbar_wait(&s.vfull[0], 0, p.err, 23) && mbar_wait(&s.zfull[0], 0, p.err, 23);
      if (ok) {
        tc_fence_after();
        issue_sdp(0);
      }
      for (int k = 0; ok && k < nsteps; ++k) {
        const int si = k % BS_KSTAGE;
        const int n = nsteps - 1 - k;
        const bool partial = has_partial && n == 0;
        // the softmax side has taken S/dP of step k into registers: issue step k+1's
        if (!mbar_wait(&s.sp_free, k & 1, p.err, 37)) { ok = false; break; }
        if (k + 1 < nsteps) {
          if (!mbar_wait(&s.full[(k + 1) % BS_KSTAGE], ((k + 1) / BS_KSTAGE) & 1, p.err, 23) ||
              !mbar_wait(&s.vfull[(k + 1) % BS_VSTAGE], ((k + 1) / BS_VSTAGE) & 1, p.err, 23) ||
              !mbar_wait(&s.zfull[(k + 1) % BS_ZSTAGE], ((k + 1) / BS_ZSTAGE) & 1, p.err, 23)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_sdp(k + 1);
        }
        // dS of step k is in TMEM, G_{n+1} is in place (shared memory and TMEM) and G_{n+2} has
        // left TM_G
        if (!mbar_wait(&s.ps_ready, k & 1, p.err, 24) || !mbar_wait(&s.gs_ready, k & 1, p.err, 27)) {
          ok = false;
          break;
        }
        tc_fence_after();
        // G_n = [dS | G_{n+1}] [K->_c ; F_c]  (a partial step keeps G_1 of rows 0-63 in TM_G)
        const uint32_t a_kr = smem_u32(s.st[si].kr);
        const uint32_t tg = partial ? TM_G2 : TM_G;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ts(tb + tg, tb + TM_DSG + 8 * kk, sdesc_sw128(a_kr + 2048 * kk, 1024, 0), i_rm, kk > 0);
        mma_commit(&s.g_full);
        mma_commit(&s.empty[si]);
        mma_commit(&s.zempty[k % BS_ZSTAGE]);
      }
    }
  } else if (warp == 10) {
    // ---------------- MMA issuer B: [dK->; dF] and dV ----------------
    if (lane == 0) {
      const uint32_t i_tt = idesc_bf16(64, 64, 1, 1);    // [64 x 64]  = A(MN-major) B(MN-major)
      const uint32_t i_st = idesc_bf16(128, 64, 1, 1);   // [128 x 64] = A(MN-major, two atoms) B(MN-major)
      const uint32_t a_do = smem_u32(s.dO), a_ps = smem_u32(s.ps), a_ds = smem_u32(s.ds);
      bool ok = mbar_wait(&s.do_full, 0, p.err, 32);
      for (int k = 0; ok && k < nsteps; ++k) {
        const int n = nsteps - 1 - k;
        const bool partial = has_partial && n == 0;
        const int zi = k % BS_ZSTAGE;
        // P, dS (shared memory) of step k, G_{n+1} (shared memory), Z_n, and [dK->; dF] of step
        // k-1 read out
        if (!mbar_wait(&s.ps_ready, k & 1, p.err, 33) || !mbar_wait(&s.gs_ready, k & 1, p.err, 34) ||
            !mbar_wait(&s.zfull[zi], (k / BS_ZSTAGE) & 1, p.err, 35) ||
            (k >= 1 && !mbar_wait(&s.dkf_free, (k - 1) & 1, p.err, 29))) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t a_z = smem_u32(s.z[zi]);
        // [dK->; dF] = [dS^T; G_{n+1}^T] Z_n over the rows that crossed chunk c (rows 64-127 at a
        // partial step, where dS of rows 0-63 is zero anyway)
        {
          const uint32_t off = partial ? 64 * 128 : 0;
          const int nk = partial ? 4 : 8;
          for (int kk = 0; kk < nk; ++kk)
            mma_ss(tb + TM_DKF, sdesc_sw128(a_ds + off + 2048 * kk, 1024, ZTILE),
                   sdesc_sw128(a_z + off + 2048 * kk, 1024, 0), i_st, kk > 0);
        }
        mma_commit(&s.g_full);
        // dV = P^T dO  (M = 64 keys, K = 128 rows) into buffer k % 2, read out two steps ago
        if (k >= 2 && !mbar_wait(&s.dv_free[k & 1], ((k - 2) >> 1) & 1, p.err, 38)) { ok = false; break; }
        tc_fence_after();
        const uint32_t tdv = TM_DV + 64 * (k & 1);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          mma_ss(tb + tdv, sdesc_sw128(a_ps + 2048 * kk, 1024, 0), sdesc_sw128(a_do + 2048 * kk, 1024, 0), i_tt, kk > 0);
        mma_commit(&s.acc_full);
        mma_commit(&s.zempty[zi]);
      }
    }
  } else if (warp < 4 || warp >= 11) {
    // ---------------- softmax side: thread (r, h) owns columns 32h..32h+31 of query row r ----------------
    const int q4 = warp & 3, h = warp < 4 ? 0 : 1;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const int grow = T * BQ + r;
    const size_t wrow = (size_t)bh * p.Lp + (size_t)T * BQ + r;
    const float lse2 = grow < p.L ? p.lse[(size_t)bh * p.L + grow] * kLog2e : INFINITY;
    const float Dr = p.Dv[wrow];
    // FOX: exponent offset of the row, A_i log2(e) - lse_i log2(e); the keys' -A_j log2(e) per step
    const float fox_row = FOX ? p.fxa[wrow] * kLog2e - lse2 : 0.f;
    const float inv_scale = FOX ? 1.f / p.scale : 0.f;
    float fox_rowsum = 0.f;  // FOX: this thread's share of its row's sum of dS' (scaled)
    const int vrow = 16 * q4 + (lane & 15), vh = lane >> 4;  // dV (M=64): row, column half
    // dV of step j (complete) -> columns 16h.. of the fp32 boxes 4, 5 -> two tensor reductions
    // issued by thread 0 (its own bulk groups: each waits for the previous one to have read the
    // boxes).  Runs after the step's P and dS are published, in the softmax side's slack.
    auto stage_dv = [&](int j) {
      const int crow = bh * p.Lp + step_chunk(has_partial, T, nsteps - 1 - j) * BK;
      if (tid == 0) bulk_wait_read0();
      soft_sync();
      uint32_t a[16];
      tmem_ld16x2_16(tb + lane_off + TM_DV + 64 * (j & 1) + 16 * h, a);
      tmem_ld_wait();
      store_box_quarter(s.stg[4 + vh], vrow, h, a);
      tc_fence_before();
      mbar_arrive(&s.dv_free[j & 1]);
      fence_proxy_async_smem();
      soft_sync();
      if (tid == 0) {
        tma_reduce_add_2d(&tm_rdv, s.stg[4], 0, crow);
        tma_reduce_add_2d(&tm_rdv, s.stg[5], 32, crow);
        bulk_commit();
      }
    };
    // Every softmax thread runs every step (soft_sync needs all 256); after a timed-out wait
    // (error recorded) the remaining waits are skipped.
    bool ok = true;
    for (int k = 0; k < nsteps; ++k) {
      const int n = nsteps - 1 - k;
      const bool partial = has_partial && n == 0;
      const bool active = !(partial && r < 64);
      ok = ok && mbar_wait(&s.sp_full, k & 1, p.err, 25);
      tc_fence_after();
      uint32_t sa[32], da[32];
      tmem_ld32(tb + lane_off + TM_S + 32 * h, sa);
      tmem_ld32(tb + lane_off + TM_DP + 32 * h, da);
      tmem_ld_wait();
      tc_fence_before();
      mbar_arrive(&s.sp_free);  // S and dP of step k may be overwritten
      float pv[32], dsv[32];
      if constexpr (FOX) {
        // the stage of this step's chunk holds its A_j (its barrier completed before S was issued)
        const int si = k % BS_KSTAGE;
        ok = ok && mbar_wait(&s.full[si], (k / BS_KSTAGE) & 1, p.err, 39);
        // key pairs through paired fp32 instructions: x = scl s - A_j log2(e) + (A_i log2(e) - lse),
        // P = 2^x, dS = scale P (dP - D)
        const ulonglong2* a4 = reinterpret_cast<const ulonglong2*>(s.fxa[si] + 32 * h);
        const uint64_t scl2 = f2(p.scl, p.scl), nle2 = f2(-kLog2e, -kLog2e), fr2 = f2(fox_row, fox_row);
        const uint64_t nd2 = f2(-Dr, -Dr), sc2 = f2(p.scale, p.scale), z2 = f2(0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const ulonglong2 av = a4[q];  // A_j of keys 4q .. 4q+3 as two pairs
#pragma unroll
          for (int e = 0; e < 2; ++e) {
            const int j = 4 * q + 2 * e;
            const uint64_t off = f2_fma(e ? av.y : av.x, nle2, fr2);
            float x0, x1;
            f2_split(f2_fma(f2(__uint_as_float(sa[j]), __uint_as_float(sa[j + 1])), scl2, off), x0, x1);
            const float p0 = active ? fast_exp2(x0) : 0.f, p1 = active ? fast_exp2(x1) : 0.f;
            pv[j] = p0;
            pv[j + 1] = p1;
            const uint64_t dd = f2_add(f2(__uint_as_float(da[j]), __uint_as_float(da[j + 1])), nd2);
            f2_split(f2_fma(f2_fma(f2(p0, p1), sc2, z2), dd, z2), dsv[j], dsv[j + 1]);
          }
        }
      } else {
        // key pairs through paired fp32 instructions: x = scl s - lse (log2 units), P = 2^x,
        // dS = scale P (dP - D); the exponentials stay scalar
        const uint64_t scl2 = f2(p.scl, p.scl), nl2 = f2(-lse2, -lse2), nd2 = f2(-Dr, -Dr), sc2 = f2(p.scale, p.scale);
        const uint64_t z2 = f2(0.f, 0.f);
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          float x0, x1;
          f2_split(f2_fma(f2(__uint_as_float(sa[2 * j]), __uint_as_float(sa[2 * j + 1])), scl2, nl2), x0, x1);
          const float p0 = active ? fast_exp2(x0) : 0.f, p1 = active ? fast_exp2(x1) : 0.f;
          pv[2 * j] = p0;
          pv[2 * j + 1] = p1;
          const uint64_t dd = f2_add(f2(__uint_as_float(da[2 * j]), __uint_as_float(da[2 * j + 1])), nd2);
          f2_split(f2_fma(f2_fma(f2(p0, p1), sc2, z2), dd, z2), dsv[2 * j], dsv[2 * j + 1]);
        }
      }
      uint32_t pk[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) pk[j] = pack_bf16(dsv[2 * j], dsv[2 * j + 1]);
      // the MMAs of step k-1 have read P, dS (shared memory) and dS (TMEM): the G chain and
      // [dK->; dF] (g_full), dV (acc_full)
      if (k > 0) ok = ok && mbar_wait(&s.g_full, (k - 1) & 1, p.err, 36) && mbar_wait(&s.acc_full, (k - 1) & 1, p.err, 26);
      tc_fence_after();
      put_half(s.ps, r, h, pv);
      put_half_packed(s.ds, r, h, pk);  // the pairs already packed for TMEM
      tmem_st16(tb + lane_off + TM_DSG + 16 * h, pk);
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.ps_ready);
      if constexpr (FOX) {  // row sum of dS' kept; column sums over this warp's 32 rows into fxcs
#pragma unroll
        for (int j = 0; j < 32; ++j) fox_rowsum += dsv[j];
        warp_column_sums(dsv, lane);
        atomicAdd(p.fxcs + (size_t)bh * p.Lp + (size_t)step_chunk(has_partial, T, n) * BK + 32 * h + lane,
                  dsv[0] * inv_scale);
      }
      if (k > 0) stage_dv(k - 1);
    }
    ok = ok && mbar_wait(&s.acc_full, (nsteps - 1) & 1, p.err, 26);
    tc_fence_after();
    stage_dv(nsteps - 1);
    if constexpr (FOX) atomicAdd(p.fxcs + wrow, -fox_rowsum * inv_scale);  // fxcs_m = colsum_m - rowsum_m
    if (tid == 0) bulk_wait0();
  } else if (warp >= 6) {
    // ---------------- gradient side: thread owns query row rg = 32 (warp % 4) + lane ----------------
    const int q4 = warp & 3;
    const int rg = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const size_t wrow = (size_t)bh * p.Lp + (size_t)T * BQ + rg;
    {  // dO into TMEM (A operand of dP); G_{nsteps} = 0 in shared memory and TMEM
      mbar_wait(&s.do_full, 0, p.err, 31);
      uint32_t buf[32];
      const uint8_t* row = s.dO + rg * 128;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(row + ((q ^ (rg & 7)) * 16));
        buf[4 * q] = v.x;
        buf[4 * q + 1] = v.y;
        buf[4 * q + 2] = v.z;
        buf[4 * q + 3] = v.w;
      }
      tmem_st32(tb + lane_off + TM_DO, buf);
#pragma unroll
      for (int j = 0; j < 32; ++j) buf[j] = 0u;
      tmem_st32(tb + lane_off + TM_DSG + 32, buf);
      uint4* grow_ = reinterpret_cast<uint4*>(s.gs + rg * 128);
#pragma unroll
      for (int q = 0; q < 8; ++q) grow_[q] = make_uint4(0, 0, 0, 0);
      fence_proxy_async_smem();
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.gs_ready);
    }
    // Every gradient thread runs every step (grad_sync needs all 128); after a timed-out wait
    // (error recorded) the remaining waits are skipped.
    bool ok = true;
    for (int k = 0; k < nsteps; ++k) {
      const int n = nsteps - 1 - k;
      const bool partial = has_partial && n == 0;
      const int c = step_chunk(has_partial, T, n);
      ok = ok && mbar_wait(&s.g_full, k & 1, p.err, 28);
      tc_fence_after();
      // G_n (rows 0-63 of a partial step keep G_1)
      {
        const uint32_t tg = (partial && rg >= 64) ? TM_G2 : TM_G;
        uint32_t ga[32], gb[32];
        tmem_ld32(tb + lane_off + tg, ga);
        tmem_ld32(tb + lane_off + tg + 32, gb);
        tmem_ld_wait();
        float g[64];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          g[j] = __uint_as_float(ga[j]);
          g[32 + j] = __uint_as_float(gb[j]);
        }
        if (partial && rg < 64 && k == 0) {  // a tile whose only step is the partial one: G_1 = 0
#pragma unroll
          for (int j = 0; j < 64; ++j) g[j] = 0.f;
        }
        if (n == 0) {
          float4* dst = reinterpret_cast<float4*>(p.dql + wrow * D);
#pragma unroll
          for (int j = 0; j < 16; ++j) dst[j] = make_float4(g[4 * j], g[4 * j + 1], g[4 * j + 2], g[4 * j + 3]);
        } else {
          uint32_t pk[32];
          pack_row_pairs(g, pk);
          put_row_packed(s.gs, rg, pk);  // the same pairs for shared memory and TMEM
          tmem_st32(tb + lane_off + TM_DSG + 32, pk);
          fence_proxy_async_smem();
          tmem_st_wait();
        }
        tc_fence_before();
        mbar_arrive(&s.gs_ready);
      }
      // [dK->; dF] of this step -> swizzled fp32 boxes 0-3 -> four tensor reductions (one bulk
      // group, which the next step's staging waits to have read the boxes).
      const int crow = bh * p.Lp + c * BK;
      const int frow = (bh * p.nc + c) * D;
      if (rg == 0) bulk_wait_read0();  // the previous step's [dK->; dF] group has read boxes 0-3
      grad_sync();
      {
        uint32_t a[32];
        tmem_ld32(tb + lane_off + TM_DKF, a);
        tmem_ld_wait();
        const int bx = rg < 64 ? 0 : 2, br = rg & 63;
        store_box_row(s.stg[bx], br, a);
        tmem_ld32(tb + lane_off + TM_DKF + 32, a);
        tmem_ld_wait();
        store_box_row(s.stg[bx + 1], br, a);
      }
      tc_fence_before();
      mbar_arrive(&s.dkf_free);
      fence_proxy_async_smem();
      grad_sync();
      if (rg == 0) {
        tma_reduce_add_2d(&tm_rdk, s.stg[0], 0, crow);
        tma_reduce_add_2d(&tm_rdk, s.stg[1], 32, crow);
        if (k > 0) {  // G_{nsteps} = 0: the first step adds nothing to dF
          tma_reduce_add_2d(&tm_rdf, s.stg[2], 0, frow);
          tma_reduce_add_2d(&tm_rdf, s.stg[3], 32, frow);
        }
        bulk_commit();
      }
    }
    bulk_wait0();
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

}  // namespace

cudaError_t launch_bwd_tc(const TcWs& w, const void* q, const void* k, const void* v, const void* wv,
                          const float* beta, const void* o, const float* lse, const void* dO, void* dq, void* dk,
                          void* dv, void* dw, float* dbeta, char* ws, int phases, cudaStream_t st, const float* logf,
                          float* dlogf) {
  cudaError_t e;
  const Geom& g = w.g64;
  const size_t rows = (size_t)g.BH * g.Lp;
  const int nt = g.Lp / BQ;
  int* err = (int*)(ws + w.p64.err);
  if (phases & 1) {
    if ((e = cudaMemsetAsync(ws + w.dkr64, 0, rows * D * 4, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(ws + w.dv, 0, rows * D * 4, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(ws + w.df64, 0, (size_t)g.BH * g.nc * D * D * 4, st)) != cudaSuccess) return e;
    // the error word starts afresh unless the backward builds on the forward's state, whose
    // timeouts it then keeps
    if (!(phases & (8 | 16)) && (e = cudaMemsetAsync(err, 0, sizeof(int), st)) != cudaSuccess) return e;
    if ((e = launch_bwd_dot(g, o, dO, (float*)(ws + w.Dv), st)) != cudaSuccess) return e;
    if (logf) {  // PaTH-FoX: prefix sums of log f, zeroed column sums of dS'
      if ((e = launch_fox_prefix(g, logf, (float*)(ws + w.fxa), st)) != cudaSuccess) return e;
      if ((e = cudaMemsetAsync(ws + w.fxcs, 0, rows * 4, st)) != cudaSuccess) return e;
    }
    if (!(phases & 8)) {  // 8: the forward's chunk-64 preparation is already in ws
      if ((e = launch_ut_prep64(w.g64, q, k, v, wv, beta, nullptr, ws, w.p64, false, st)) != cudaSuccess) return e;
    }
    if (!(phases & 16)) {  // 16: the forward stored the transported query tiles in ws
      CUtensorMap m_ql, m_f;
      if (!make_map_rows64(&m_ql, ws + w.p64.ql, rows, BQ) ||
          !make_map_rows64(&m_f, ws + w.p64.f, (uint64_t)g.BH * g.nc * D, D))
        return cudaErrorInvalidValue;
      ZcParams zp{g.L, g.Lp, g.nc, g.BH, nt, (uint8_t*)(ws + w.zs), err};
      const size_t smem = sizeof(ZcSmem) + 1024;
      if ((e = cudaFuncSetAttribute(zchain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
        return e;
      zchain_tc_kernel<<<(unsigned)((long)nt * g.BH), 160, smem, st>>>(m_ql, m_f, zp);
      if ((e = cudaGetLastError()) != cudaSuccess) return e;
    }
  }
  if (phases & 2) {
    CUtensorMap m_do, m_kr, m_v, m_f, m_rdk, m_rdv, m_rdf;
    if (!make_map_f32_rows64(&m_rdk, ws + w.dkr64, rows) || !make_map_f32_rows64(&m_rdv, ws + w.dv, rows) ||
        !make_map_f32_rows64(&m_rdf, ws + w.df64, (uint64_t)g.BH * g.nc * D))
      return cudaErrorInvalidValue;
    if (!make_map_rows64(&m_do, dO, (uint64_t)g.BH * g.L, BQ) ||
        !make_map_rows64(&m_kr, ws + w.p64.kr, rows, BK) || !make_map_rows64(&m_v, v, (uint64_t)g.BH * g.L, BK) ||
        !make_map_rows64(&m_f, ws + w.p64.f, (uint64_t)g.BH * g.nc * D, D))
      return cudaErrorInvalidValue;
    BsParams bp;
    bp.L = g.L;
    bp.Lp = g.Lp;
    bp.nc = g.nc;
    bp.BH = g.BH;
    bp.ntiles = nt;
    bp.scale = g.scale;
    bp.scl = g.scale * kLog2e;
    bp.lse = lse;
    bp.Dv = (const float*)(ws + w.Dv);
    bp.zs = (const uint8_t*)(ws + w.zs);
    bp.dql = (float*)(ws + w.dql64);
    bp.dkr = (float*)(ws + w.dkr64);
    bp.dv = (float*)(ws + w.dv);
    bp.df = (float*)(ws + w.df64);
    bp.err = err;
    bp.fxa = logf ? (const float*)(ws + w.fxa) : nullptr;
    bp.fxcs = logf ? (float*)(ws + w.fxcs) : nullptr;
    const size_t smem = sizeof(BsSmem) + 1024;
    auto kern = logf ? bwd_scan_tc_kernel<true> : bwd_scan_tc_kernel<false>;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
      return e;
    kern<<<(unsigned)((long)nt * g.BH), BS_THREADS, smem, st>>>(m_do, m_kr, m_v, m_f, m_rdk, m_rdv, m_rdf, bp);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (phases & 4) {
    float* cs = logf ? (float*)(ws + w.fxcs) : nullptr;
    if ((e = launch_ut_bwd64(g, q, k, v, wv, beta, lse, dO, (const float*)(ws + w.Dv), (const float*)(ws + w.dql64),
                             (const float*)(ws + w.dkr64), (const float*)(ws + w.dv), (const float*)(ws + w.df64), dq,
                             dk, dv, dw, dbeta, err, st, logf, cs)) != cudaSuccess)
      return e;
    if (dlogf && (e = launch_fox_dlogf(g, cs, dlogf, st)) != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace pathattn
