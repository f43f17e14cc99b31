// Per-chunk UT backward on tcgen05 (bf16 operands, fp32 accumulation in TMEM), chunk B = 64.
//
// The pages give no backward.  For one chunk, given the adjoints dQ<-, dK->, dF coming from the
// chunk scan and the diagonal-chunk attention, this is the chain rule through the per-chunk
// quantities of the PaTH reading notes (cc.laoqi.cc/papers/2505.16381) §2.6–§2.7:
//   S_d = lower(Q K^T) - lower(Q W^T) X,  X = U strictLower(W K^T),
//   Q<- = Q - lower(Q W^T) U W,  K-> = K - X^T W,  F = I - W^T U^T W,
//   U = Y D,  Y = (I + strictLower(D W W^T))^{-1}
// giving dq, dk, dv (diagonal part added to the accumulated dV), dw and dbeta.  With
// M1 = lower(QW^T), N2 = strictLower(WK^T), Y1 = U W, P/dS the diagonal probabilities and their
// logit adjoint (scale included):
//   gQ = dQ<- + dS K + gM1 W,            gK = dK-> + dS^T Q + gN2^T W
//   gM1 = lower(-dS X^T - dQ<- Y1^T),     gX = -M1^T dS - W dK->^T
//   E3 = M1^T dQ<- + W dF^T,              gN2 = strictLower(U^T gX)
//   gU = lower(-E3 W^T + gX N2^T),        A1 = gU U^T,   gN = strictLower(-Y^T A1)
//   gW = -U^T E3 - X dK-> - Y1 dF + gM1^T Q + gN2 K + diag(beta) gN W + gN^T diag(beta) W
//   dbeta_j = sum_i gU_ij Y_ij + sum_{m<j} gN_jm G_jm
// Every product is an M=64 N=64 K=64 tcgen05 MMA on 64x64 bf16 tiles (128-byte swizzled),
// K-major or MN-major per operand; accumulators gQ, gK, gW stay in TMEM across phases.
#include "internal.h"
#include "dev_common.cuh"
#include "tc_common.cuh"
#include "ut_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace pathattn {

bool make_map_rows64(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows);  // fwd_tc.cu

namespace {
using namespace tc;

constexpr int B = 64;
constexpr int D = kHeadDim;
constexpr uint32_t TILE = 64 * 128;
constexpr int GS = 65;
// TMEM columns: temporaries 0..319, persistent accumulators gW, gQ, gK
constexpr uint32_t C_GW = 320, C_GQ = 384, C_GK = 448;

// Tile slots (a slot is reused once its first tenant is dead).
enum {
  T_W, T_Q, T_K,
  T_V,   // V (P2), then E3 (P7..P8)
  T_DO,  // dO (P2, P6), then gN2 (P7..P8)
  T_DQ,  // dQ<- (P6, P7), then gU (P8..P9)
  T_DK,  // dK-> (P6, P7), then A1 (P9..P10)
  T_DF,  // dF (P7), then gN (P10..P11)
  T_M1,  // M1 (P5..P7), then diag(beta) gN (P10..P11)
  T_N2, T_U, T_Y, T_X,
  T_Y1,  // Y1 (P6, P7), then diag(beta) W (P9..P11)
  T_P,   // P (P6), then gX (P6..P8)
  T_DS, T_GM1, NTILES
};
constexpr int T_E3 = T_V, T_GN2 = T_DO, T_GU = T_DQ, T_A1 = T_DK, T_GN = T_DF, T_GNB = T_M1, T_BW = T_Y1, T_GX = T_P;

struct __align__(1024) UbSmem {
  uint8_t t[NTILES][TILE];
  float g[B * GS];   // G (strictly lower, fp32)
  float y[B * GS];   // Y (fp32) for dbeta
  float beta[B], lse2[B], dv[B], gb[B];
  uint64_t bar_in, bar_mma;
  uint32_t tmem_base;
};

struct UbParams {
  int L, Lp, nc, BH;
  float scale, scl;
  const float* beta;
  const float* lse;
  const float* Dv;
  const float* dql;    // dQ<-  [BH][Lp][64]
  const float* dkr;    // dK->  [BH][Lp][64]
  const float* dvacc;  // dV of the off-diagonal chunks [BH][Lp][64]
  const float* df;     // dF    [BH][nc][64][64]
  __nv_bfloat16* dq;
  __nv_bfloat16* dk;
  __nv_bfloat16* dv;
  __nv_bfloat16* dw;
  float* dbeta;
  int* err;
};

__device__ __forceinline__ void store_bf16_row(__nv_bfloat16* dst, const float* x) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    d4[q] = make_uint4(pack_bf16(x[8 * q], x[8 * q + 1]), pack_bf16(x[8 * q + 2], x[8 * q + 3]),
                       pack_bf16(x[8 * q + 4], x[8 * q + 5]), pack_bf16(x[8 * q + 6], x[8 * q + 7]));
}

__global__ void __launch_bounds__(128, 1) ut_bwd64_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                         const __grid_constant__ CUtensorMap tm_k,
                                                         const __grid_constant__ CUtensorMap tm_v,
                                                         const __grid_constant__ CUtensorMap tm_w,
                                                         const __grid_constant__ CUtensorMap tm_do,
                                                         const UbParams p) {
  extern __shared__ uint8_t smem_raw[];
  UbSmem& s = *reinterpret_cast<UbSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, bh = blockIdx.y;
  const int row0 = c * B;
  const size_t in_row = (size_t)bh * p.L;
  const size_t ws_row = (size_t)bh * p.Lp + row0;
  const bool lead = tid == 0;
  const int i = 16 * warp + lane;  // M=64 accumulator row of this thread (lanes < 16)
  const bool has_row = lane < 16;
  const bool row_ok = has_row && row0 + i < p.L;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  auto ta = [&](int slot) { return smem_u32(s.t[slot]); };

  if (lead) {
    mbar_init(&s.bar_in, 1);
    mbar_init(&s.bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&s.tmem_base, 512);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  uint32_t mph = 0;
  // Issues the MMAs of one phase (lead thread), then every thread waits for them.
  auto run = [&](auto issue, int code) {
    if (lead) {
      tc_fence_after();
      issue();
      mma_commit(&s.bar_mma);
    }
    mbar_wait(&s.bar_mma, mph, p.err, code);
    mph ^= 1;
    tc_fence_after();
  };
  auto publish = [&]() {  // tiles written by the threads -> visible to the next MMAs
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  };

  // ---- loads ----
  if (lead) {
    const int y0 = (int)(in_row + row0);
    mbar_arrive_expect_tx(&s.bar_in, 5 * TILE);
    tma_load_2d(s.t[T_W], &tm_w, 0, y0, &s.bar_in);
    tma_load_2d(s.t[T_Q], &tm_q, 0, y0, &s.bar_in);
    tma_load_2d(s.t[T_K], &tm_k, 0, y0, &s.bar_in);
    tma_load_2d(s.t[T_V], &tm_v, 0, y0, &s.bar_in);
    tma_load_2d(s.t[T_DO], &tm_do, 0, y0, &s.bar_in);
  }
  if (tid < B) {
    const int gi = row0 + tid;
    const bool ok = gi < p.L;
    s.beta[tid] = ok ? clamp_beta(p.beta[in_row + gi]) : 0.f;
    s.lse2[tid] = ok ? p.lse[in_row + gi] * kLog2e : INFINITY;
    s.dv[tid] = p.Dv[ws_row + tid];
  }
  {  // dQ<-, dK->, dF as bf16 operand tiles (2 threads per row, 32 columns each)
    const int r = tid >> 1, h = tid & 1;
    const bool ok = row0 + r < p.L;
    float x[64];
    const float* dqs = p.dql + (ws_row + r) * D;
    const float* dks = p.dkr + (ws_row + r) * D;
    const float* dfs = p.df + (((size_t)bh * p.nc + c) * D + r) * D;
    for (int j = 0; j < 64; ++j) x[j] = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) x[32 * h + j] = ok ? dqs[32 * h + j] : 0.f;
    // each thread writes its 4 chunks of 16 bytes (8 bf16) of the row
#pragma unroll
    for (int qq = 4 * h; qq < 4 * h + 4; ++qq)
      *reinterpret_cast<uint4*>(s.t[T_DQ] + r * 128 + ((qq ^ (r & 7)) * 16)) =
          make_uint4(pack_bf16(x[8 * qq], x[8 * qq + 1]), pack_bf16(x[8 * qq + 2], x[8 * qq + 3]),
                     pack_bf16(x[8 * qq + 4], x[8 * qq + 5]), pack_bf16(x[8 * qq + 6], x[8 * qq + 7]));
#pragma unroll
    for (int j = 0; j < 32; ++j) x[32 * h + j] = ok ? dks[32 * h + j] : 0.f;
#pragma unroll
    for (int qq = 4 * h; qq < 4 * h + 4; ++qq)
      *reinterpret_cast<uint4*>(s.t[T_DK] + r * 128 + ((qq ^ (r & 7)) * 16)) =
          make_uint4(pack_bf16(x[8 * qq], x[8 * qq + 1]), pack_bf16(x[8 * qq + 2], x[8 * qq + 3]),
                     pack_bf16(x[8 * qq + 4], x[8 * qq + 5]), pack_bf16(x[8 * qq + 6], x[8 * qq + 7]));
#pragma unroll
    for (int j = 0; j < 32; ++j) x[32 * h + j] = dfs[32 * h + j];
#pragma unroll
    for (int qq = 4 * h; qq < 4 * h + 4; ++qq)
      *reinterpret_cast<uint4*>(s.t[T_DF] + r * 128 + ((qq ^ (r & 7)) * 16)) =
          make_uint4(pack_bf16(x[8 * qq], x[8 * qq + 1]), pack_bf16(x[8 * qq + 2], x[8 * qq + 3]),
                     pack_bf16(x[8 * qq + 4], x[8 * qq + 5]), pack_bf16(x[8 * qq + 6], x[8 * qq + 7]));
  }
  mbar_wait(&s.bar_in, 0, p.err, 41);
  if (row0 + B > p.L) {  // rows beyond L are zero
    for (int r = tid; r < B; r += 128)
      if (row0 + r >= p.L)
        for (int si = 0; si < 5; ++si) {
          const int slot = si == 0 ? T_W : si == 1 ? T_Q : si == 2 ? T_K : si == 3 ? T_V : T_DO;
          for (int qq = 0; qq < 8; ++qq) reinterpret_cast<uint4*>(s.t[slot] + r * 128)[qq] = make_uint4(0, 0, 0, 0);
        }
  }
  publish();

  // ---- P2: G, M1, N2, QK^T, dP ----
  run([&] {
    mma64(tb + 0, ta(T_W), 0, ta(T_W), 0, 0);
    mma64(tb + 64, ta(T_Q), 0, ta(T_W), 0, 0);
    mma64(tb + 128, ta(T_W), 0, ta(T_K), 0, 0);
    mma64(tb + 192, ta(T_Q), 0, ta(T_K), 0, 0);
    mma64(tb + 256, ta(T_DO), 0, ta(T_V), 0, 0);
  }, 42);
  {
    float x[64];
    ld_row(tb, lane_off, 0, x);
    if (has_row) {
#pragma unroll
      for (int j = 0; j < 64; ++j) s.g[i * GS + j] = j < i ? x[j] : 0.f;
    }
    ld_row(tb, lane_off, 64, x);
    if (has_row) {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = j <= i ? x[j] : 0.f;
      put_row(s.t[T_M1], i, x);
    }
    ld_row(tb, lane_off, 128, x);
    if (has_row) {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = j < i ? x[j] : 0.f;
      put_row(s.t[T_N2], i, x);
    }
  }
  publish();

  // ---- P3: Y = T^{-1} (fp32 forward substitution, lane = column), U = Y diag(beta) ----
  if (warp < 2) {
    const int cc = 32 * warp + lane;
    float yc[64];
#pragma unroll
    for (int r = 0; r < 64; ++r) {
      float a0 = 0.f, a1 = 0.f;
#pragma unroll
      for (int m = 0; m + 1 < r; m += 2) {
        a0 += s.g[r * GS + m] * yc[m];
        a1 += s.g[r * GS + m + 1] * yc[m + 1];
      }
      if (r & 1) a0 += s.g[r * GS + r - 1] * yc[r - 1];
      yc[r] = (cc == r ? 1.f : 0.f) - s.beta[r] * (a0 + a1);
    }
    const float bc = s.beta[cc];
#pragma unroll
    for (int r = 0; r < 64; ++r) {
      s.y[r * GS + cc] = yc[r];
      *reinterpret_cast<__nv_bfloat16*>(s.t[T_Y] + sw128_offset(r, cc)) = __float2bfloat16_rn(yc[r]);
      *reinterpret_cast<__nv_bfloat16*>(s.t[T_U] + sw128_offset(r, cc)) = __float2bfloat16_rn(yc[r] * bc);
    }
  }
  publish();

  // ---- P4: X = U N2, Y1 = U W ----
  run([&] {
    mma64(tb + 0, ta(T_U), 0, ta(T_N2), 1, 0);
    mma64(tb + 64, ta(T_U), 0, ta(T_W), 1, 0);
  }, 43);
  {
    float x[64];
    ld_row(tb, lane_off, 0, x);
    if (has_row) put_row(s.t[T_X], i, x);
    ld_row(tb, lane_off, 64, x);
    if (has_row) put_row(s.t[T_Y1], i, x);
  }
  publish();

  // ---- P5: S_d = QK^T - M1 X ; P ; dS = scale P (dP - D) ----
  run([&] { mma64(tb + 192, ta(T_M1), 0, ta(T_X), 1, 1, 1); }, 44);
  {
    float sx[64], dp[64];
    ld_row(tb, lane_off, 192, sx);
    ld_row(tb, lane_off, 256, dp);
    if (has_row) {
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        const float pj = (j <= i && row_ok) ? fast_exp2(sx[j] * p.scl - s.lse2[i]) : 0.f;
        sx[j] = pj;
        dp[j] = p.scale * pj * (dp[j] - s.dv[i]);
      }
      put_row(s.t[T_P], i, sx);
      put_row(s.t[T_DS], i, dp);
    }
  }
  publish();

  // ---- P6: dvp = P^T dO ; gQ = dS K ; gK = dS^T Q ; gM1 = -dS X^T - dQ<- Y1^T ; gX = -M1^T dS - W dK->^T ----
  run([&] {
    mma64(tb + 0, ta(T_P), 1, ta(T_DO), 1, 0);
    mma64(tb + C_GQ, ta(T_DS), 0, ta(T_K), 1, 0);
    mma64(tb + C_GK, ta(T_DS), 1, ta(T_Q), 1, 0);
    mma64(tb + 64, ta(T_DS), 0, ta(T_X), 0, 0, 1);
    mma64(tb + 64, ta(T_DQ), 0, ta(T_Y1), 0, 1, 1);
    mma64(tb + 128, ta(T_M1), 1, ta(T_DS), 1, 0, 1);
    mma64(tb + 128, ta(T_W), 0, ta(T_DK), 0, 1, 1);
  }, 45);
  {
    float x[64];
    ld_row(tb, lane_off, 0, x);
    if (row_ok) {
      const size_t orow = in_row + row0 + i;
      const float* acc = p.dvacc + (ws_row + i) * D;
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] += acc[j];
      store_bf16_row(p.dv + orow * D, x);
    }
    ld_row(tb, lane_off, 64, x);
    if (has_row) {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = j <= i ? x[j] : 0.f;
      put_row(s.t[T_GM1], i, x);
    }
    ld_row(tb, lane_off, 128, x);
    if (has_row) put_row(s.t[T_GX], i, x);
  }
  publish();

  // ---- P7: E3 = M1^T dQ<- + W dF^T ; gN2 = U^T gX ; gW = -X dK-> - Y1 dF + gM1^T Q ; gQ += gM1 W ----
  run([&] {
    mma64(tb + 0, ta(T_M1), 1, ta(T_DQ), 1, 0);
    mma64(tb + 0, ta(T_W), 0, ta(T_DF), 0, 1);
    mma64(tb + 64, ta(T_U), 1, ta(T_GX), 1, 0);
    mma64(tb + C_GW, ta(T_X), 0, ta(T_DK), 1, 0, 1);
    mma64(tb + C_GW, ta(T_Y1), 0, ta(T_DF), 1, 1, 1);
    mma64(tb + C_GW, ta(T_GM1), 1, ta(T_Q), 1, 1);
    mma64(tb + C_GQ, ta(T_GM1), 0, ta(T_W), 1, 1);
  }, 46);
  {
    float x[64];
    ld_row(tb, lane_off, 0, x);
    if (has_row) put_row(s.t[T_E3], i, x);
    ld_row(tb, lane_off, 64, x);
    if (has_row) {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = j < i ? x[j] : 0.f;
      put_row(s.t[T_GN2], i, x);
    }
  }
  publish();

  // ---- P8: gU = -E3 W^T + gX N2^T ; gW += -U^T E3 + gN2 K ; gK += gN2^T W ----
  run([&] {
    mma64(tb + 0, ta(T_E3), 0, ta(T_W), 0, 0, 1);
    mma64(tb + 0, ta(T_GX), 0, ta(T_N2), 0, 1);
    mma64(tb + C_GW, ta(T_U), 1, ta(T_E3), 1, 1, 1);
    mma64(tb + C_GW, ta(T_GN2), 0, ta(T_K), 1, 1);
    mma64(tb + C_GK, ta(T_GN2), 1, ta(T_W), 1, 1);
  }, 47);
  {
    float x[64];
    ld_row(tb, lane_off, 0, x);
    if (has_row) {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = j <= i ? x[j] : 0.f;
      put_row(s.t[T_GU], i, x);
      // gU .* Y in place of Y (its fp32 copy has no other use); column sums give dbeta
#pragma unroll
      for (int j = 0; j < 64; ++j) s.y[i * GS + j] *= x[j];
    }
  }
  // diag(beta) W (Y1's slot is free now)
  if (tid < B) {
    float x[64];
    get_row(s.t[T_W], tid, x);
    const float bt = s.beta[tid];
#pragma unroll
    for (int j = 0; j < 64; ++j) x[j] *= bt;
    put_row(s.t[T_BW], tid, x);
  }
  publish();

  // ---- P9: A1 = gU U^T ; dbeta_j = sum_i gU_ij Y_ij ----
  run([&] { mma64(tb + 64, ta(T_GU), 0, ta(T_U), 0, 0); }, 48);
  if (tid < B) {
    float acc = 0.f;
    for (int r = tid; r < B; ++r) acc += s.y[r * GS + tid];
    s.gb[tid] = acc;
  }
  {
    float x[64];
    ld_row(tb, lane_off, 64, x);
    if (has_row) put_row(s.t[T_A1], i, x);
  }
  publish();

  // ---- P10: gN = strictLower(-Y^T A1) ; dbeta_i += sum_{j<i} gN_ij G_ij ----
  run([&] { mma64(tb + 128, ta(T_Y), 1, ta(T_A1), 1, 0, 1); }, 49);
  {
    float x[64];
    ld_row(tb, lane_off, 128, x);
    if (has_row) {
      float acc = 0.f;
#pragma unroll
      for (int j = 0; j < 64; ++j) {
        x[j] = j < i ? x[j] : 0.f;
        acc += x[j] * s.g[i * GS + j];
      }
      s.gb[i] += acc;
      put_row(s.t[T_GN], i, x);
      const float bi = s.beta[i];
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] *= bi;
      put_row(s.t[T_GNB], i, x);
    }
  }
  publish();

  // ---- P11: gW += diag(beta) gN W + gN^T diag(beta) W ----
  run([&] {
    mma64(tb + C_GW, ta(T_GNB), 0, ta(T_W), 1, 1);
    mma64(tb + C_GW, ta(T_GN), 1, ta(T_BW), 1, 1);
  }, 50);

  // ---- outputs ----
  {
    float x[64];
    const size_t orow = in_row + row0 + i;
    ld_row(tb, lane_off, C_GQ, x);
    if (row_ok) {
      const float* a = p.dql + (ws_row + i) * D;
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] += a[j];
      store_bf16_row(p.dq + orow * D, x);
    }
    ld_row(tb, lane_off, C_GK, x);
    if (row_ok) {
      const float* a = p.dkr + (ws_row + i) * D;
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] += a[j];
      store_bf16_row(p.dk + orow * D, x);
    }
    ld_row(tb, lane_off, C_GW, x);
    if (row_ok) store_bf16_row(p.dw + orow * D, x);
  }
  __syncthreads();
  if (tid < B && row0 + tid < p.L) p.dbeta[in_row + row0 + tid] = s.gb[tid];
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, 512);
  }
}

}  // namespace

cudaError_t launch_ut_bwd64(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                            const float* beta, const float* lse, const void* dO, const float* Dv, const float* dql,
                            const float* dkr, const float* dvacc, const float* df, void* dq, void* dk, void* dv,
                            void* dw, float* dbeta, int* err, cudaStream_t st) {
  if (g.B != 64) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv, mw, mdo;
  const uint64_t rows = (uint64_t)g.BH * g.L;
  if (!make_map_rows64(&mq, q, rows, B) || !make_map_rows64(&mk, k, rows, B) || !make_map_rows64(&mv, v, rows, B) ||
      !make_map_rows64(&mw, w, rows, B) || !make_map_rows64(&mdo, dO, rows, B))
    return cudaErrorInvalidValue;
  UbParams p;
  p.L = g.L;
  p.Lp = g.Lp;
  p.nc = g.nc;
  p.BH = g.BH;
  p.scale = g.scale;
  p.scl = g.scale * kLog2e;
  p.beta = beta;
  p.lse = lse;
  p.Dv = Dv;
  p.dql = dql;
  p.dkr = dkr;
  p.dvacc = dvacc;
  p.df = df;
  p.dq = (__nv_bfloat16*)dq;
  p.dk = (__nv_bfloat16*)dk;
  p.dv = (__nv_bfloat16*)dv;
  p.dw = (__nv_bfloat16*)dw;
  p.dbeta = dbeta;
  p.err = err;
  const size_t smem = sizeof(UbSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(ut_bwd64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ut_bwd64_kernel<<<dim3(g.nc, g.BH), 128, smem, st>>>(mq, mk, mv, mw, mdo, p);
  return cudaGetLastError();
}

}  // namespace pathattn
