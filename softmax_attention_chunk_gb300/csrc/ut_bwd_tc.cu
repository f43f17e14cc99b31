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
// K-major or MN-major per operand.  The schedule keeps at most four 64-column accumulators in
// TMEM (256 columns) and thirteen tiles in shared memory (Q and K are re-read by TMA after their
// slots have served other operands), so that two CTAs share an SM and hide each other's phase
// latencies.  Accumulator rows are read with the 16x32bx2 shape: every thread of a warp holds
// 32 columns of one of the warp's 16 rows.
#include "internal.h"
#include "dev_common.cuh"
#include "tc_common.cuh"
#include "ut_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace pathattn {

bool make_map_head_rows64(CUtensorMap* m, const void* base, uint64_t L, uint64_t heads);  // fwd_tc.cu

namespace {
using namespace tc;

constexpr int B = 64;
constexpr int D = kHeadDim;
constexpr uint32_t TILE = 64 * 128;
constexpr uint32_t C0 = 0, C1 = 64, C2 = 128, C3 = 192;  // TMEM accumulator columns

// Shared-memory tile slots.  A slot takes a new tenant once every MMA and thread that reads the
// previous one has finished (phases in brackets).
enum {
  S_W,   // W [all]
  S_Q,   // Q [P2] | L fp32 low half [P2-P3] | P [P5-P6] | gM1 [P6-P7] | gU [P8-P9]
  S_K,   // K [P2] | L fp32 high half [P2-P3] | dS [P5-P8] | diag(beta) W [P8-P11]
  S_V,   // V [P3] | dF [P3-P7] | gN2 [P7-P8] | A1 [P9-P10]
  S_DO,  // dO [P3-P6] | gX [P6-P8] | gU.*Y fp32 low half [P8-P9] | diag(beta) gN [P10-P11]
  S_M1,  // M1 [P2-P7] | gU.*Y fp32 high half [P8-P9]
  S_N2,  // N2 [P2-P8] | gN [P10-P11]
  S_U,   // U [P3-P9]
  S_Y,   // Y [P3-P10]
  S_DQ,  // dQ<- [P3-P7] | E3 [P7-P8]
  S_DK,  // dK-> [P3-P6]
  S_X,   // X [P4-P6] | Q again [P7-P8]
  S_Y1,  // Y1 [P4-P6] | K again [P7-P8]
  NSLOT
};
constexpr int S_G = S_Q, S_P = S_Q, S_GM1 = S_Q, S_GU = S_Q, S_DS = S_K, S_BW = S_K, S_DF = S_V, S_GN2 = S_V,
              S_A1 = S_V, S_GX = S_DO, S_SCR = S_DO, S_GNB = S_DO, S_GN = S_N2, S_E3 = S_DQ, S_Q2 = S_X,
              S_K2 = S_Y1;

struct __align__(1024) UbSmem {
  uint8_t t[NSLOT][TILE];
  float beta[B], lse2[B], dv[B], gb[B];
  uint64_t bar_in, bar_mma;
  uint32_t tmem_base;
  float pre[B];  // PaTH-FoX: chunk-local inclusive prefix of log f
  uint64_t bar_mma2;  // the second issuer's commits (phases whose MMAs two threads issue)
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
  const float* logf;  // PaTH-FoX: log f [BH][L]
  float* fxcs;        // PaTH-FoX: column sums of dS' (accumulated) [BH][Lp]
};

// FOX (PaTH-FoX, notes §2.5): the diagonal logits gain pre_i - pre_j (chunk-local prefix sums of
// log f) and the column sums of the chunk's dS' are added into fxcs.
template <bool FOX>
__global__ void __launch_bounds__(128, 2) ut_bwd64_kernel(const __grid_constant__ CUtensorMap tm_q,
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
  // this thread's half row of the M=64 accumulators: row i, columns 32h .. 32h+31
  const int i = 16 * warp + (lane & 15), h = lane >> 4;
  const bool row_ok = row0 + i < p.L;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  auto ta = [&](int slot) { return smem_u32(s.t[slot]); };
  float* sg = reinterpret_cast<float*>(s.t[S_G]);
  float* scr = reinterpret_cast<float*>(s.t[S_SCR]);

  if (lead) {
    mbar_init(&s.bar_in, 1);
    mbar_init(&s.bar_mma, 1);
    mbar_init(&s.bar_mma2, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&s.tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  uint32_t mph = 0;
  auto issue = [&](auto fn) {  // the lead thread issues one phase's MMAs and commits them
    if (lead) {
      tc_fence_after();
      fn();
      mma_commit(&s.bar_mma);
    }
  };
  // Phases with many products split them over two issuing threads (a tcgen05.mma costs tens of
  // cycles to issue), by accumulator so that every accumulation chain stays in one thread's order.
  uint32_t mph2 = 0;
  auto issue2 = [&](auto fa, auto fb) {
    if (lead) {
      tc_fence_after();
      fa();
      mma_commit(&s.bar_mma);
    } else if (tid == 32) {
      tc_fence_after();
      fb();
      mma_commit(&s.bar_mma2);
    }
  };
  auto wait_mma2 = [&](int code) {
    mbar_wait_lean(&s.bar_mma, mph, p.err, code);
    mbar_wait_lean(&s.bar_mma2, mph2, p.err, code);
    mph ^= 1;
    mph2 ^= 1;
    tc_fence_after();
  };
  auto wait_mma = [&](int code) {
    mbar_wait_lean(&s.bar_mma, mph, p.err, code);
    mph ^= 1;
    tc_fence_after();
  };
  auto publish = [&]() {  // tiles written by the threads -> visible to the next MMAs
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  };

  // ---- loads: W, Q, K, V, dO by TMA (rows >= L read as zero); the fp32 gradients that the
  //      epilogues read later are brought into L2 meanwhile ----
  if (lead) {
    bulk_prefetch_l2(p.dql + ws_row * D, B * D * 4);
    bulk_prefetch_l2(p.dkr + ws_row * D, B * D * 4);
    bulk_prefetch_l2(p.dvacc + ws_row * D, B * D * 4);
    bulk_prefetch_l2(p.df + ((size_t)bh * p.nc + c) * D * D, D * D * 4);
    mbar_arrive_expect_tx(&s.bar_in, 5 * TILE);
    tma_load_3d(s.t[S_W], &tm_w, 0, row0, bh, &s.bar_in);
    tma_load_3d(s.t[S_Q], &tm_q, 0, row0, bh, &s.bar_in);
    tma_load_3d(s.t[S_K], &tm_k, 0, row0, bh, &s.bar_in);
    tma_load_3d(s.t[S_V], &tm_v, 0, row0, bh, &s.bar_in);
    tma_load_3d(s.t[S_DO], &tm_do, 0, row0, bh, &s.bar_in);
  }
  if (tid < B) {
    const int gi = row0 + tid;
    const bool ok = gi < p.L;
    s.beta[tid] = ok ? clamp_beta(p.beta[in_row + gi]) : 0.f;
    s.lse2[tid] = ok ? p.lse[in_row + gi] * kLog2e : INFINITY;
    s.dv[tid] = p.Dv[ws_row + tid];
  }
  if constexpr (FOX) {
    if (warp == 3) {  // chunk-local inclusive prefix of log f
      const int ga = row0 + lane, gb2 = row0 + 32 + lane;
      float a = ga < p.L ? p.logf[in_row + ga] : 0.f;
      float b2 = gb2 < p.L ? p.logf[in_row + gb2] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float ta = __shfl_up_sync(0xffffffffu, a, o), tb2 = __shfl_up_sync(0xffffffffu, b2, o);
        if (lane >= o) {
          a += ta;
          b2 += tb2;
        }
      }
      const float tot_a = __shfl_sync(0xffffffffu, a, 31);
      s.pre[lane] = a;
      s.pre[32 + lane] = b2 + tot_a;
    }
  }
  mbar_wait_lean(&s.bar_in, 0, p.err, 41);
  publish();

  // ---- P2: G = W W^T, M1 = Q W^T, N2 = W K^T, Q K^T ----
  issue2([&] {
    mma64(tb + C0, ta(S_W), 0, ta(S_W), 0, 0);
    mma64(tb + C1, ta(S_Q), 0, ta(S_W), 0, 0);
  }, [&] {
    mma64(tb + C2, ta(S_W), 0, ta(S_K), 0, 0);
    mma64(tb + C3, ta(S_Q), 0, ta(S_K), 0, 0);
  });
  wait_mma2(42);
  {
    float x[32];
    ld_half(tb, lane_off, C0, x);  // L = strictLower(diag(beta) G), fp32 into the slots of Q and K
    const float bi = s.beta[i];
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const int j = 32 * h + 4 * q;
      *reinterpret_cast<float4*>(sg + f32_idx(i, j)) =
          make_float4(j < i ? bi * x[4 * q] : 0.f, j + 1 < i ? bi * x[4 * q + 1] : 0.f,
                      j + 2 < i ? bi * x[4 * q + 2] : 0.f, j + 3 < i ? bi * x[4 * q + 3] : 0.f);
    }
    ld_half(tb, lane_off, C1, x);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = 32 * h + j <= i ? x[j] : 0.f;
    put_half(s.t[S_M1], i, h, x);
    ld_half(tb, lane_off, C2, x);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = 32 * h + j < i ? x[j] : 0.f;
    put_half(s.t[S_N2], i, h, x);
  }
  publish();

  // ---- P3: dP = dO V^T goes to the tensor core first (its accumulator is free).  Warps 0-1 solve
  //      the diagonal blocks of Y = (I + strictLower(D G))^{-1} and write them (and U = Y D) as bf16
  //      tiles while warps 2-3 write dQ<- and dK-> as bf16 operand tiles (coalesced loads) and dF into
  //      V's slot once dP has read V; then all
  //      four warps form the off-diagonal block ----
  if (tid == 64) {
    tc_fence_after();
    mma64(tb + C2, ta(S_DO), 0, ta(S_V), 0, 0);
    mma_commit(&s.bar_mma);
  }
  if (warp < 2) {
    ut_inv_diag64(sg, s.beta, s.t[S_U], s.t[S_Y], tid);
  } else {
    {  // dQ<- and dK-> (prefetched into L2 at the start), zero past L
      RowsToTile<2> t;
      t.load(p.dql + ws_row * D, min(B, p.L - row0), warp - 2, lane);
      t.store(s.t[S_DQ], warp - 2, lane);
      t.load(p.dkr + ws_row * D, min(B, p.L - row0), warp - 2, lane);
      t.store(s.t[S_DK], warp - 2, lane);
    }
    RowsToTile<2> f;
    f.load(p.df + ((size_t)bh * p.nc + c) * D * D, B, warp - 2, lane);
    mbar_wait_lean(&s.bar_mma, mph, p.err, 52);  // dP has read V
    f.store(s.t[S_DF], warp - 2, lane);
  }
  mph ^= 1;
  ut_sync();  // the diagonal blocks of Y are in sl
  ut_inv_offdiag128(sg, s.beta, s.t[S_U], s.t[S_Y], tid);
  publish();

  // ---- P4: X = U N2, Y1 = U W ----
  issue([&] {
    mma64(tb + C0, ta(S_U), 0, ta(S_N2), 1, 0);
    mma64(tb + C1, ta(S_U), 0, ta(S_W), 1, 0);
  });
  wait_mma(43);
  {
    float x[32];
    ld_half(tb, lane_off, C0, x);
    put_half(s.t[S_X], i, h, x);
    ld_half(tb, lane_off, C1, x);
    put_half(s.t[S_Y1], i, h, x);
  }
  publish();

  // ---- P5: S_d = Q K^T - M1 X ; P ; dS = scale P (dP - D_i) ----
  issue([&] { mma64(tb + C3, ta(S_M1), 0, ta(S_X), 1, 1, 1); });
  wait_mma(44);
  {
    float sx[32], dp[32];
    ld_half(tb, lane_off, C3, sx);
    ld_half(tb, lane_off, C2, dp);
    const float l2 = s.lse2[i], dvi = s.dv[i];
    const float fox_i = FOX ? s.pre[i] * kLog2e - l2 : -l2;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      const float off = FOX ? fmaf(-s.pre[32 * h + j], kLog2e, fox_i) : fox_i;
      const float pj = (32 * h + j <= i && row_ok) ? fast_exp2(fmaf(sx[j], p.scl, off)) : 0.f;
      sx[j] = pj;
      dp[j] = p.scale * pj * (dp[j] - dvi);
    }
    put_half(s.t[S_P], i, h, sx);
    put_half(s.t[S_DS], i, h, dp);
    if constexpr (FOX) {
      // the row's sum of dS' (this half) leaves fxcs_i = colsum_i - rowsum_i ...
      float rs = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) rs += dp[j];
      atomicAdd(p.fxcs + ws_row + i, -rs / p.scale);
      // ... and the column sums of dS' over the half-warp's 16 rows (reduce-scatter: lane l keeps
      // columns 2 (l % 16), 2 (l % 16) + 1 of its half) are added
#pragma unroll
      for (int o = 8; o >= 1; o >>= 1) {
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int j = 0; j < 2 * o; ++j) {
          const float send = up ? dp[j] : dp[j + 2 * o];
          const float keep = up ? dp[j + 2 * o] : dp[j];
          dp[j] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
      }
      const float inv_scale = 1.f / p.scale;
      float* cs = p.fxcs + ws_row + 32 * h + 2 * (lane & 15);
      atomicAdd(cs, dp[0] * inv_scale);
      atomicAdd(cs + 1, dp[1] * inv_scale);
    }
  }
  publish();

  // ---- P6: dV_diag = P^T dO ; gM1 = -dS X^T - dQ<- Y1^T ; gX = -M1^T dS - W dK->^T ;
  //          gW = -X dK-> - Y1 dF ----
  issue2([&] {
    mma64(tb + C0, ta(S_P), 1, ta(S_DO), 1, 0);
    mma64(tb + C1, ta(S_DS), 0, ta(S_X), 0, 0, 1);
    mma64(tb + C1, ta(S_DQ), 0, ta(S_Y1), 0, 1, 1);
  }, [&] {
    mma64(tb + C2, ta(S_M1), 1, ta(S_DS), 1, 0, 1);
    mma64(tb + C2, ta(S_W), 0, ta(S_DK), 0, 1, 1);
    mma64(tb + C3, ta(S_X), 0, ta(S_DK), 1, 0, 1);
    mma64(tb + C3, ta(S_Y1), 0, ta(S_DF), 1, 1, 1);
  });
  {
    float x[32], a[32];
    if (row_ok) load_f32_half(p.dvacc + (ws_row + i) * D + 32 * h, a);  // in flight during the MMAs
    wait_mma2(45);
    if (lead) {  // X and Y1 are consumed: Q and K come back into their slots
      mbar_arrive_expect_tx(&s.bar_in, 2 * TILE);
      tma_load_3d(s.t[S_Q2], &tm_q, 0, row0, bh, &s.bar_in);
      tma_load_3d(s.t[S_K2], &tm_k, 0, row0, bh, &s.bar_in);
    }
    ld_half(tb, lane_off, C0, x);
    if (row_ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] += a[j];
      store_bf16_half(p.dv + (in_row + row0 + i) * D + 32 * h, x);
    }
    ld_half(tb, lane_off, C1, x);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = 32 * h + j <= i ? x[j] : 0.f;
    put_half(s.t[S_GM1], i, h, x);
    ld_half(tb, lane_off, C2, x);
    put_half(s.t[S_GX], i, h, x);
  }
  publish();

  // ---- P7: gQ = dS K + gM1 W ; E3 = M1^T dQ<- + W dF^T ; gN2 = U^T gX ; gW += gM1^T Q ----
  if (lead || tid == 32) mbar_wait_lean(&s.bar_in, 1, p.err, 46);  // both issuers read Q and K again
  issue2([&] {
    mma64(tb + C0, ta(S_DS), 0, ta(S_K2), 1, 0);
    mma64(tb + C0, ta(S_GM1), 0, ta(S_W), 1, 1);
    mma64(tb + C1, ta(S_M1), 1, ta(S_DQ), 1, 0);
    mma64(tb + C1, ta(S_W), 0, ta(S_DF), 0, 1);
  }, [&] {
    mma64(tb + C2, ta(S_U), 1, ta(S_GX), 1, 0);
    mma64(tb + C3, ta(S_GM1), 1, ta(S_Q2), 1, 1);
  });
  {
    float x[32], a[32];
    if (row_ok) load_f32_half(p.dql + (ws_row + i) * D + 32 * h, a);
    wait_mma2(47);
    ld_half(tb, lane_off, C0, x);
    if (row_ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] += a[j];
      store_bf16_half(p.dq + (in_row + row0 + i) * D + 32 * h, x);
    }
    ld_half(tb, lane_off, C1, x);
    put_half(s.t[S_E3], i, h, x);
    ld_half(tb, lane_off, C2, x);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = 32 * h + j < i ? x[j] : 0.f;
    put_half(s.t[S_GN2], i, h, x);
  }
  publish();

  // ---- P8: gK = dS^T Q + gN2^T W ; gU = -E3 W^T + gX N2^T ; gW += -U^T E3 + gN2 K ----
  issue2([&] {
    mma64(tb + C0, ta(S_DS), 1, ta(S_Q2), 1, 0);
    mma64(tb + C0, ta(S_GN2), 1, ta(S_W), 1, 1);
    mma64(tb + C1, ta(S_E3), 0, ta(S_W), 0, 0, 1);
    mma64(tb + C1, ta(S_GX), 0, ta(S_N2), 0, 1);
  }, [&] {
    mma64(tb + C3, ta(S_U), 1, ta(S_E3), 1, 1, 1);
    mma64(tb + C3, ta(S_GN2), 0, ta(S_K2), 1, 1);
  });
  {
    float x[32], a[32];
    if (row_ok) load_f32_half(p.dkr + (ws_row + i) * D + 32 * h, a);
    wait_mma2(48);
    ld_half(tb, lane_off, C0, x);
    if (row_ok) {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] += a[j];
      store_bf16_half(p.dk + (in_row + row0 + i) * D + 32 * h, x);
    }
    ld_half(tb, lane_off, C1, x);
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = 32 * h + j <= i ? x[j] : 0.f;
    put_half(s.t[S_GU], i, h, x);
    // gU .* Y (fp32) for the column sums that give dbeta
    get_half(s.t[S_Y], i, h, a);
#pragma unroll
    for (int q = 0; q < 8; ++q)
      *reinterpret_cast<float4*>(scr + f32_idx(i, 32 * h + 4 * q)) =
          make_float4(x[4 * q] * a[4 * q], x[4 * q + 1] * a[4 * q + 1], x[4 * q + 2] * a[4 * q + 2],
                      x[4 * q + 3] * a[4 * q + 3]);
    // diag(beta) W
    get_half(s.t[S_W], i, h, x);
    const float bi = s.beta[i];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] *= bi;
    put_half(s.t[S_BW], i, h, x);
  }
  publish();

  // ---- P9: A1 = gU U^T ; G again (for dbeta) ; dbeta_j = sum_i gU_ij Y_ij ----
  issue([&] {
    mma64(tb + C0, ta(S_GU), 0, ta(S_U), 0, 0);
    mma64(tb + C2, ta(S_W), 0, ta(S_W), 0, 0);
  });
  if (tid < B) {  // column sums; the rows above the diagonal hold exact zeros (gU and Y are lower)
    float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;
#pragma unroll
    for (int r = 0; r < B; r += 4) {
      a0 += scr[f32_idx(r, tid)];
      a1 += scr[f32_idx(r + 1, tid)];
      a2 += scr[f32_idx(r + 2, tid)];
      a3 += scr[f32_idx(r + 3, tid)];
    }
    s.gb[tid] = (a0 + a1) + (a2 + a3);
  }
  wait_mma(49);
  {
    float x[32];
    ld_half(tb, lane_off, C0, x);
    put_half(s.t[S_A1], i, h, x);
  }
  publish();

  // ---- P10: gN = strictLower(-Y^T A1) ; dbeta_i += sum_{j<i} gN_ij G_ij ----
  issue([&] { mma64(tb + C1, ta(S_Y), 1, ta(S_A1), 1, 0, 1); });
  wait_mma(50);
  {
    float x[32], g[32];
    ld_half(tb, lane_off, C1, x);
    ld_half(tb, lane_off, C2, g);
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      x[j] = 32 * h + j < i ? x[j] : 0.f;
      acc += x[j] * g[j];
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 16);
    if (h == 0) s.gb[i] += acc;
    put_half(s.t[S_GN], i, h, x);
    const float bi = s.beta[i];
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] *= bi;
    put_half(s.t[S_GNB], i, h, x);
  }
  publish();

  // ---- P11: gW += diag(beta) gN W + gN^T diag(beta) W ; outputs dw, dbeta ----
  issue([&] {
    mma64(tb + C3, ta(S_GNB), 0, ta(S_W), 1, 1);
    mma64(tb + C3, ta(S_GN), 1, ta(S_BW), 1, 1);
  });
  wait_mma(51);
  {
    float x[32];
    ld_half(tb, lane_off, C3, x);
    if (row_ok) store_bf16_half(p.dw + (in_row + row0 + i) * D + 32 * h, x);
  }
  tc_fence_before();
  __syncthreads();
  if (tid < B && row0 + tid < p.L) p.dbeta[in_row + row0 + tid] = s.gb[tid];
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, 256);
  }
}

}  // namespace

cudaError_t launch_ut_bwd64(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                            const float* beta, const float* lse, const void* dO, const float* Dv, const float* dql,
                            const float* dkr, const float* dvacc, const float* df, void* dq, void* dk, void* dv,
                            void* dw, float* dbeta, int* err, cudaStream_t st, const float* logf, float* fxcs) {
  if (g.B != 64) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv, mw, mdo;
  if (!make_map_head_rows64(&mq, q, g.L, g.BH) || !make_map_head_rows64(&mk, k, g.L, g.BH) ||
      !make_map_head_rows64(&mv, v, g.L, g.BH) || !make_map_head_rows64(&mw, w, g.L, g.BH) ||
      !make_map_head_rows64(&mdo, dO, g.L, g.BH))
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
  p.logf = logf;
  p.fxcs = fxcs;
  const size_t smem = sizeof(UbSmem) + 1024;
  auto kern = logf ? ut_bwd64_kernel<true> : ut_bwd64_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                           (int)cudaSharedmemCarveoutMaxShared);
  if (e != cudaSuccess) return e;
  kern<<<dim3(g.nc, g.BH), 128, smem, st>>>(mq, mk, mv, mw, mdo, p);
  return cudaGetLastError();
}

}  // namespace pathattn
