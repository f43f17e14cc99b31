// Per-chunk UT preparation on tcgen05 at head dim 128 (bf16 operands, fp32 accumulation in TMEM),
// chunk B = 64: persistent CTAs of 128 threads, two per SM, each taking chunk after chunk.
//
// Method: PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.6 (UT representation) and §2.7
// (boundary-adjusted queries/keys, chunk transform), the same quantities as at head dim 64:
//   G = strictLower(W W^T), M1 = lower(Q W^T), N2 = strictLower(W K^T)
//   U = (I + strictLower(D G))^{-1} D        (fp32, two-level block inversion)
//   A = M1 U,  X = U N2,  Y = U^T W
//   Q<- = Q - A W,  K-> = K - X^T W,  F = I - W^T Y,  S_d = Q K^T - M1 X (masked j <= i)
// and the diagonal chunk's softmax partial state (m, l, acc = P V).
//
// Every operand with a head-dim side (W, K, Q, V, Y, and the outputs) is held as two 64-column
// halves x = a, b (columns 0-63, 64-127), each a 64 x 64 bf16 tile in the 128-byte swizzled layout,
// so every product is built from the head-dim-64 kernel's M=64 N=64 K=64 MMAs:
//   products over d (G, N2, M1, Q K^T) add the two halves' MMAs (K = 128);
//   products onto d (Y, A W, X^T W, P V) form one 64-column accumulator per half;
//   F (128 x 128) is four 64 x 64 blocks F_xy = delta_xy I - W_x^T Y_y.
// TMEM: 256 columns (four 64-column accumulators), two CTAs per SM.  Tile slots (thirteen, 8 KB):
//   0 W_a, 1 K_a, 2 W_b, 3 K_b   P1 .. (the pairs [W_x; K_x] are adjacent: one N=128 MMA per half)
//   4 Q_a, 5 Q_b                 P1 .. R3 epilogue
//   6-7 fp32 L (P1 .. P2), then A (6) and X (7) (R1 .. R3)
//   8 N2 (P1 .. R1), then Y_a (R2 .. R4)
//   9 U^T (P2 .. R2), then V_a (loaded once R2 has read U)
//   10 M1 (P2 .. R2), then Y_b (R2 .. R4)
//   11 P (R2 .. R5)
//   12 V_b (loaded with the inputs)
// Rounds: P1 [G | N2]; M1 (during the substitution P2); R1 A, X; R2 Y_a, Y_b, S_d; R3 A W_a,
// A W_b, X^T W_a, X^T W_b; R4 the four F blocks; R5 P V_a, P V_b.
#include "internal.h"
#include "dev_common.cuh"
#include "tc_common.cuh"
#include "ut_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

namespace pathattn {

bool make_map_head_rows128(CUtensorMap* m, const void* base, uint64_t L, uint64_t heads);  // fwd128_tc.cu

namespace {
using namespace tc;

constexpr int B = 64;
constexpr int D = kHeadDimWide;
constexpr uint32_t TILE = 64 * 128;  // one 64x64 bf16 tile
constexpr int NSLOT = 13;
constexpr uint32_t TMEM_COLS = 256;
enum { S_WA = 0, S_KA, S_WB, S_KB, S_QA, S_QB, S_L, S_L2, S_N2, S_U, S_M1, S_P, S_VB };
constexpr int S_A = S_L, S_X = S_L2, S_YA = S_N2, S_VA = S_U, S_YB = S_M1;

struct Ut128Params {
  int L, Lp, nc, BH;
  float scl;  // scale * log2(e)
  const float* beta;
  const float* logf;
  __nv_bfloat16* ql;  // [BH][Lp][128]
  __nv_bfloat16* kr;  // [BH][Lp][128]
  __nv_bfloat16* f;   // [BH][nc][128][128]
  float* dm;          // [BH][Lp]
  float* dl;
  float* dacc;        // [BH][Lp][128]
  float* fa;
  float* fr;
  float* ft;
  int* err;
};

struct __align__(1024) Ut128Smem {
  uint8_t t[NSLOT][TILE];
  float beta[B], pre[B];
  uint64_t bar_in, bar_v, bar_mma;
  uint32_t tmem_base;
};


__global__ void __launch_bounds__(128, 2) ut_prep128_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                            const __grid_constant__ CUtensorMap tm_k,
                                                            const __grid_constant__ CUtensorMap tm_v,
                                                            const __grid_constant__ CUtensorMap tm_w,
                                                            const Ut128Params p) {
  extern __shared__ uint8_t smem_raw[];
  Ut128Smem& s = *reinterpret_cast<Ut128Smem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool lead = tid == 0;
  // this thread's half row of the M=64 accumulators: row i, columns 32h .. 32h+31
  const int i = 16 * warp + (lane & 15), h = lane >> 4;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  auto ta = [&](int slot) { return smem_u32(s.t[slot]); };
  float* sg = reinterpret_cast<float*>(s.t[S_L]);  // fp32 L = strictLower(D G) over slots 6 and 7

  if (lead) {
    mbar_init(&s.bar_in, 1);
    mbar_init(&s.bar_v, 1);
    mbar_init(&s.bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&s.tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  uint32_t mph = 0;  // phase of bar_mma
  auto issue = [&](auto fn) {  // lead issues one round's MMAs and commits them
    if (lead) {
      tc_fence_after();
      fn();
      mma_commit(&s.bar_mma);
    }
  };
  auto wait_mma = [&](int code) {
    mbar_wait_lean(&s.bar_mma, mph, p.err, code);
    mph ^= 1;
    tc_fence_after();
  };
  auto publish = [&]() {  // tiles written by the threads -> visible to the next MMAs; TMEM reads done
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
  };

  // Persistent: the CTA takes chunks blockIdx.x, blockIdx.x + gridDim.x, ... (chunk c of head bh at
  // index bh * nc + c), keeping its barriers (phases carried over) and its TMEM.
  const int nchunks = p.BH * p.nc;
  uint32_t it = 0;  // chunks done by this CTA: the phase of bar_in and bar_v
  for (int idx = blockIdx.x; idx < nchunks; idx += gridDim.x, ++it) {
    const int c = idx % p.nc, bh = idx / p.nc;
    const int row0 = c * B;
    const size_t in_row = (size_t)bh * p.L;
    const size_t ws_row = (size_t)bh * p.Lp + row0;
    if (lead) {
      fence_proxy_async_smem();  // the previous chunk's reads of the slots come before the copies
      mbar_arrive_expect_tx(&s.bar_in, 7 * TILE);
      tma_load_3d(s.t[S_WA], &tm_w, 0, row0, bh, &s.bar_in);
      tma_load_3d(s.t[S_WB], &tm_w, 64, row0, bh, &s.bar_in);
      tma_load_3d(s.t[S_KA], &tm_k, 0, row0, bh, &s.bar_in);
      tma_load_3d(s.t[S_KB], &tm_k, 64, row0, bh, &s.bar_in);
      tma_load_3d(s.t[S_QA], &tm_q, 0, row0, bh, &s.bar_in);
      tma_load_3d(s.t[S_QB], &tm_q, 64, row0, bh, &s.bar_in);
      tma_load_3d(s.t[S_VB], &tm_v, 64, row0, bh, &s.bar_in);
    }
    if (tid < B) {
      const int gi = row0 + tid;
      s.beta[tid] = gi < p.L ? clamp_beta(p.beta[in_row + gi]) : 0.f;
    }
    if (warp == 3) {  // chunk-local inclusive prefix of log f
      const int ga = row0 + lane, gb = row0 + 32 + lane;
      float a = (p.logf && ga < p.L) ? p.logf[in_row + ga] : 0.f;
      float b2 = (p.logf && gb < p.L) ? p.logf[in_row + gb] : 0.f;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const float ta2 = __shfl_up_sync(0xffffffffu, a, o), tb2 = __shfl_up_sync(0xffffffffu, b2, o);
        if (lane >= o) { a += ta2; b2 += tb2; }
      }
      const float tot_a = __shfl_sync(0xffffffffu, a, 31);
      s.pre[lane] = a;
      s.pre[32 + lane] = b2 + tot_a;
    }
    mbar_wait_lean(&s.bar_in, it & 1, p.err, 31);
    __syncthreads();

    // ---- P1: [G | N2] = W_a [W_a; K_a]^T + W_b [W_b; K_b]^T (two N=128 MMAs over adjacent slots) ----
    issue([&] {
      const uint32_t idesc = idesc_bf16(64, 128, 0, 0);
#pragma unroll
      for (int x = 0; x < 2; ++x) {
        const uint32_t base = ta(x ? S_WB : S_WA);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint64_t d = sdesc_sw128(base + 32u * kk, 1024, 16);
          mma_ss(tb + 0, d, d, idesc, (x > 0 || kk > 0) ? 1u : 0u);
        }
      }
    });
    wait_mma(32);
    {
      float x[32];
      ld_half(tb, lane_off, 0, x);  // L = strictLower(diag(beta) G), fp32
      const float bi = s.beta[i];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int j = 32 * h + 4 * q;
        *reinterpret_cast<float4*>(sg + f32_idx(i, j)) =
            make_float4(j < i ? bi * x[4 * q] : 0.f, j + 1 < i ? bi * x[4 * q + 1] : 0.f,
                        j + 2 < i ? bi * x[4 * q + 2] : 0.f, j + 3 < i ? bi * x[4 * q + 3] : 0.f);
      }
      ld_half(tb, lane_off, 64, x);  // N2 = strictLower(W K^T)
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = 32 * h + j < i ? x[j] : 0.f;
      put_half(s.t[S_N2], i, h, x);
    }
    // every thread has read P1's accumulators: M1 = Q W^T goes to the tensor core while the
    // threads substitute
    tc_fence_before();
    __syncthreads();
    issue([&] {
      mma64(tb + 0, ta(S_QA), 0, ta(S_WA), 0, 0);
      mma64(tb + 0, ta(S_QB), 0, ta(S_WB), 0, 1);
    });

    // ---- P2: U = (I + strictLower(D G))^{-1} D ----
    ut_solve_blocked_t<false>(sg, s.beta, s.t[S_U], nullptr, tid);  // U^T tile
    wait_mma(33);
    {
      float x[32];
      ld_half(tb, lane_off, 0, x);  // M1 = lower(Q W^T)
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = 32 * h + j <= i ? x[j] : 0.f;
      put_half(s.t[S_M1], i, h, x);
    }
    publish();

    // ---- R1: A = M1 U, X = U N2 ----
    issue([&] {
      mma64(tb + 0, ta(S_M1), 0, ta(S_U), 0, 0);   // B = U read from U^T (K-major)
      mma64(tb + 64, ta(S_U), 1, ta(S_N2), 1, 0);  // A = U read from U^T (MN-major)
    });
    wait_mma(34);
    {
      float x[32];
      ld_half(tb, lane_off, 0, x);
      put_half(s.t[S_A], i, h, x);
      ld_half(tb, lane_off, 64, x);
      put_half(s.t[S_X], i, h, x);
    }
    publish();

    // ---- R2: Y_x = U^T W_x, S_d = Q K^T - M1 X; then V_a into U's slot ----
    issue([&] {
      mma64(tb + 0, ta(S_U), 0, ta(S_WA), 1, 0);  // A = U^T (K-major)
      mma64(tb + 64, ta(S_U), 0, ta(S_WB), 1, 0);
      mma64(tb + 128, ta(S_QA), 0, ta(S_KA), 0, 0);
      mma64(tb + 128, ta(S_QB), 0, ta(S_KB), 0, 1);
      mma64(tb + 128, ta(S_M1), 0, ta(S_X), 1, 1, /*neg_a=*/1);
    });
    wait_mma(35);
    if (lead) {  // U has been read by R2's products: its slot takes V_a
      mbar_arrive_expect_tx(&s.bar_v, TILE);
      tma_load_3d(s.t[S_VA], &tm_v, 0, row0, bh, &s.bar_v);
    }
    {
      float x[32];
      ld_half(tb, lane_off, 0, x);
      put_half(s.t[S_YA], i, h, x);  // N2's slot (last read by R1)
      ld_half(tb, lane_off, 64, x);
      put_half(s.t[S_YB], i, h, x);  // M1's slot (last read by R2)
      ld_half(tb, lane_off, 128, x);  // S_d: the diagonal chunk's softmax partial state
      const float pi = s.pre[i];
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const int jj = 32 * h + j;
        const float sv = (jj <= i && row0 + jj < p.L) ? fmaf(x[j], p.scl, (pi - s.pre[jj]) * kLog2e) : -INFINITY;
        x[j] = sv;
        mx = fmaxf(mx, sv);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      float l = 0.f;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float pj = x[j] == -INFINITY ? 0.f : fast_exp2(x[j] - mx);
        x[j] = pj;
        l += pj;
      }
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      put_half(s.t[S_P], i, h, x);
      if (h == 0) {
        p.dm[ws_row + i] = mx;
        p.dl[ws_row + i] = l;
      }
    }
    if (p.logf && tid < B) {
      const float tot = s.pre[B - 1];
      p.fa[ws_row + tid] = s.pre[tid];
      p.fr[ws_row + tid] = tot - s.pre[tid];
      if (tid == 0) p.ft[(size_t)bh * p.nc + c] = tot;
    }
    publish();
    // ---- R3: A W_x, X^T W_x -> Q<- = Q - A W, K-> = K - X^T W ----
    issue([&] {
      mma64(tb + 0, ta(S_A), 0, ta(S_WA), 1, 0);
      mma64(tb + 64, ta(S_A), 0, ta(S_WB), 1, 0);
      mma64(tb + 128, ta(S_X), 1, ta(S_WA), 1, 0);
      mma64(tb + 192, ta(S_X), 1, ta(S_WB), 1, 0);
    });
    wait_mma(36);
    {
      float x[32], src[32];
      const size_t orow = ws_row + i;
#pragma unroll
      for (int xh = 0; xh < 2; ++xh) {
        ld_half(tb, lane_off, 64 * xh, x);
        get_half(s.t[xh ? S_QB : S_QA], i, h, src);
#pragma unroll
        for (int j = 0; j < 32; ++j) src[j] -= x[j];
        store_bf16_half(p.ql + orow * D + 64 * xh + 32 * h, src);
        ld_half(tb, lane_off, 128 + 64 * xh, x);
        get_half(s.t[xh ? S_KB : S_KA], i, h, src);
#pragma unroll
        for (int j = 0; j < 32; ++j) src[j] -= x[j];
        store_bf16_half(p.kr + orow * D + 64 * xh + 32 * h, src);
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- R4: F_xy = delta_xy I - W_x^T Y_y, F row-major [128][128] ----
    issue([&] {
      mma64(tb + 0, ta(S_WA), 1, ta(S_YA), 1, 0);
      mma64(tb + 64, ta(S_WA), 1, ta(S_YB), 1, 0);
      mma64(tb + 128, ta(S_WB), 1, ta(S_YA), 1, 0);
      mma64(tb + 192, ta(S_WB), 1, ta(S_YB), 1, 0);
    });
    wait_mma(37);
    {
      float x[32];
      __nv_bfloat16* fc = p.f + ((size_t)bh * p.nc + c) * D * D;
#pragma unroll
      for (int blk = 0; blk < 4; ++blk) {
        const int xr = blk >> 1, yc = blk & 1;  // row half (of W^T), column half (of Y)
        ld_half(tb, lane_off, 64 * blk, x);
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = ((xr == yc && 32 * h + j == i) ? 1.f : 0.f) - x[j];
        store_bf16_half(fc + (size_t)(64 * xr + i) * D + 64 * yc + 32 * h, x);
      }
    }
    tc_fence_before();
    __syncthreads();

    // ---- R5: P V_x -> acc ----
    mbar_wait_lean(&s.bar_v, it & 1, p.err, 38);
    issue([&] {
      mma64(tb + 0, ta(S_P), 0, ta(S_VA), 1, 0);
      mma64(tb + 64, ta(S_P), 0, ta(S_VB), 1, 0);
    });
    wait_mma(39);
    {
      float x[32];
#pragma unroll
      for (int xh = 0; xh < 2; ++xh) {
        ld_half(tb, lane_off, 64 * xh, x);
        float4* dst = reinterpret_cast<float4*>(p.dacc + (ws_row + i) * D + 64 * xh + 32 * h);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
      }
    }
    tc_fence_before();
    __syncthreads();  // TMEM and the slots are read out before the next chunk reuses them
    tc_fence_after();
  }
  if (warp == 1) tmem_dealloc(tb, TMEM_COLS);
}

}  // namespace

cudaError_t launch_ut_prep128(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                              const float* beta, const float* logf, char* ws, const FwdWs& lay, cudaStream_t st) {
  if (g.B != 64 || g.D != D || g.Lp != g.nc * B) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv, mw;
  if (!make_map_head_rows128(&mq, q, g.L, g.BH) || !make_map_head_rows128(&mk, k, g.L, g.BH) ||
      !make_map_head_rows128(&mv, v, g.L, g.BH) || !make_map_head_rows128(&mw, w, g.L, g.BH))
    return cudaErrorInvalidValue;
  Ut128Params p;
  p.L = g.L;
  p.Lp = g.Lp;
  p.nc = g.nc;
  p.BH = g.BH;
  p.scl = g.scale * kLog2e;
  p.beta = beta;
  p.logf = logf;
  p.ql = (__nv_bfloat16*)(ws + lay.ql);
  p.kr = (__nv_bfloat16*)(ws + lay.kr);
  p.f = (__nv_bfloat16*)(ws + lay.f);
  p.dm = (float*)(ws + lay.dm);
  p.dl = (float*)(ws + lay.dl);
  p.dacc = (float*)(ws + lay.dacc);
  p.fa = (float*)(ws + lay.fa);
  p.fr = (float*)(ws + lay.fr);
  p.ft = (float*)(ws + lay.ft);
  p.err = (int*)(ws + lay.err);
  const size_t smem = sizeof(Ut128Smem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(ut_prep128_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // one wave of persistent CTAs: as many as the SMs hold at once, by shared memory (with the
  // per-block reservation) and by TMEM columns (two per SM)
  int dev = 0, nsm = 0, smem_sm = 0, reserved = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess) return e;
  const int per_sm = std::max(1, std::min(smem_sm / (int)(smem + reserved), (int)(512 / TMEM_COLS)));
  const long nchunks = (long)g.nc * g.BH;
  const long grid = std::min(nchunks, (long)nsm * per_sm);
  ut_prep128_kernel<<<(unsigned)grid, 128, smem, st>>>(mq, mk, mv, mw, p);
  return cudaGetLastError();
}

}  // namespace pathattn
