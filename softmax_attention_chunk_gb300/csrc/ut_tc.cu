// Per-chunk UT preparation on tcgen05 (bf16 operands, fp32 accumulation in TMEM), chunk B = 64:
// persistent CTAs of 128 threads, three per SM, each taking chunk after chunk.
//
// Method: PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.6 (UT representation) and §2.7
// (boundary-adjusted queries/keys, chunk transform):
//   G = strictLower(W W^T), M1 = lower(Q W^T), N2 = strictLower(W K^T)
//   U = (I + strictLower(D G))^{-1} D        (fp32, two-level block inversion)
//   A = M1 U,  X = U N2,  Y = U^T W
//   Q<- = Q - A W,  K-> = K - X^T W,  F = I - W^T Y,  S_d = Q K^T - M1 X (masked j <= i)
// and the diagonal chunk's softmax partial state (m, l, acc = P V).
//
// Every product is an M=64 MMA whose operands are 64x64 bf16 tiles in the 128-byte swizzled
// layout (TMA-loaded inputs or tiles written by the warps), K-major or MN-major as the product
// needs.  Accumulators are read with the 16x32bx2 TMEM shape: each thread of warp w holds 32
// columns (half h = lane / 16) of row 16w + lane % 16, so all 128 threads work in every epilogue;
// the two halves of a row meet through one shuffle where a row reduction is needed.  Inputs come
// through 3-D tensor maps ([heads][L][64]) that read rows >= L as zero.
//
// The kernel is latency bound (a chain of product rounds, each an MMA -> TMEM -> registers ->
// shared-memory tile round trip, and the substitution), so it is laid out for three CTAs per SM:
// 128 TMEM columns (two 64-column accumulators per round) and nine 8 KB tile slots, reused as
// their tenants die:
//   slot 0 W          P1 .. R4           slot 5 M1 (M1 epilogue .. R2), then Y (R2 .. R4)
//   slot 1 K          P1 .. R3 epilogue  slot 6 N2 (P1 .. R1), then P (R2 .. R4) or Y_lo (split F)
//   slot 2 Q          P1 .. R3 epilogue  slot 7 U^T (P2 .. R2), then V (loaded once R2 has read it)
//   slots 3-4 fp32 L (P1 .. P2), then A (slot 3) and X (slot 4) (R1 .. R3)
//   slot 8 U_lo^T (split F only)
// The split-F instances (the walks of the hand-off and of the context-parallel shards) write F as
// F_hi + F_lo, two bf16 tiles of about 16 significant bits together.  The keys-only instance (the
// hand-off) loads no Q, skips M1, A, X and Q<-, and forms K-> = K - N2^T Y (X^T W = N2^T U^T W)
// and F = I - W^T Y in one round, with Y_lo in Q's slot (N2 stays in its own until then).
// U is stored transposed (the block inversion writes each column it holds as a contiguous row), and
// the products read it with the matching operand major-ness.
// W and K are adjacent: the first round's two products share the stacked [W; K] tile as one N=128
// B operand.  Rounds: P1 [G | N2]; M1 (its MMA runs during the substitution P2); R1 A, X;
// R2 Y, S_d; R3 A W, X^T W; R4 W^T Y, P V.
#include "internal.h"
#include "dev_common.cuh"
#include "tc_common.cuh"
#include "ut_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>

namespace pathattn {

bool make_map_head_rows64(CUtensorMap* m, const void* base, uint64_t L, uint64_t heads);  // fwd_tc.cu
bool make_map_head_rows64_pitch(CUtensorMap* m, const void* base, uint64_t L, uint64_t heads, uint64_t head_rows);

namespace {
using namespace tc;

constexpr int B = 64;
constexpr int D = kHeadDim;
constexpr uint32_t TILE = 64 * 128;  // one 64x64 bf16 tile
constexpr int NSLOT = 9;
constexpr uint32_t TMEM_COLS = 128;
enum { S_W = 0, S_K, S_Q, S_L, S_X, S_M1, S_N2, S_U, S_ULO };
constexpr int S_A = S_L, S_Y = S_M1, S_P = S_N2, S_YLO = S_N2, S_V = S_U;

struct UtParams {
  int L, Lp, nc, BH;
  float scl;  // scale * log2(e)
  const float* beta;
  const float* logf;
  __nv_bfloat16* ql;
  __nv_bfloat16* kr;
  __nv_bfloat16* f;
  float* dm;
  float* dl;
  float* dacc;
  float* fa;
  float* fr;
  float* ft;
  int with_diag;
  int* err;
  uint32_t stall_ns;  // test hook: nonzero makes every CTA give up a wait (see the kernel's start)
};

struct __align__(1024) UtSmem {
  uint8_t t[NSLOT][TILE];
  float beta[B], pre[B];
  uint64_t bar_in, bar_v, bar_mma;
  uint32_t tmem_base;
};

// F32: F split into bf16 high and low tiles.  KO (keys only, with F32; the hand-off): no query
// side and no diagonal state: K-> = K - N2^T Y and F = I - W^T Y both come from Y = U^T W in one
// round; the chunk's values are copied to the value cache (tm_vc) on the way, through the fp32 L
// slots once the substitution is done with them (TMA load, then TMA store: rows >= L are clipped).
template <bool F32, bool KO>
__global__ void __launch_bounds__(128, 3) ut_prep64_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                           const __grid_constant__ CUtensorMap tm_k,
                                                           const __grid_constant__ CUtensorMap tm_v,
                                                           const __grid_constant__ CUtensorMap tm_w,
                                                           const __grid_constant__ CUtensorMap tm_vc,
                                                           const UtParams p) {
  extern __shared__ uint8_t smem_raw[];
  UtSmem& s = *reinterpret_cast<UtSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool lead = tid == 0;
  const bool diag = p.with_diag != 0;
  // this thread's half row of the M=64 accumulators: row i, columns 32h .. 32h+31
  const int i = 16 * warp + (lane & 15), h = lane >> 4;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  auto ta = [&](int slot) { return smem_u32(s.t[slot]); };
  float* sg = reinterpret_cast<float*>(s.t[S_L]);  // fp32 L = strictLower(D G) over slots 3 and 4

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
  if (p.stall_ns) {
    // Test hook of the failure path: a wait on a barrier that nothing arrives at runs out after
    // stall_ns, records code 99 and ends the CTA before any copy or MMA has been issued, with its
    // TMEM freed, as a pipeline wait that gives up does.
    if (lead) mbar_wait_ns(&s.bar_v, 0, p.err, 99, p.stall_ns);
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
      tc_fence_after();
      tmem_dealloc(tb, TMEM_COLS);
    }
    return;
  }
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
      mbar_arrive_expect_tx(&s.bar_in, (KO ? 2 : 3) * TILE);
      tma_load_3d(s.t[S_W], &tm_w, 0, row0, bh, &s.bar_in);
      if (!KO) tma_load_3d(s.t[S_Q], &tm_q, 0, row0, bh, &s.bar_in);
      tma_load_3d(s.t[S_K], &tm_k, 0, row0, bh, &s.bar_in);
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

    // ---- P1: [G | N2] = W [W; K]^T (one N=128 MMA: the w and k slots are adjacent) ----
    issue([&] {
      const uint32_t idesc = idesc_bf16(64, 128, 0, 0);
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint64_t d = sdesc_sw128(ta(S_W) + 32u * kk, 1024, 16);
        mma_ss(tb + 0, d, d, idesc, kk > 0 ? 1u : 0u);
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
    if constexpr (!KO) issue([&] { mma64(tb + 0, ta(S_Q), 0, ta(S_W), 0, 0); });

    // ---- P2: U = (I + strictLower(D G))^{-1} D (split F: U = U_hi + U_lo) ----
    ut_solve_blocked_t<F32>(sg, s.beta, s.t[S_U], s.t[S_ULO], tid);  // U^T (and U_lo^T) tiles
    if constexpr (!KO) {
      wait_mma(33);
      float x[32];
      ld_half(tb, lane_off, 0, x);  // M1 = lower(Q W^T)
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = 32 * h + j <= i ? x[j] : 0.f;
      put_half(s.t[S_M1], i, h, x);
    }
    publish();
    if (KO && lead) {  // the values through slot 3 (free once the substitution has read L)
      mbar_arrive_expect_tx(&s.bar_v, TILE);
      tma_load_3d(s.t[S_A], &tm_v, 0, row0, bh, &s.bar_v);
    }

    // ---- R1: A = M1 U, X = U N2 ----
    if constexpr (!KO) {
      issue([&] {
        mma64(tb + 0, ta(S_M1), 0, ta(S_U), 0, 0);   // B = U read from U^T (K-major)
        mma64(tb + 64, ta(S_U), 1, ta(S_N2), 1, 0);  // A = U read from U^T (MN-major)
      });
      wait_mma(34);
      float x[32];
      ld_half(tb, lane_off, 0, x);
      put_half(s.t[S_A], i, h, x);
      ld_half(tb, lane_off, 64, x);
      put_half(s.t[S_X], i, h, x);
      publish();
    }

    // ---- R2: Y = U^T W (+ U_lo^T W for an fp32 F), S_d = Q K^T - M1 X; then V into U's slot ----
    issue([&] {
      mma64(tb + 0, ta(S_U), 0, ta(S_W), 1, 0);  // A = U^T (K-major)
      if constexpr (F32) mma64(tb + 0, ta(S_ULO), 0, ta(S_W), 1, 1);
      if (diag) {
        mma64(tb + 64, ta(S_Q), 0, ta(S_K), 0, 0);
        mma64(tb + 64, ta(S_M1), 0, ta(S_X), 1, 1, /*neg_a=*/1);
      }
    });
    wait_mma(35);
    if (lead && diag) {  // U has been read by R2's products: its slot takes V
      mbar_arrive_expect_tx(&s.bar_v, TILE);
      tma_load_3d(s.t[S_V], &tm_v, 0, row0, bh, &s.bar_v);
    }
    {
      float x[32];
      ld_half(tb, lane_off, 0, x);
      if constexpr (F32) {  // Y = Y_hi + Y_lo, both bf16
        float lo[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float hi = __bfloat162float(__float2bfloat16_rn(x[j]));
          lo[j] = x[j] - hi;
          x[j] = hi;
        }
        put_half(s.t[KO ? S_Q : S_YLO], i, h, lo);  // keys only: N2 stays for K->
      }
      put_half(s.t[S_Y], i, h, x);
      if (diag) {
        ld_half(tb, lane_off, 64, x);  // S_d: the diagonal chunk's softmax partial state
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
    }
    if (p.logf && tid < B) {
      const float tot = s.pre[B - 1];
      p.fa[ws_row + tid] = s.pre[tid];
      p.fr[ws_row + tid] = tot - s.pre[tid];
      if (tid == 0) p.ft[(size_t)bh * p.nc + c] = tot;
    }
    publish();

    // F (row i, half h) as F_hi + F_lo, two bf16 tiles in the 128-byte swizzled layout, 16 KB per
    // chunk at the F pointer (the caller's layout gives it room), for the chunk walks to load as
    // they are
    auto store_split_f = [&](float (&fv)[32]) {
      float lo[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float v = fv[j];
        fv[j] = __bfloat162float(__float2bfloat16_rn(v));
        lo[j] = v - fv[j];
      }
      uint8_t* ft = reinterpret_cast<uint8_t*>(p.f + ((size_t)bh * p.nc + c) * 2 * D * D);
      put_half(ft, i, h, fv);
      put_half(ft + TILE, i, h, lo);
    };
    if constexpr (KO) {
      // ---- R3': W^T Y (+ W^T Y_lo), N2^T Y (+ N2^T Y_lo) -> F = I - W^T Y, K-> = K - N2^T Y
      // (X^T W = N2^T U^T W) ----
      issue([&] {
        mma64(tb + 0, ta(S_W), 1, ta(S_Y), 1, 0);
        mma64(tb + 0, ta(S_W), 1, ta(S_Q), 1, 1);
        mma64(tb + 64, ta(S_N2), 1, ta(S_Y), 1, 0);
        mma64(tb + 64, ta(S_N2), 1, ta(S_Q), 1, 1);
      });
      wait_mma(36);
      if (lead && mbar_wait_lean(&s.bar_v, it & 1, p.err, 37)) {
        tma_store_3d(&tm_vc, s.t[S_A], 0, row0, bh);
        bulk_commit();
      }
      float x[32], src[32];
      ld_half(tb, lane_off, 64, x);
      get_half(s.t[S_K], i, h, src);
#pragma unroll
      for (int j = 0; j < 32; ++j) src[j] -= x[j];
      store_bf16_half(p.kr + (ws_row + i) * D + 32 * h, src);
      ld_half(tb, lane_off, 0, x);
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = (32 * h + j == i ? 1.f : 0.f) - x[j];  // F = I - W^T Y, row i
      store_split_f(x);
    } else {
      // ---- R3: A W, X^T W -> Q<- = Q - A W, K-> = K - X^T W ----
      issue([&] {
        mma64(tb + 0, ta(S_A), 0, ta(S_W), 1, 0);
        mma64(tb + 64, ta(S_X), 1, ta(S_W), 1, 0);
      });
      wait_mma(36);
      {
        float x[32], src[32];
        const size_t orow = ws_row + i;
        ld_half(tb, lane_off, 0, x);
        get_half(s.t[S_Q], i, h, src);
#pragma unroll
        for (int j = 0; j < 32; ++j) src[j] -= x[j];
        store_bf16_half(p.ql + orow * D + 32 * h, src);
        ld_half(tb, lane_off, 64, x);
        get_half(s.t[S_K], i, h, src);
#pragma unroll
        for (int j = 0; j < 32; ++j) src[j] -= x[j];
        store_bf16_half(p.kr + orow * D + 32 * h, src);
      }
      tc_fence_before();
      __syncthreads();

      // ---- R4: W^T Y (+ W^T Y_lo) -> F = I - W^T Y; P V -> acc ----
      if (diag) mbar_wait_lean(&s.bar_v, it & 1, p.err, 37);
      issue([&] {
        mma64(tb + 0, ta(S_W), 1, ta(S_Y), 1, 0);
        if constexpr (F32) mma64(tb + 0, ta(S_W), 1, ta(S_YLO), 1, 1);
        if (diag) mma64(tb + 64, ta(S_P), 0, ta(S_V), 1, 0);
      });
      wait_mma(38);
      {
        float x[32];
        ld_half(tb, lane_off, 0, x);  // F = I - W^T Y, row i
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = (32 * h + j == i ? 1.f : 0.f) - x[j];
        if constexpr (F32) {
          store_split_f(x);
        } else {
          store_bf16_half(p.f + (((size_t)bh * p.nc + c) * D + i) * D + 32 * h, x);
        }
        if (diag) {
          ld_half(tb, lane_off, 64, x);
          float4* dst = reinterpret_cast<float4*>(p.dacc + (ws_row + i) * D + 32 * h);
#pragma unroll
          for (int q = 0; q < 8; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
        }
      }
    }
    if (KO && lead) bulk_wait_read0();  // the value store has read slot 3
    tc_fence_before();
    __syncthreads();  // TMEM and the slots are read out before the next chunk reuses them
    tc_fence_after();
  }
  if (KO && lead) bulk_wait0();
  if (warp == 1) tmem_dealloc(tb, TMEM_COLS);
}

}  // namespace

cudaError_t launch_ut_prep64(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                             const float* beta, const float* logf, char* ws, const FwdWs& lay, bool with_diag,
                             cudaStream_t st, bool f32_f, uint32_t stall_ns, bool with_q, void* v_cache,
                             int cap) {
  if (g.B != 64 || (f32_f && with_diag) || (!with_q && (!f32_f || !v_cache || cap < g.L))) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv, mw, mvc;
  if (!make_map_head_rows64(&mq, q, g.L, g.BH) || !make_map_head_rows64(&mk, k, g.L, g.BH) ||
      !make_map_head_rows64(&mv, v, g.L, g.BH) || !make_map_head_rows64(&mw, w, g.L, g.BH))
    return cudaErrorInvalidValue;
  if (with_q) mvc = mv;  // unused
  else if (!make_map_head_rows64_pitch(&mvc, v_cache, g.L, g.BH, cap)) return cudaErrorInvalidValue;
  UtParams p;
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
  p.with_diag = with_diag ? 1 : 0;
  p.err = (int*)(ws + lay.err);
  p.stall_ns = stall_ns;
  const size_t smem = sizeof(UtSmem) + 1024;
  auto kern = !with_q ? ut_prep64_kernel<true, true>
                      : (f32_f ? ut_prep64_kernel<true, false> : ut_prep64_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  // one wave of persistent CTAs: as many as the SMs hold at once, by shared memory (with the
  // per-block reservation) and by TMEM columns (three per SM on a GB300)
  int dev = 0, nsm = 0, smem_sm = 0, reserved = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess) return e;
  const int per_sm = std::max(1, std::min(smem_sm / (int)(smem + reserved), (int)(512 / TMEM_COLS)));
  const long nchunks = (long)g.nc * g.BH;
  const long grid = std::min(nchunks, (long)nsm * per_sm);
  kern<<<(unsigned)grid, 128, smem, st>>>(mq, mk, mv, mw, mvc, p);
  return cudaGetLastError();
}

}  // namespace pathattn
