// Per-chunk UT preparation on tcgen05 (bf16 operands, fp32 accumulation in TMEM), chunk B = 64:
// one CTA of 128 threads per chunk.
//
// Method: PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.6 (UT representation) and §2.7
// (boundary-adjusted queries/keys, chunk transform):
//   G = strictLower(W W^T), M1 = lower(Q W^T), N2 = strictLower(W K^T)
//   U = (I + strictLower(D G))^{-1} D        (fp32, two-level block inversion)
//   A = M1 U,  X = U N2,  Y = U^T W
//   Q<- = Q - A W,  K-> = K - X^T W,  F = I - W^T Y,  S_d = Q K^T - M1 X (masked j <= i)
// and the diagonal chunk's softmax partial state (m, l, acc = P V).
// Every product is an M=64 MMA whose operands are 64x64 bf16 tiles in the 128-byte swizzled layout
// (TMA-loaded inputs or tiles written by the warps), K-major or MN-major as the product needs; the
// four products of the first phase share their B operands two by two, so they run as two N=128
// MMAs over the stacked [W; K] tile.  Accumulators are read with the 16x32bx2 TMEM shape: each
// thread of warp w holds 32 columns (half h = lane / 16) of row 16w + lane % 16, so all 128
// threads work in every epilogue; the two halves of a row meet through one shuffle where a row
// reduction is needed.  Inputs come through 3-D tensor maps ([heads][L][64]) that read rows >= L
// as zero.
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

constexpr uint32_t kUtTile = 64 * 128;  // one 64x64 bf16 tile
constexpr uint32_t kUtSlotBytes = 11 * kUtTile;

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
};

// Shared memory of one chunk's preparation: eleven 1024-byte aligned tiles in this order (w and k
// adjacent: the stacked B operand of the first phase; a and x adjacent: the fp32 L of the
// substitution), beta and the forget-gate prefix (16-byte aligned), and two mbarriers.
struct UtSlots {
  uint8_t *w, *k, *q, *v, *m1, *n2, *u, *a, *x, *y, *p;
  float* beta;
  float* pre;
  uint64_t* bar_in;
  uint64_t* bar_mma;
};
__device__ __forceinline__ UtSlots ut_slots(uint8_t* base, float* beta, float* pre, uint64_t* bar_in,
                                            uint64_t* bar_mma) {
  UtSlots s;
  uint8_t** t[11] = {&s.w, &s.k, &s.q, &s.v, &s.m1, &s.n2, &s.u, &s.a, &s.x, &s.y, &s.p};
#pragma unroll
  for (int j = 0; j < 11; ++j) *t[j] = base + j * kUtTile;
  s.beta = beta;
  s.pre = pre;
  s.bar_in = bar_in;
  s.bar_mma = bar_mma;
  return s;
}

// Prepares chunk c of head bh.  Run by the CTA's 128 threads together; thread 0 issues the TMA
// loads and the MMAs.  tb: 256 TMEM columns of the CTA; in_par / mph: phases of
// bar_in (one completion per call) and bar_mma (advanced here).  zimg (optional): a swizzled
// 64-row bf16 tile image that also receives Q<- of the chunk.  The mbarriers are initialised by
// the caller; on return every TMEM access and every MMA of the chunk has completed, and the
// slots may be reused.
template <bool F32>
__device__ __forceinline__ void ut_prep_chunk(const UtSlots& s, uint32_t tb, const CUtensorMap* tm_q,
                                              const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                                              const CUtensorMap* tm_w, const UtParams& p, int bh, int c,
                                              uint32_t in_par, uint32_t& mph, uint8_t* zimg) {
  constexpr int B = 64;
  constexpr int D = kHeadDim;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int row0 = c * B;
  const size_t in_row = (size_t)bh * p.L;
  const size_t ws_row = (size_t)bh * p.Lp + row0;
  const bool lead = tid == 0;
  // this thread's half row of the M=64 accumulators: row i, columns 32h .. 32h+31
  const int i = 16 * warp + (lane & 15), h = lane >> 4;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  float* sg = reinterpret_cast<float*>(s.a);  // fp32 L = strictLower(D G) over the a and x slots
  const uint32_t aw = smem_u32(s.w), aq = smem_u32(s.q), ak = smem_u32(s.k), av = smem_u32(s.v);
  const uint32_t am1 = smem_u32(s.m1), an2 = smem_u32(s.n2), au = smem_u32(s.u);
  const uint32_t aa = smem_u32(s.a), ax = smem_u32(s.x), ay = smem_u32(s.y), ap = smem_u32(s.p);
  auto run = [&](auto issue, int code) {  // lead issues one phase's MMAs; every thread waits
    if (lead) {
      tc_fence_after();
      issue();
      mma_commit(s.bar_mma);
    }
    mbar_wait(s.bar_mma, mph, p.err, code);
    mph ^= 1;
    tc_fence_after();
  };
  auto publish = [&]() {  // tiles written by the threads -> visible to the next MMAs
    fence_proxy_async_smem();
    tc_fence_before();
    ut_sync();
  };

  if (lead) {
    mbar_arrive_expect_tx(s.bar_in, (p.with_diag ? 4 : 3) * kUtTile);
    tma_load_3d(s.w, tm_w, 0, row0, bh, s.bar_in);
    tma_load_3d(s.q, tm_q, 0, row0, bh, s.bar_in);
    tma_load_3d(s.k, tm_k, 0, row0, bh, s.bar_in);
    if (p.with_diag) tma_load_3d(s.v, tm_v, 0, row0, bh, s.bar_in);
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
      const float ta = __shfl_up_sync(0xffffffffu, a, o), tb2 = __shfl_up_sync(0xffffffffu, b2, o);
      if (lane >= o) { a += ta; b2 += tb2; }
    }
    const float tot_a = __shfl_sync(0xffffffffu, a, 31);
    s.pre[lane] = a;
    s.pre[32 + lane] = b2 + tot_a;
  }
  mbar_wait(s.bar_in, in_par, p.err, 31);
  ut_sync();

  // ---- P1: [G | N2] = W [W; K]^T, [M1 | Q K^T] = Q [W; K]^T ----
  run([&] {
    const uint32_t idesc = idesc_bf16(64, 128, 0, 0);
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      const uint64_t bd = sdesc_sw128(aw + 32u * kk, 1024, 16);  // 128 rows: the w tile, then the k tile
      mma_ss(tb + 0, sdesc_sw128(aw + 32u * kk, 1024, 16), bd, idesc, kk > 0 ? 1u : 0u);
      mma_ss(tb + 128, sdesc_sw128(aq + 32u * kk, 1024, 16), bd, idesc, kk > 0 ? 1u : 0u);
    }
  }, 32);
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
    ld_half(tb, lane_off, 128, x);  // M1 = lower(Q W^T)
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = 32 * h + j <= i ? x[j] : 0.f;
    put_half(s.m1, i, h, x);
    ld_half(tb, lane_off, 64, x);  // N2 = strictLower(W K^T)
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = 32 * h + j < i ? x[j] : 0.f;
    put_half(s.n2, i, h, x);
  }
  ut_sync();

  // ---- P2: U = (I + strictLower(D G))^{-1} D (with an fp32 F: U = U_hi + U_lo, U_lo in P's
  //      slot, unused without the diagonal state) ----
  ut_solve_blocked<F32>(sg, s.beta, s.u, s.p, tid);
  publish();

  // ---- P3: A = M1 U, X = U N2, Y = U^T W (+ U_lo^T W for an fp32 F) ----
  run([&] {
    mma64(tb + 0, am1, 0, au, 1, 0);
    mma64(tb + 64, au, 0, an2, 1, 0);
    mma64(tb + 128, au, 1, aw, 1, 0);
    if constexpr (F32) mma64(tb + 128, ap, 1, aw, 1, 1);
  }, 33);
  {
    float x[32];
    ld_half(tb, lane_off, 0, x);
    put_half(s.a, i, h, x);
    ld_half(tb, lane_off, 64, x);
    put_half(s.x, i, h, x);
    ld_half(tb, lane_off, 128, x);
    if constexpr (F32) {  // Y = Y_hi + Y_lo, both bf16 (Y_lo in V's slot, never loaded without the diagonal state)
      float lo[32];
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float hi = __bfloat162float(__float2bfloat16_rn(x[j]));
        lo[j] = x[j] - hi;
        x[j] = hi;
      }
      put_half(s.v, i, h, lo);
    }
    put_half(s.y, i, h, x);
  }
  publish();

  // ---- P4: A W, X^T W, S_d = QK^T - M1 X (accumulated onto QK^T), W^T Y ----
  run([&] {
    mma64(tb + 0, aa, 0, aw, 1, 0);
    mma64(tb + 64, ax, 1, aw, 1, 0);
    mma64(tb + 192, am1, 0, ax, 1, 1, /*neg_a=*/1);
    mma64(tb + 128, aw, 1, ay, 1, 0);
    if constexpr (F32) mma64(tb + 128, aw, 1, av, 1, 1);
  }, 34);
  {
    float x[32], src[32];
    const size_t orow = ws_row + i;
    ld_half(tb, lane_off, 0, x);  // Q<- = Q - A W
    get_half(s.q, i, h, src);
#pragma unroll
    for (int j = 0; j < 32; ++j) src[j] -= x[j];
    store_bf16_half(p.ql + orow * D + 32 * h, src);
    if (zimg) put_half(zimg, i, h, src);
    ld_half(tb, lane_off, 64, x);  // K-> = K - X^T W
    get_half(s.k, i, h, src);
#pragma unroll
    for (int j = 0; j < 32; ++j) src[j] -= x[j];
    store_bf16_half(p.kr + orow * D + 32 * h, src);
    ld_half(tb, lane_off, 128, x);  // F = I - W^T Y, row i
#pragma unroll
    for (int j = 0; j < 32; ++j) x[j] = (32 * h + j == i ? 1.f : 0.f) - x[j];
    if constexpr (F32) {
      // fp32 F at the same F pointer (the caller's layout gives it room for fp32)
      float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.f) + (((size_t)bh * p.nc + c) * D + i) * D + 32 * h);
#pragma unroll
      for (int q = 0; q < 8; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
    } else {
      store_bf16_half(p.f + (((size_t)bh * p.nc + c) * D + i) * D + 32 * h, x);
    }
    if (p.with_diag) {
      ld_half(tb, lane_off, 192, x);  // S_d: the diagonal chunk's softmax partial state
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
      put_half(s.p, i, h, x);
      if (h == 0) {
        p.dm[orow] = mx;
        p.dl[orow] = l;
      }
    }
  }
  if (p.logf && tid < B) {
    const float tot = s.pre[B - 1];
    p.fa[ws_row + tid] = s.pre[tid];
    p.fr[ws_row + tid] = tot - s.pre[tid];
    if (tid == 0) p.ft[(size_t)bh * p.nc + c] = tot;
  }
  if (p.with_diag) {
    publish();
    // ---- P5: acc = P V ----
    run([&] { mma64(tb + 0, ap, 0, av, 1, 0); }, 35);
    float x[32];
    ld_half(tb, lane_off, 0, x);
    float4* dst = reinterpret_cast<float4*>(p.dacc + (ws_row + i) * D + 32 * h);
#pragma unroll
    for (int q = 0; q < 8; ++q) dst[q] = make_float4(x[4 * q], x[4 * q + 1], x[4 * q + 2], x[4 * q + 3]);
  }
  // every thread's TMEM loads are complete (tcgen05.wait::ld in ld_half); the slots and the TMEM
  // columns may be reused after the caller's next barrier
  tc_fence_before();
  ut_sync();
  tc_fence_after();
}

struct __align__(1024) UtSmem {
  uint8_t tiles[kUtSlotBytes];  // the eleven preparation slots (ut_slots order)
  float beta[64], pre[64];
  uint64_t bar_in, bar_mma;
  uint32_t tmem_base;
};

template <bool F32>
__global__ void __launch_bounds__(128) ut_prep64_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                        const __grid_constant__ CUtensorMap tm_k,
                                                        const __grid_constant__ CUtensorMap tm_v,
                                                        const __grid_constant__ CUtensorMap tm_w,
                                                        const UtParams p) {
  extern __shared__ uint8_t smem_raw[];
  UtSmem& s = *reinterpret_cast<UtSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5;
  if (tid == 0) {
    mbar_init(&s.bar_in, 1);
    mbar_init(&s.bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&s.tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  const UtSlots sl = ut_slots(s.tiles, s.beta, s.pre, &s.bar_in, &s.bar_mma);
  uint32_t mph = 0;
  ut_prep_chunk<F32>(sl, tb, &tm_q, &tm_k, &tm_v, &tm_w, p, (int)blockIdx.y, (int)blockIdx.x, 0, mph, nullptr);
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, 256);
  }
}

}  // namespace

cudaError_t launch_ut_prep64(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                             const float* beta, const float* logf, char* ws, const FwdWs& lay, bool with_diag,
                             cudaStream_t st, bool f32_f) {
  if (g.B != 64 || (f32_f && with_diag)) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv, mw;
  if (!make_map_head_rows64(&mq, q, g.L, g.BH) || !make_map_head_rows64(&mk, k, g.L, g.BH) ||
      !make_map_head_rows64(&mv, v, g.L, g.BH) || !make_map_head_rows64(&mw, w, g.L, g.BH))
    return cudaErrorInvalidValue;
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
  const size_t smem = sizeof(UtSmem) + 1024;
  auto kern = f32_f ? ut_prep64_kernel<true> : ut_prep64_kernel<false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<dim3(g.nc, g.BH), 128, smem, st>>>(mq, mk, mv, mw, p);
  return cudaGetLastError();
}

}  // namespace pathattn
