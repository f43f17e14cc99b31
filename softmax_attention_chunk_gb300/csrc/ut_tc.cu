// Per-chunk UT preparation on tcgen05 (bf16 operands, fp32 accumulation in TMEM), chunk B = 64.
//
// Method: PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.6 (UT representation) and §2.7
// (boundary-adjusted queries/keys, chunk transform):
//   G = strictLower(W W^T), M1 = lower(Q W^T), N2 = strictLower(W K^T)
//   U = (I + strictLower(D G))^{-1} D        (forward substitution, fp32, two warps)
//   A = M1 U,  X = U N2,  Y = U^T W
//   Q<- = Q - A W,  K-> = K - X^T W,  F = I - W^T Y,  S_d = Q K^T - M1 X (masked j <= i)
// and the diagonal chunk's softmax partial state (m, l, acc = P V).
// Every product is one M=64 N=64 K=64 MMA whose operands are 64x64 bf16 tiles in the 128-byte
// swizzled layout (TMA-loaded inputs or tiles written by the warps), K-major or MN-major as the
// product needs; results are read back from TMEM (M=64 layout: row 16w+l in lane l of warp w).
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
constexpr uint32_t TILE = 64 * 128;  // one 64x64 bf16 tile
constexpr int GS = 65;               // fp32 G row stride

struct __align__(1024) UtSmem {
  uint8_t w[TILE], q[TILE], k[TILE], v[TILE];   // inputs (rows >= L zeroed)
  uint8_t m1[TILE], n2[TILE], u[TILE];          // lower(QW^T), strictLower(WK^T), U
  uint8_t a[TILE], x[TILE], y[TILE], p[TILE];   // M1 U, U N2, U^T W, P
  float g[B * GS];                              // G (fp32) for the solve
  float beta[B], pre[B];
  uint64_t bar_in, bar_mma;
  uint32_t tmem_base;
};

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

__global__ void __launch_bounds__(128) ut_prep64_kernel(const __grid_constant__ CUtensorMap tm_q,
                                                        const __grid_constant__ CUtensorMap tm_k,
                                                        const __grid_constant__ CUtensorMap tm_v,
                                                        const __grid_constant__ CUtensorMap tm_w,
                                                        const UtParams p) {
  extern __shared__ uint8_t smem_raw[];
  UtSmem& s = *reinterpret_cast<UtSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, bh = blockIdx.y;
  const int row0 = c * B;
  const size_t in_row = (size_t)bh * p.L;
  const size_t ws_row = (size_t)bh * p.Lp + row0;
  const bool lead = tid == 0;
  const int i = 16 * warp + lane;          // accumulator row held by this thread (lanes < 16)
  const bool has_row = lane < 16;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;

  if (lead) {
    mbar_init(&s.bar_in, 1);
    mbar_init(&s.bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&s.tmem_base, 256);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;
  const uint32_t aw = smem_u32(s.w), aq = smem_u32(s.q), ak = smem_u32(s.k), av = smem_u32(s.v);
  const uint32_t am1 = smem_u32(s.m1), an2 = smem_u32(s.n2), au = smem_u32(s.u);
  const uint32_t aa = smem_u32(s.a), ax = smem_u32(s.x), ay = smem_u32(s.y), ap = smem_u32(s.p);
  uint32_t mph = 0;  // phase of bar_mma

  if (lead) {
    const int y0 = (int)(in_row + row0);
    mbar_arrive_expect_tx(&s.bar_in, (p.with_diag ? 4 : 3) * TILE);
    tma_load_2d(s.w, &tm_w, 0, y0, &s.bar_in);
    tma_load_2d(s.q, &tm_q, 0, y0, &s.bar_in);
    tma_load_2d(s.k, &tm_k, 0, y0, &s.bar_in);
    if (p.with_diag) tma_load_2d(s.v, &tm_v, 0, y0, &s.bar_in);
  }
  if (tid < B) {
    const int gi = row0 + tid;
    const bool ok = gi < p.L;
    s.beta[tid] = ok ? clamp_beta(p.beta[in_row + gi]) : 0.f;
  }
  mbar_wait(&s.bar_in, 0, p.err, 31);
  // rows beyond L (ragged tail / padding chunk) are zero: H = I, q = k = v = 0
  if (row0 + B > p.L) {
    for (int r = tid; r < B; r += 128)
      if (row0 + r >= p.L) {
        uint4 z = make_uint4(0, 0, 0, 0);
        for (int qq = 0; qq < 8; ++qq) {
          reinterpret_cast<uint4*>(s.w + r * 128)[qq] = z;
          reinterpret_cast<uint4*>(s.q + r * 128)[qq] = z;
          reinterpret_cast<uint4*>(s.k + r * 128)[qq] = z;
          reinterpret_cast<uint4*>(s.v + r * 128)[qq] = z;
        }
      }
    fence_proxy_async_smem();
  }
  if (warp == 3) {  // chunk-local inclusive prefix of log f (read here: no barrier since the loads above)
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
  __syncthreads();

  // ---- P1: G = W W^T, M1 = Q W^T, N2 = W K^T, QK^T ----
  if (lead) {
    tc_fence_after();
    mma64(tb + 0, aw, 0, aw, 0, 0);
    mma64(tb + 64, aq, 0, aw, 0, 0);
    mma64(tb + 128, aw, 0, ak, 0, 0);
    mma64(tb + 192, aq, 0, ak, 0, 0);
    mma_commit(&s.bar_mma);
  }
  mbar_wait(&s.bar_mma, mph, p.err, 32);
  mph ^= 1;
  tc_fence_after();
  {
    float x[64];
    ld_row(tb, lane_off, 0, x);
    if (has_row)
      for (int j = 0; j < 64; ++j) s.g[i * GS + j] = j < i ? x[j] : 0.f;
    ld_row(tb, lane_off, 64, x);
    if (has_row) {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = j <= i ? x[j] : 0.f;
      put_row(s.m1, i, x);
    }
    ld_row(tb, lane_off, 128, x);
    if (has_row) {
#pragma unroll
      for (int j = 0; j < 64; ++j) x[j] = j < i ? x[j] : 0.f;
      put_row(s.n2, i, x);
    }
  }
  __syncthreads();

  // ---- P2: U by forward substitution (fp32): warps 0-1, lane = column ----
  if (warp < 2) {
    const int cc = 32 * warp + lane;
    float uc[64];
#pragma unroll
    for (int r = 0; r < 64; ++r) {
      float a0 = (cc == r) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
      for (int m = 0; m + 1 < r; m += 2) {
        a0 -= s.g[r * GS + m] * uc[m];
        a1 -= s.g[r * GS + m + 1] * uc[m + 1];
      }
      if (r & 1) a0 -= s.g[r * GS + r - 1] * uc[r - 1];
      uc[r] = s.beta[r] * (a0 + a1);
    }
#pragma unroll
    for (int r = 0; r < 64; ++r)
      *reinterpret_cast<__nv_bfloat16*>(s.u + sw128_offset(r, cc)) = __float2bfloat16_rn(uc[r]);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- P3: A = M1 U, X = U N2, Y = U^T W ----
  if (lead) {
    tc_fence_after();
    mma64(tb + 0, am1, 0, au, 1, 0);
    mma64(tb + 64, au, 0, an2, 1, 0);
    mma64(tb + 128, au, 1, aw, 1, 0);
    mma_commit(&s.bar_mma);
  }
  mbar_wait(&s.bar_mma, mph, p.err, 33);
  mph ^= 1;
  tc_fence_after();
  {
    float x[64];
    ld_row(tb, lane_off, 0, x);
    if (has_row) put_row(s.a, i, x);
    ld_row(tb, lane_off, 64, x);
    if (has_row) put_row(s.x, i, x);
    ld_row(tb, lane_off, 128, x);
    if (has_row) put_row(s.y, i, x);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();

  // ---- P4: A W, X^T W, S_d = QK^T - M1 X (accumulated onto QK^T), W^T Y ----
  if (lead) {
    tc_fence_after();
    mma64(tb + 0, aa, 0, aw, 1, 0);
    mma64(tb + 64, ax, 1, aw, 1, 0);
    mma64(tb + 192, am1, 0, ax, 1, 1, /*neg_a=*/1);
    mma64(tb + 128, aw, 1, ay, 1, 0);
    mma_commit(&s.bar_mma);
  }
  mbar_wait(&s.bar_mma, mph, p.err, 34);
  mph ^= 1;
  tc_fence_after();
  {
    float x[64], src[64];
    const size_t orow = ws_row + i;
    ld_row(tb, lane_off, 0, x);  // A W
    if (has_row) {
      get_row(s.q, i, src);
      uint4* dst = reinterpret_cast<uint4*>(p.ql + orow * D);
#pragma unroll
      for (int qq = 0; qq < 8; ++qq)
        dst[qq] = make_uint4(pack_bf16(src[8 * qq] - x[8 * qq], src[8 * qq + 1] - x[8 * qq + 1]),
                             pack_bf16(src[8 * qq + 2] - x[8 * qq + 2], src[8 * qq + 3] - x[8 * qq + 3]),
                             pack_bf16(src[8 * qq + 4] - x[8 * qq + 4], src[8 * qq + 5] - x[8 * qq + 5]),
                             pack_bf16(src[8 * qq + 6] - x[8 * qq + 6], src[8 * qq + 7] - x[8 * qq + 7]));
    }
    ld_row(tb, lane_off, 64, x);  // X^T W
    if (has_row) {
      get_row(s.k, i, src);
      uint4* dst = reinterpret_cast<uint4*>(p.kr + orow * D);
#pragma unroll
      for (int qq = 0; qq < 8; ++qq)
        dst[qq] = make_uint4(pack_bf16(src[8 * qq] - x[8 * qq], src[8 * qq + 1] - x[8 * qq + 1]),
                             pack_bf16(src[8 * qq + 2] - x[8 * qq + 2], src[8 * qq + 3] - x[8 * qq + 3]),
                             pack_bf16(src[8 * qq + 4] - x[8 * qq + 4], src[8 * qq + 5] - x[8 * qq + 5]),
                             pack_bf16(src[8 * qq + 6] - x[8 * qq + 6], src[8 * qq + 7] - x[8 * qq + 7]));
    }
    ld_row(tb, lane_off, 128, x);  // W^T Y, row n = i of F
    if (has_row) {
      uint4* dst = reinterpret_cast<uint4*>(p.f + (((size_t)bh * p.nc + c) * D + i) * D);
#pragma unroll
      for (int qq = 0; qq < 8; ++qq) {
        float e[8];
#pragma unroll
        for (int h = 0; h < 8; ++h) e[h] = (8 * qq + h == i ? 1.f : 0.f) - x[8 * qq + h];
        dst[qq] = make_uint4(pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]), pack_bf16(e[4], e[5]),
                             pack_bf16(e[6], e[7]));
      }
    }
    if (p.with_diag) {
      ld_row(tb, lane_off, 192, x);  // S_d
      if (has_row) {
        const int gi = row0 + i;
        float mx = -INFINITY;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          float sv = -INFINITY;
          if (j <= i && row0 + j < p.L) sv = x[j] * p.scl + (s.pre[i] - s.pre[j]) * kLog2e;
          x[j] = sv;
          mx = fmaxf(mx, sv);
        }
        float l = 0.f;
#pragma unroll
        for (int j = 0; j < 64; ++j) {
          const float pj = (x[j] == -INFINITY) ? 0.f : fast_exp2(x[j] - mx);
          x[j] = pj;
          l += pj;
        }
        put_row(s.p, i, x);
        p.dm[orow] = mx;
        p.dl[orow] = l;
        (void)gi;
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
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- P5: acc = P V ----
    if (lead) {
      tc_fence_after();
      mma64(tb + 0, ap, 0, av, 1, 0);
      mma_commit(&s.bar_mma);
    }
    mbar_wait(&s.bar_mma, mph, p.err, 35);
    mph ^= 1;
    tc_fence_after();
    float x[64];
    ld_row(tb, lane_off, 0, x);
    if (has_row) {
      float4* dst = reinterpret_cast<float4*>(p.dacc + (ws_row + i) * D);
#pragma unroll
      for (int j = 0; j < 16; ++j) dst[j] = make_float4(x[4 * j], x[4 * j + 1], x[4 * j + 2], x[4 * j + 3]);
    }
  }
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
                             cudaStream_t st) {
  if (g.B != 64) return cudaErrorInvalidValue;
  CUtensorMap mq, mk, mv, mw;
  const uint64_t rows = (uint64_t)g.BH * g.L;
  if (!make_map_rows64(&mq, q, rows, B) || !make_map_rows64(&mk, k, rows, B) || !make_map_rows64(&mv, v, rows, B) ||
      !make_map_rows64(&mw, w, rows, B))
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
  cudaError_t e = cudaFuncSetAttribute(ut_prep64_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  ut_prep64_kernel<<<dim3(g.nc, g.BH), 128, smem, st>>>(mq, mk, mv, mw, p);
  return cudaGetLastError();
}

}  // namespace pathattn
