// Chunk walks on tcgen05 (head dim 64, 64-row chunks): the prefill -> decode hand-off and the
// context-parallel shard transports.
//
// PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.8, last paragraph: after a prefill every
// key is moved to the prompt end with the block suffix products, and sequence parallelism moves
// keys and queries across whole shards the same way.  Blockwise (§2.6-§2.7), with the chunk
// transforms F_c = H_{s(c)} ... H_{e(c)} and rows X_c already moved to their chunk's end (K->) or
// start (Q<-), a walk over the chunks of one head computes
//   right to left:  M_{nc-1} = I,  out_c = X_c M_c^T,  M_{c-1} = M_c F_c^T   (M_c = S_c, the suffix
//                   product F_{nc-1}^T ... F_{c+1}^T; out = the keys moved to the sequence end)
//   left to right:  M_0 = I,       out_c = X_c M_c^T,  M_{c+1} = M_c F_c     (M_c = P_c^T with
//                   P_c = F_{c-1}^T ... F_0^T; out = the queries moved to the sequence start)
// and, right to left, the product of the whole sequence as M_{-1} = S_{-1}.
//
// One CTA of 128 threads per head.  The chain M is the only serial dependency, and each step is
// small (five 64 x 64 x 64 products), so the walk runs on the tensor cores: M is kept as a bf16
// high/low pair (M = M_hi + M_lo, about 16 significant bits) and F comes from the preparation in
// the same split form, so that
//   out_c  = X_c M_hi^T + X_c M_lo^T                      (X is bf16: exact as an operand)
//   M_next = M_hi F_hi^T + M_hi F_lo^T + M_lo F_hi^T      (F^T read as an MN-major B left to right)
// accumulate in fp32 in TMEM (two 64-column accumulators); only M_lo F_lo (about 2^-16 relative)
// is dropped.  A long chain of such steps does not accumulate bf16 rounding: every step rounds at
// the 2^-17 level and the transforms are contractions (eigenvalues of H in [-1, 1]).
// Per step the 128 threads read both accumulators (one half row each, the 16x32bx2 TMEM shape),
// split M_next into the two tiles the next step's MMAs read, and write out_c's rows to global
// memory after the next step's MMAs have been issued.  X_c and the split F_c come in a two-stage
// ring (TMA for X through a [heads][rows][64] tensor map, one 16 KB bulk copy for F_hi | F_lo).
#include "internal.h"
#include "dev_common.cuh"
#include "tc_common.cuh"
#include "ut_common.cuh"

#include <cuda.h>

namespace pathattn {

bool make_map_head_rows64(CUtensorMap* m, const void* base, uint64_t L, uint64_t heads);  // fwd_tc.cu

namespace {
using namespace tc;

constexpr int D = kHeadDim;
constexpr uint32_t TILE = 64 * 128;  // one 64x64 bf16 tile
constexpr uint32_t TMEM_COLS = 128;  // out_c at column 0, the next M at column 64
constexpr int NSTAGE = 2;

struct WalkParams {
  int nc, nrows;                // chunks per head; rows written per head
  const __nv_bfloat16* fs;      // split chunk transforms [BH][nc][2][64 x 64], swizzled tiles
  void* out;                    // rows [BH][out_head][64]
  size_t out_head;
  float* t_out;                 // right to left: M_{-1} [BH][64][64], or null
  int* err;
};

struct __align__(1024) WalkSmem {
  uint8_t x[NSTAGE][TILE];     // X_c
  uint8_t f[NSTAGE][2][TILE];  // F_hi, F_lo of chunk c (one bulk copy)
  uint8_t m[2][TILE];          // M_hi, M_lo
  uint64_t full[NSTAGE], bar_mma;
  uint32_t tmem_base;
};

template <bool ASC, bool OUT_F32>
__device__ __forceinline__ void walk_head(const CUtensorMap& tm_x, const WalkParams& p, int bh) {
  extern __shared__ uint8_t smem_raw[];
  WalkSmem& s = *reinterpret_cast<WalkSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  if (launch_failed(p.err)) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const bool lead = tid == 0;
  // this thread's half row of the M=64 accumulators: row i, columns 32h .. 32h+31
  const int i = 16 * warp + (lane & 15), h = lane >> 4;
  const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
  const int nc = p.nc;

  if (lead) {
    for (int st = 0; st < NSTAGE; ++st) mbar_init(&s.full[st], 1);
    mbar_init(&s.bar_mma, 1);
    fence_barrier_init();
  }
  if (warp == 1) tmem_alloc(&s.tmem_base, TMEM_COLS);
  {  // M = I
    float one[32], zero[32];
#pragma unroll
    for (int j = 0; j < 32; ++j) {
      one[j] = 32 * h + j == i ? 1.f : 0.f;
      zero[j] = 0.f;
    }
    put_half(s.m[0], i, h, one);
    put_half(s.m[1], i, h, zero);
  }
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;

  auto chunk_of = [&](int n) { return ASC ? n : nc - 1 - n; };
  // step n forms the next M unless it is the last step (right to left with t_out: M_{-1} as well)
  auto need_next = [&](int n) { return n + 1 < nc || (!ASC && p.t_out != nullptr); };
  auto load = [&](int n) {  // lead: X and the split F of step n's chunk into stage n % 2
    const int st = n & 1, c = chunk_of(n);
    mbar_arrive_expect_tx(&s.full[st], 3 * TILE);
    tma_load_3d(s.x[st], &tm_x, 0, c * 64, bh, &s.full[st]);
    bulk_load(s.f[st][0], p.fs + ((size_t)bh * nc + c) * 2 * D * D, 2 * TILE, &s.full[st]);
  };
  auto issue = [&](int n) {  // lead: the five products of step n, one commit
    const int st = n & 1;
    tc_fence_after();
    const uint32_t xa = smem_u32(s.x[st]), mh = smem_u32(s.m[0]), ml = smem_u32(s.m[1]);
    mma64(tb + 0, xa, 0, mh, 0, 0);  // X M_hi^T
    mma64(tb + 0, xa, 0, ml, 0, 1);  // + X M_lo^T
    if (need_next(n)) {
      const uint32_t fh = smem_u32(s.f[st][0]), fl = smem_u32(s.f[st][1]);
      const int fmn = ASC ? 1 : 0;  // B = F_c (K-major rows) right to left, F_c^T (MN-major) left to right
      mma64(tb + 64, mh, 0, fh, fmn, 0);
      mma64(tb + 64, mh, 0, fl, fmn, 1);
      mma64(tb + 64, ml, 0, fh, fmn, 1);
    }
    mma_commit(&s.bar_mma);
  };

  bool ok = true;
  if (lead) {
    load(0);
    if (nc > 1) load(1);
    ok = mbar_wait(&s.full[0], 0, p.err, 61);
    if (ok) issue(0);
  }
  for (int n = 0; n < nc; ++n) {
    const int c = chunk_of(n);
    const bool next = need_next(n);
    ok = mbar_wait(&s.bar_mma, n & 1, p.err, 62) && ok;
    tc_fence_after();
    if (lead && ok && n + 2 < nc) load(n + 2);  // stage n % 2 has been read by step n's MMAs
    uint32_t ro[32], rn[32];
    tmem_ld16x2(tb + lane_off + 0, ro);
    if (next) tmem_ld16x2(tb + lane_off + 64, rn);
    tmem_ld_wait();
    if (next) {
      if (n + 1 < nc) {  // M_next = hi + lo, the next step's operands
        float hi[32], lo[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) {
          const float v = __uint_as_float(rn[j]);
          hi[j] = __bfloat162float(__float2bfloat16_rn(v));
          lo[j] = v - hi[j];
        }
        put_half(s.m[0], i, h, hi);
        put_half(s.m[1], i, h, lo);
      } else {  // right to left, past the first chunk: M_{-1}
        float4* dst = reinterpret_cast<float4*>(p.t_out + ((size_t)bh * D + i) * D + 32 * h);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(rn[4 * q]), __uint_as_float(rn[4 * q + 1]),
                               __uint_as_float(rn[4 * q + 2]), __uint_as_float(rn[4 * q + 3]));
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(!ok)) break;  // a wait gave up: end the walk
    if (lead && n + 1 < nc) {
      ok = mbar_wait(&s.full[(n + 1) & 1], ((n + 1) >> 1) & 1, p.err, 61);
      if (ok) issue(n + 1);
    }
    const int r = c * 64 + i;  // out_c's row, written while the next step runs
    if (r < p.nrows) {
      if constexpr (OUT_F32) {
        float4* dst = reinterpret_cast<float4*>(reinterpret_cast<float*>(p.out) + ((size_t)bh * p.out_head + r) * D +
                                                32 * h);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(ro[4 * q]), __uint_as_float(ro[4 * q + 1]),
                               __uint_as_float(ro[4 * q + 2]), __uint_as_float(ro[4 * q + 3]));
      } else {
        float x[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __uint_as_float(ro[j]);
        store_bf16_half(reinterpret_cast<__nv_bfloat16*>(p.out) + ((size_t)bh * p.out_head + r) * D + 32 * h, x);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tb, TMEM_COLS);
  }
}

template <bool ASC, bool OUT_F32>
__global__ void __launch_bounds__(128, 3) walk_tc_kernel(const __grid_constant__ CUtensorMap tm_x, const WalkParams p) {
  walk_head<ASC, OUT_F32>(tm_x, p, (int)blockIdx.x);
}

// Both walks of a context-parallel shard in one launch (they are independent): CTAs 0 .. BH-1
// move the keys right to left (fp32 rows and the shard product), CTAs BH .. 2BH-1 the queries
// left to right (bf16 rows).
__global__ void __launch_bounds__(128, 3) walk_tc_pair_kernel(const __grid_constant__ CUtensorMap tm_k,
                                                              const __grid_constant__ CUtensorMap tm_q,
                                                              const WalkParams pk, const WalkParams pq, int BH) {
  if ((int)blockIdx.x < BH) walk_head<false, true>(tm_k, pk, (int)blockIdx.x);
  else walk_head<true, false>(tm_q, pq, (int)blockIdx.x - BH);
}

WalkParams walk_params(const Geom& g, const void* fs, void* out, size_t out_head, float* t_out, int* err) {
  WalkParams p;
  p.nc = g.nc;
  p.nrows = g.L;
  p.fs = (const __nv_bfloat16*)fs;
  p.out = out;
  p.out_head = out_head;
  p.t_out = t_out;
  p.err = err;
  return p;
}

}  // namespace

cudaError_t launch_walk_tc(const Geom& g, bool asc, bool out_f32, const void* x, const void* fs, void* out,
                           size_t out_head, float* t_out, int* err, cudaStream_t st) {
  if (g.B != 64 || g.D != D || g.Lp != g.nc * 64 || (asc && t_out) || g.nc <= 0) return cudaErrorInvalidValue;
  if (out_head < (size_t)g.L) return cudaErrorInvalidValue;
  CUtensorMap mx;
  if (!make_map_head_rows64(&mx, x, g.Lp, g.BH)) return cudaErrorInvalidValue;
  const WalkParams p = walk_params(g, fs, out, out_head, t_out, err);
  const size_t smem = sizeof(WalkSmem) + 1024;
  auto kern = asc ? (out_f32 ? walk_tc_kernel<true, true> : walk_tc_kernel<true, false>)
                  : (out_f32 ? walk_tc_kernel<false, true> : walk_tc_kernel<false, false>);
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)g.BH, 128, smem, st>>>(mx, p);
  return cudaGetLastError();
}

}  // namespace pathattn

namespace pathattn {

cudaError_t launch_walk_tc_pair(const Geom& g, const void* xk, const void* xq, const void* fs, float* k_out,
                                void* q_out, size_t out_head, float* t_out, int* err, cudaStream_t st) {
  if (g.B != 64 || g.D != D || g.Lp != g.nc * 64 || g.nc <= 0 || out_head < (size_t)g.L) return cudaErrorInvalidValue;
  CUtensorMap mk, mq;
  if (!make_map_head_rows64(&mk, xk, g.Lp, g.BH) || !make_map_head_rows64(&mq, xq, g.Lp, g.BH))
    return cudaErrorInvalidValue;
  const WalkParams pk = walk_params(g, fs, k_out, out_head, t_out, err);
  const WalkParams pq = walk_params(g, fs, q_out, out_head, nullptr, err);
  const size_t smem = sizeof(WalkSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(walk_tc_pair_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  walk_tc_pair_kernel<<<(unsigned)(2 * g.BH), 128, smem, st>>>(mk, mq, pk, pq, g.BH);
  return cudaGetLastError();
}

}  // namespace pathattn
