// tcgen05 forward scan of PaTH attention (bf16 operands, fp32 accumulation in TMEM).
//
// Method: the right-to-left chunk scan of the PaTH reading notes (cc.laoqi.cc/papers/2505.16381),
// §2.7: for a query tile, Z starts at the boundary-adjusted queries Q<-; for each earlier key
// chunk c (right to left) the scores are Z K->_c^T, the online softmax accumulates P V_c, and
// Z <- Z F_c^T carries the queries across chunk c.
//
// GB300 mapping (one CTA = one 128-row query tile = two 64-row UT chunks; 2 CTAs per SM):
//   * warp 4 streams [K->_c ; F_c] (one 128x64 tile) and V_c with TMA into a 3-stage ring;
//   * warp 5 issues the MMAs: one M=128 N=128 K=64 MMA gives the scores S and the transported
//     queries Z' = Z F_c^T together (the B operand stacks K->_c over F_c), and an M=128 N=64
//     K=64 MMA with P read from TMEM accumulates O += P V_c;
//   * warps 0-3 (one thread per query row / TMEM lane) run the online softmax on S (lazy
//     rescaling of O when the running max grows by more than 8 in log2 units), write P to TMEM
//     and Z' (rounded to bf16) to the swizzled shared-memory Z tile for the next step.
// The upper chunk of the tile first meets the lower chunk as an ordinary earlier chunk (the
// "partial" step: lower rows masked, only upper rows transported), then all 128 rows scan
// together.  The diagonal chunks come from the preparation kernel as softmax partial states.
#include "internal.h"
#include "dev_common.cuh"
#include "tc_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace pathattn {
namespace {
using namespace tc;

constexpr int BQ = 128;
constexpr int BK = 64;
constexpr int D = kHeadDim;
constexpr int NSTAGE = 3;
constexpr int NTHREADS = 192;
constexpr uint32_t TMEM_COLS = 256;
// S double-buffered (P of step n is written over S of step n), one Z' buffer, O.
constexpr uint32_t COL_S0 = 0, COL_Z = 128, COL_O = 192;
constexpr float kTau = 8.f;  // lazy-rescale threshold (log2 units)

struct __align__(1024) ScanSmem {
  uint8_t z[BQ * 128];                // Z tile, bf16, 128-byte swizzled rows
  uint8_t kf[NSTAGE][128 * 128];      // rows 0-63: K->_c, rows 64-127: F_c
  uint8_t v[NSTAGE][BK * 128];        // V_c
  uint64_t full[NSTAGE], empty[NSTAGE];
  // p_ready alternates by step parity: a thread may arrive for step n+1 before a slower one has
  // arrived for step n (the next score MMA only waits for z_ready), never two steps ahead.
  uint64_t s_full[2], z_ready, p_ready[2], pv_done, o_done, z_init;
  uint32_t tmem_base;
};

struct ScanParams {
  int L, Lp, nc, BH, ntiles;
  float scl;  // scale * log2(e)
  const float* dm;
  const float* dl;
  const float* dacc;
  const float* fa;
  const float* fr;
  const float* ft;
  int fox;
  __nv_bfloat16* o;
  float* lse;
  int* err;
};

__global__ void __launch_bounds__(NTHREADS, 2)
    fwd_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_ql, const __grid_constant__ CUtensorMap tm_kr,
                       const __grid_constant__ CUtensorMap tm_f, const __grid_constant__ CUtensorMap tm_v,
                       const ScanParams p) {
  extern __shared__ uint8_t smem_raw[];
  ScanSmem& s = *reinterpret_cast<ScanSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bh, T;
  tile_of_block((int)blockIdx.x, p.ntiles, p.BH, bh, T);
  const bool has_partial = (2 * T + 1) * BK < p.L;
  const int nsteps = (has_partial ? 1 : 0) + 2 * T;

  if (tid == 0) {
    for (int k = 0; k < NSTAGE; ++k) {
      mbar_init(&s.full[k], 1);
      mbar_init(&s.empty[k], 1);
    }
    mbar_init(&s.s_full[0], 1);
    mbar_init(&s.s_full[1], 1);
    mbar_init(&s.z_ready, 128);
    mbar_init(&s.p_ready[0], 128);
    mbar_init(&s.p_ready[1], 128);
    mbar_init(&s.pv_done, 1);
    mbar_init(&s.o_done, 1);
    mbar_init(&s.z_init, 1);
    fence_barrier_init();
  }
  if (warp == 5) tmem_alloc(&s.tmem_base, TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tb = s.tmem_base;

  if (warp == 4) {
    // ---------------- TMA producer ----------------
    if (lane == 0 && nsteps > 0) {
      prefetch_tmap(&tm_ql);
      prefetch_tmap(&tm_kr);
      prefetch_tmap(&tm_f);
      prefetch_tmap(&tm_v);
      mbar_arrive_expect_tx(&s.z_init, BQ * 128);
      tma_load_2d(s.z, &tm_ql, 0, bh * p.Lp + T * BQ, &s.z_init);
      for (int n = 0; n < nsteps; ++n) {
        const int st = n % NSTAGE;
        if (n >= NSTAGE && !mbar_wait(&s.empty[st], ((n / NSTAGE) - 1) & 1, p.err, 1)) break;
        const int c = has_partial ? 2 * T - n : 2 * T - 1 - n;
        mbar_arrive_expect_tx(&s.full[st], 128 * 128 + BK * 128);
        tma_load_2d(s.kf[st], &tm_kr, 0, bh * p.Lp + c * BK, &s.full[st]);
        tma_load_2d(s.kf[st] + 64 * 128, &tm_f, 0, (bh * p.nc + c) * D, &s.full[st]);
        tma_load_2d(s.v[st], &tm_v, 0, bh * p.L + c * BK, &s.full[st]);
      }
    }
  } else if (warp == 5) {
    // ---------------- MMA issuer ----------------
    // order: S(n), Z'(n) as soon as Z(n) is in shared memory; then O += P(n-1) V(n-1).
    if (lane == 0 && nsteps > 0) {
      const uint32_t idesc_n64 = idesc_bf16(128, 64, 0, 0);
      const uint32_t idesc_pv = idesc_bf16(128, 64, 0, 1);
      const uint32_t zaddr = smem_u32(s.z);
      bool ok = mbar_wait(&s.z_init, 0, p.err, 2);
      auto issue_pv = [&](int m) {
        const uint32_t va = smem_u32(s.v[m % NSTAGE]);
        const uint32_t pcol = COL_S0 + 64 * (m & 1);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ts(tb + COL_O, tb + pcol + 8 * k, sdesc_sw128(va + 2048 * k, 1024, 0), idesc_pv, 1);
        mma_commit(&s.empty[m % NSTAGE]);
        mma_commit(&s.pv_done);
      };
      for (int n = 0; ok && n < nsteps; ++n) {
        const int st = n % NSTAGE;
        if (!mbar_wait(&s.full[st], (n / NSTAGE) & 1, p.err, 3)) { ok = false; break; }
        if (n > 0 && !mbar_wait(&s.z_ready, (n - 1) & 1, p.err, 4)) { ok = false; break; }
        tc_fence_after();
        const uint32_t kfa = smem_u32(s.kf[st]);
        const uint32_t scol = COL_S0 + 64 * (n & 1);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tb + scol, sdesc_sw128(zaddr + 32 * k, 1024, 16), sdesc_sw128(kfa + 32 * k, 1024, 16),
                 idesc_n64, k > 0 ? 1u : 0u);
#pragma unroll
        for (int k = 0; k < 4; ++k)
          mma_ss(tb + COL_Z, sdesc_sw128(zaddr + 32 * k, 1024, 16),
                 sdesc_sw128(kfa + 64 * 128 + 32 * k, 1024, 16), idesc_n64, k > 0 ? 1u : 0u);
        mma_commit(&s.s_full[n & 1]);
        if (n > 0) {
          if (!mbar_wait(&s.p_ready[(n - 1) & 1], ((n - 1) >> 1) & 1, p.err, 5)) { ok = false; break; }
          tc_fence_after();
          issue_pv(n - 1);
        }
      }
      if (ok && mbar_wait(&s.p_ready[(nsteps - 1) & 1], ((nsteps - 1) >> 1) & 1, p.err, 5)) {
        tc_fence_after();
        issue_pv(nsteps - 1);
        mma_commit(&s.o_done);
      }
    }
  } else {
    // ---------------- softmax / transport warpgroup: thread r owns query row r ----------------
    const int r = tid;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    const int grow = T * BQ + r;
    const size_t wrow = (size_t)bh * p.Lp + (size_t)T * BQ + r;
    float m = p.dm[wrow], l = p.dl[wrow];
    uint32_t buf[32];
    if (nsteps > 0) {
#pragma unroll
      for (int h = 0; h < 2; ++h) {
#pragma unroll
        for (int j = 0; j < 32; ++j) buf[j] = __float_as_uint(p.dacc[wrow * D + h * 32 + j]);
        tmem_st32(tb + lane_off + COL_O + h * 32, buf);
      }
      tmem_st_wait();
    }
    const float arow = p.fox ? p.fa[wrow] : 0.f;
    float R = 0.f;
    bool ok = true;
    for (int n = 0; n < nsteps; ++n) {
      if (!mbar_wait(&s.s_full[n & 1], (n >> 1) & 1, p.err, 6)) { ok = false; break; }
      tc_fence_after();
      const int c = has_partial ? 2 * T - n : 2 * T - 1 - n;
      const bool active = !(has_partial && n == 0 && r < 64);
      const uint32_t scol = COL_S0 + 64 * (n & 1);
      uint32_t buf2[32];
      // transport first: Z <- Z F_c^T (bf16) so that the next score MMA can start
      if (n + 1 < nsteps) {
        if (active) {
          tmem_ld32(tb + lane_off + COL_Z, buf);
          tmem_ld32(tb + lane_off + COL_Z + 32, buf2);
          tmem_ld_wait();
          uint8_t* zrow = s.z + r * 128;
#pragma unroll
          for (int q = 0; q < 8; ++q) {
            const uint32_t* src = (q < 4) ? (buf + 8 * q) : (buf2 + 8 * (q - 4));
            uint4 pk;
            pk.x = pack_bf16(__uint_as_float(src[0]), __uint_as_float(src[1]));
            pk.y = pack_bf16(__uint_as_float(src[2]), __uint_as_float(src[3]));
            pk.z = pack_bf16(__uint_as_float(src[4]), __uint_as_float(src[5]));
            pk.w = pack_bf16(__uint_as_float(src[6]), __uint_as_float(src[7]));
            *reinterpret_cast<uint4*>(zrow + ((q ^ (r & 7)) * 16)) = pk;
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&s.z_ready);
      }
      // scores (log2 domain, in place in the load registers)
      tmem_ld32(tb + lane_off + scol, buf);
      tmem_ld32(tb + lane_off + scol + 32, buf2);
      tmem_ld_wait();
      const float rb = (arow + R) * kLog2e;
      float mx = -INFINITY;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        float x0 = fmaf(__uint_as_float(buf[j]), p.scl, rb);
        float x1 = fmaf(__uint_as_float(buf2[j]), p.scl, rb);
        if (p.fox) {
          x0 += __ldg(p.fr + (size_t)bh * p.Lp + (size_t)c * BK + j) * kLog2e;
          x1 += __ldg(p.fr + (size_t)bh * p.Lp + (size_t)c * BK + 32 + j) * kLog2e;
        }
        if (!active) {
          x0 = -INFINITY;
          x1 = -INFINITY;
        }
        mx = fmaxf(mx, fmaxf(x0, x1));
        buf[j] = __float_as_uint(x0);
        buf2[j] = __float_as_uint(x1);
      }
      const float mnew = fmaxf(m, mx);
      const bool resc = mnew > m + kTau;
      if (__any_sync(0xffffffffu, resc)) {
        // O holds P(n-1) V(n-1) only once that MMA has completed
        if (n > 0 && !mbar_wait(&s.pv_done, (n - 1) & 1, p.err, 8)) { ok = false; break; }
        tc_fence_after();
        const float corr = resc ? fast_exp2(m - mnew) : 1.f;
        if (resc) m = mnew;
        l *= corr;
        uint32_t ob[32];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          tmem_ld32(tb + lane_off + COL_O + h * 32, ob);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) ob[j] = __float_as_uint(__uint_as_float(ob[j]) * corr);
          tmem_st32(tb + lane_off + COL_O + h * 32, ob);
        }
      }
      // probabilities, packed bf16 pairs (key 2j in the low half), written over S(n)
      float ls = 0.f;
      {
        uint32_t pk[32];
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          const float p0 = fast_exp2(__uint_as_float(buf[2 * j]) - m);
          const float p1 = fast_exp2(__uint_as_float(buf[2 * j + 1]) - m);
          const float p2 = fast_exp2(__uint_as_float(buf2[2 * j]) - m);
          const float p3 = fast_exp2(__uint_as_float(buf2[2 * j + 1]) - m);
          ls += (p0 + p1) + (p2 + p3);
          pk[j] = pack_bf16(p0, p1);
          pk[16 + j] = pack_bf16(p2, p3);
        }
        tmem_st32(tb + lane_off + scol, pk);
      }
      l += ls;
      if (active && p.fox) R += p.ft[(size_t)bh * p.nc + c];
      tmem_st_wait();
      tc_fence_before();
      mbar_arrive(&s.p_ready[n & 1]);
    }
    // ---------------- epilogue ----------------
    if (nsteps > 0) {
      if (ok) ok = mbar_wait(&s.o_done, 0, p.err, 7);
      tc_fence_after();
    }
    const float inv = 1.f / l;
    uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)bh * p.L + (grow < p.L ? grow : 0)) * D);
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      if (nsteps > 0) {
        tmem_ld32(tb + lane_off + COL_O + h * 32, buf);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) buf[j] = __float_as_uint(p.dacc[wrow * D + h * 32 + j]);
      }
      if (grow < p.L) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 pk;
          pk.x = pack_bf16(__uint_as_float(buf[8 * q]) * inv, __uint_as_float(buf[8 * q + 1]) * inv);
          pk.y = pack_bf16(__uint_as_float(buf[8 * q + 2]) * inv, __uint_as_float(buf[8 * q + 3]) * inv);
          pk.z = pack_bf16(__uint_as_float(buf[8 * q + 4]) * inv, __uint_as_float(buf[8 * q + 5]) * inv);
          pk.w = pack_bf16(__uint_as_float(buf[8 * q + 6]) * inv, __uint_as_float(buf[8 * q + 7]) * inv);
          dst[h * 4 + q] = pk;
        }
      }
    }
    if (grow < p.L) p.lse[(size_t)bh * p.L + grow] = (m + log2f(l)) * kLn2;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tb, TMEM_COLS);
  }
}

}  // namespace

// ---------------- host side ----------------
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  }
  return fn;
}

// 2-D map over a [rows][64] bf16 matrix with 128-byte swizzled boxes of box_rows x 64.
bool make_map_rows64(CUtensorMap* m, const void* base, uint64_t rows, uint32_t box_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {64, rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {64, box_rows};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [heads][L][64] bf16 tensor seen in 64-row boxes of one head; rows >= L read as zero.
bool make_map_head_rows64(CUtensorMap* m, const void* base, uint64_t L, uint64_t heads) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, L, heads};
  cuuint64_t strides[2] = {128, L * 128};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_scan_tc(const Geom& g, const void* v, const float* logf, char* ws,
                           const FwdWs& lay, void* o, float* lse, cudaStream_t st) {
  if (g.B != BK || (g.nc & 1) || g.Lp != g.nc * BK) return cudaErrorInvalidValue;
  CUtensorMap m_ql, m_kr, m_f, m_v;
  const uint64_t prow = (uint64_t)g.BH * g.Lp;
  if (!make_map_rows64(&m_ql, ws + lay.ql, prow, BQ) || !make_map_rows64(&m_kr, ws + lay.kr, prow, BK) ||
      !make_map_rows64(&m_f, ws + lay.f, (uint64_t)g.BH * g.nc * D, D) ||
      !make_map_rows64(&m_v, v, (uint64_t)g.BH * g.L, BK))
    return cudaErrorInvalidValue;
  ScanParams p;
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
  p.fox = logf ? 1 : 0;
  p.o = (__nv_bfloat16*)o;
  p.lse = lse;
  p.err = (int*)(ws + lay.err);
  const size_t smem = sizeof(ScanSmem) + 1024;
  cudaError_t e = cudaFuncSetAttribute(fwd_scan_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const long ntiles = (long)p.ntiles * g.BH;
  fwd_scan_tc_kernel<<<(unsigned)ntiles, NTHREADS, smem, st>>>(m_ql, m_kr, m_f, m_v, p);
  return cudaGetLastError();
}

}  // namespace pathattn
