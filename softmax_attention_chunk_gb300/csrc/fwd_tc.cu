// tcgen05 forward scan of PaTH attention (bf16 operands, fp32 accumulation in TMEM).
//
// Method: the right-to-left chunk scan of the PaTH reading notes (cc.laoqi.cc/papers/2505.16381),
// §2.7: for a query tile, Z starts at the boundary-adjusted queries Q<-; for each earlier key
// chunk c (right to left) the scores are Z K->_c^T, the online softmax accumulates P V_c, and
// Z <- Z F_c^T carries the queries across chunk c.
//
// GB300 mapping (one CTA = one 128-row query tile = two 64-row UT chunks; 2 CTAs per SM):
//   * warp 8 streams [K->_c ; F_c] (one 128x64 tile) and V_c with TMA into a 3-stage ring;
//   * warp 9 issues the MMAs, all with the A operand in TMEM: one N=128 MMA gives the scores
//     S = Z K->_c^T and the transported queries Z' = Z F_c^T together (the B tile stacks K->_c
//     over F_c) from the bf16 Z held in TMEM, and O += P V_c reads P from TMEM; shared memory
//     only supplies the B tiles;
//   * warps 0-7 run the softmax, two threads per query row (TMEM lane): warps w and w+4 share
//     the lanes of quarter w and take the column halves 0-31 and 32-63 of S, Z', O and the
//     matching halves of Z and P.  Each step a thread first turns its half of Z' into bf16 Z
//     (TMEM to registers to TMEM) and reads its half of S, which frees both for the next
//     MMAs, then runs the online softmax.  The two halves of a row share the running max: it
//     only changes when some row's scores exceed it by more than 8 (log2 units, lazy
//     rescaling of O); one barrier-reduction per step tells all threads whether that happened,
//     and only then do the halves exchange their maxima through shared memory.  The softmax
//     is instruction-issue bound: without a forget gate the maximum is taken over the raw
//     scores (3-input max), and the scaling, the max subtraction and the row sums use paired
//     fp32 instructions.
// The upper chunk of the tile first meets the lower chunk as an ordinary earlier chunk (the
// "partial" step: lower rows masked, only upper rows transported), then all 128 rows scan
// together.  The diagonal chunks come from the preparation kernel as softmax partial states.
#include "internal.h"
#include "dev_common.cuh"
#include "tc_common.cuh"
#include "scan_common.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace pathattn {
namespace {
using namespace tc;

constexpr int BQ = 128;
constexpr int BK = 64;
constexpr int D = kHeadDim;
constexpr int NSTAGE = 3;
constexpr int NSOFT = 256;  // softmax threads: two per query row
constexpr int NTHREADS = NSOFT + 64;
constexpr uint32_t TMEM_COLS = 256;
// TMEM: scores S, transported queries Z' (fp32), output O, probabilities P (bf16 pairs), transported
// queries Z (bf16 pairs, A operand of the score and transport MMAs).
constexpr uint32_t COL_S = 0, COL_ZP = 64, COL_O = 128, COL_P = 192, COL_Z = 224;
constexpr float kTau = 8.f;  // lazy-rescale threshold (log2 units)

struct __align__(1024) ScanSmem {
  uint8_t z0[BQ * 128];               // Q<- tile (bf16, 128-byte swizzled rows): the first Z; after
                                      // step 0 the image buffer of the even Z tiles
  uint8_t kf[NSTAGE][128 * 128];      // rows 0-63: K->_c, rows 64-127: F_c
  uint8_t v[NSTAGE][BK * 128];        // V_c
  float xm[2][BQ];                    // per-half row maxima / sums exchanged between the halves
  float frs[NSTAGE][BK];              // PaTH-FoX: the chunk's suffix sums of log f (with K->_c, F_c, V_c)
  uint64_t full[NSTAGE], empty[NSTAGE];
  uint64_t z_init, z_ready, s_full, p_ready, pv_done, o_done, zbuf_free[2];
  uint32_t tmem_base;
  // last, so that a launch without the Z store leaves it out of its shared memory (16 KB less
  // per CTA: more of the SM's unified memory stays L1)
  alignas(1024) uint8_t zout[BQ * 128];  // image buffer of the odd Z tiles on their way to the Z store
};
// Dynamic shared memory of a launch (with the 1 KB alignment slack): without the Z store the
// buffer that only the store uses is not allocated.
constexpr size_t scan_smem_bytes(bool zstore) {
  return (zstore ? sizeof(ScanSmem) : offsetof(ScanSmem, zout)) + 1024;
}

struct ScanParams {
  int L, Lp, nc, BH, ntiles;
  int Lk;     // rows per head of the K-> (and, in block mode, V) tensor: Lp, or the block's length
  int nkc;    // block mode: key chunks of the block
  float scl;  // scale * log2(e)
  float* dm;  // diagonal-chunk softmax state (read; block mode also writes it back)
  float* dl;
  float* dacc;
  const float* fa;
  const float* fr;
  const float* ft;
  __nv_bfloat16* o;
  float* lse;
  uint8_t* zs;  // if set: every transported query tile Z_n is stored for the backward (bulk copies
                // of a shared-memory tile image issued by the MMA warp)
  int* err;
};

// Part of a 128-row bf16 tile in its 128-byte swizzled image (the layout TMA writes and the
// backward bulk-copies): the four 16-byte chunks 4h..4h+3 of row r.
__device__ __forceinline__ void put_tile_quarter(uint8_t* tile, int r, int h, const uint32_t* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(tile + r * 128 + (((4 * h + q) ^ (r & 7)) * 16)) =
        make_uint4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
}


// BLOCK (context-parallel block mode): every query tile visits every 64-row chunk of a separate
// key block (K-> = the block's keys, V = the block's values, no transport: the queries stay where
// the shard start put them, so no F is loaded, the MMA forms S alone and Z is never rewritten; FoX: fa holds
// the queries' bias, fr the keys'), starting from and writing back the softmax state in dm, dl,
// dacc (unnormalised), instead of the causal chunk range and the o / lse epilogue.
template <bool FOX, bool BLOCK>
__global__ void __launch_bounds__(NTHREADS, 2)
    fwd_scan_tc_kernel(const __grid_constant__ CUtensorMap tm_ql, const __grid_constant__ CUtensorMap tm_kr,
                       const __grid_constant__ CUtensorMap tm_f, const __grid_constant__ CUtensorMap tm_v,
                       const ScanParams p) {
  extern __shared__ uint8_t smem_raw[];
  ScanSmem& s = *reinterpret_cast<ScanSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int err0 = threadIdx.x == 0 ? peek_err(p.err) : 0;  // consumed at the setup barrier
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  int bh, T;
  if constexpr (BLOCK) {
    bh = (int)blockIdx.x / p.ntiles;
    T = (int)blockIdx.x % p.ntiles;
  } else {
    tile_of_block((int)blockIdx.x, p.ntiles, p.BH, bh, T);
  }
  const bool has_partial = !BLOCK && (2 * T + 1) * BK < p.L;
  const int nsteps = BLOCK ? p.nkc : (has_partial ? 1 : 0) + 2 * T;
  auto step_chunk = [&](int n) { return BLOCK ? p.nkc - 1 - n : (has_partial ? 2 * T - n : 2 * T - 1 - n); };

  if (tid == 0) {
    for (int k = 0; k < NSTAGE; ++k) {
      mbar_init(&s.full[k], 1);
      mbar_init(&s.empty[k], 1);
    }
    mbar_init(&s.z_init, 1);
    mbar_init(&s.z_ready, NSOFT);
    mbar_init(&s.s_full, 1);
    mbar_init(&s.p_ready, NSOFT);
    mbar_init(&s.pv_done, 1);
    mbar_init(&s.o_done, 1);
    mbar_init(&s.zbuf_free[0], 1);
    mbar_init(&s.zbuf_free[1], 1);
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
      mbar_arrive_expect_tx(&s.z_init, BQ * 128);
      tma_load_2d(s.z0, &tm_ql, 0, bh * p.Lp + T * BQ, &s.z_init);
      for (int n = 0; n < nsteps; ++n) {
        const int st = n % NSTAGE;
        if (n >= NSTAGE && !mbar_wait(&s.empty[st], ((n / NSTAGE) - 1) & 1, p.err, 1)) break;
        const int c = step_chunk(n);
        mbar_arrive_expect_tx(&s.full[st], (BLOCK ? 64 : 128) * 128 + BK * 128 + (FOX ? BK * 4 : 0));
        tma_load_2d(s.kf[st], &tm_kr, 0, bh * p.Lk + c * BK, &s.full[st]);
        if (!BLOCK) tma_load_2d(s.kf[st] + 64 * 128, &tm_f, 0, (bh * p.nc + c) * D, &s.full[st]);
        tma_load_2d(s.v[st], &tm_v, 0, bh * (BLOCK ? p.Lk : p.L) + c * BK, &s.full[st]);
        if constexpr (FOX) bulk_load(s.frs[st], p.fr + (size_t)bh * p.Lk + (size_t)c * BK, BK * 4, &s.full[st]);
      }
    }
  } else if (warp == 9) {
    // ---------------- MMA issuer ----------------
    // order: S(n), Z'(n) once Z(n) is in TMEM and S(n-1), Z'(n-1) have been read; then
    // O += P(n-1) V(n-1) once P(n-1) is written.
    if (lane == 0 && nsteps > 0) {
      // S and Z' come from one N=128 MMA: the stage tile stacks K->_c (rows 0-63) over F_c, and
      // the S and Z' TMEM blocks are adjacent.  Descriptors advance by plain 64-bit adds (the
      // start-address field counts 16-byte units).
      const uint32_t idesc_sz = idesc_bf16(128, BLOCK ? 64 : 128, 0, 0);  // block mode: S alone
      const uint32_t idesc_pv = idesc_bf16(128, 64, 0, 1);
      // stage st of the kf / v rings lies st * 16 KB / st * 8 KB after stage 0
      const uint64_t dkf0 = sdesc_sw128(smem_u32(s.kf[0]), 1024, 16);
      const uint64_t dv0 = sdesc_sw128(smem_u32(s.v[0]), 1024, 0);
      bool ok = true;
      auto issue_pv = [&](int m) {
        const uint64_t d0 = dv0 + (uint64_t)(512 * (m % NSTAGE));
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_ts(tb + COL_O, tb + COL_P + 8 * k, d0 + (uint64_t)(128 * k), idesc_pv, 1);
        mma_commit(&s.empty[m % NSTAGE]);
        mma_commit(&s.pv_done);
      };
      // Z store of this tile: tile n of the tile's sequence at n * 16 KB (the tiles of earlier query
      // tiles of the head come first: sum_{t<T} (2t+1) = T^2)
      uint8_t* zstore = p.zs ? p.zs + ((size_t)bh * p.ntiles * p.ntiles + (size_t)T * T) * (BQ * 128) : nullptr;
      for (int n = 0; ok && n < nsteps; ++n) {
        const int st = n % NSTAGE;
        if (!mbar_wait(&s.full[st], (n / NSTAGE) & 1, p.err, 3)) { ok = false; break; }
        if (!mbar_wait(&s.z_ready, n & 1, p.err, 4)) { ok = false; break; }
        tc_fence_after();
        if (zstore) {  // Z_n from image buffer n % 2 (Z_0 is the Q<- tile itself)
          bulk_store(zstore + (size_t)n * (BQ * 128), (n & 1) ? s.zout : s.z0, BQ * 128);
          bulk_commit();
        }
        const uint64_t d0 = dkf0 + (uint64_t)(1024 * st);
#pragma unroll
        for (int k = 0; k < 4; ++k) mma_ts(tb + COL_S, tb + COL_Z + 8 * k, d0 + (uint64_t)(2 * k), idesc_sz, k > 0 ? 1u : 0u);
        mma_commit(&s.s_full);
        if (zstore && n >= 1) {  // the copy of Z_{n-1} has read its buffer, which may take Z_{n+1}
          bulk_wait_read1();
          mbar_arrive(&s.zbuf_free[(n - 1) & 1]);
        }
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
      if (zstore) bulk_wait0();  // the Z store is complete before the CTA exits
    }
  } else {
    // ---------------- softmax / transport: thread (r, h) owns columns 32h..32h+31 of row r ----------------
    const int q4 = warp & 3, h = warp >> 2;
    const int r = 32 * q4 + lane;
    const uint32_t lane_off = (uint32_t)(q4 * 32) << 16;
    const uint32_t c_s = tb + lane_off + COL_S + 32 * h, c_zp = tb + lane_off + COL_ZP + 32 * h;
    const uint32_t c_o = tb + lane_off + COL_O + 32 * h, c_p = tb + lane_off + COL_P + 16 * h;
    const uint32_t c_z = tb + lane_off + COL_Z + 16 * h;
    const int grow = T * BQ + r;
    const size_t wrow = (size_t)bh * p.Lp + (size_t)T * BQ + r;
    float m = p.dm[wrow], l = h == 0 ? p.dl[wrow] : 0.f;  // l: this half's share of the row sum
    uint32_t x[32];
    bool ok = true;
    if (nsteps > 0) {
#pragma unroll
      for (int j = 0; j < 32; ++j) x[j] = __float_as_uint(p.dacc[wrow * D + h * 32 + j]);
      tmem_st32(c_o, x);
      // Z_0 = Q<- of the tile: shared memory (swizzled rows) -> TMEM
      ok = mbar_wait(&s.z_init, 0, p.err, 2);  // (on a timeout the tile below is garbage; err is set)
      const uint8_t* zrow = s.z0 + r * 128;
      uint32_t z16[16];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const uint4 v = *reinterpret_cast<const uint4*>(zrow + (((4 * h + q) ^ (r & 7)) * 16));
        z16[4 * q] = v.x;
        z16[4 * q + 1] = v.y;
        z16[4 * q + 2] = v.z;
        z16[4 * q + 3] = v.w;
      }
      tmem_st16(c_z, z16);
      tmem_st_wait();
      tc_fence_before();
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
      // transport first: Z <- bf16(Z F_c^T) into TMEM, so that the next MMAs can start
      if (!BLOCK && n + 1 < nsteps && active) {
        tmem_ld32(c_zp, x);
        tmem_ld_wait();
        uint32_t z16[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) z16[j] = pack_bf16(__uint_as_float(x[2 * j]), __uint_as_float(x[2 * j + 1]));
        tmem_st16(c_z, z16);
        if (p.zs) {  // Z_{n+1} into image buffer (n+1) % 2 once the bulk copy of Z_{n-1} has read it
          if (n >= 1) ok = ok && mbar_wait(&s.zbuf_free[(n + 1) & 1], ((n - 1) >> 1) & 1, p.err, 10);
          put_tile_quarter((n & 1) ? s.z0 : s.zout, r, h, z16);
          fence_proxy_async_smem();
        }
      } else if (n + 1 < nsteps && p.zs) {  // rows not transported at the partial step keep Z_0
        const uint4* src = reinterpret_cast<const uint4*>(s.z0 + r * 128);
        uint32_t z16[16];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const uint4 v = src[(4 * h + q) ^ (r & 7)];
          z16[4 * q] = v.x;
          z16[4 * q + 1] = v.y;
          z16[4 * q + 2] = v.z;
          z16[4 * q + 3] = v.w;
        }
        if (n >= 1) ok = ok && mbar_wait(&s.zbuf_free[(n + 1) & 1], ((n - 1) >> 1) & 1, p.err, 10);
        put_tile_quarter((n & 1) ? s.z0 : s.zout, r, h, z16);
        fence_proxy_async_smem();
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
      if (FOX) {
        // the keys' suffix sums came with the chunk's stage (its barrier completed before S was
        // issued; the stage is refilled only after this step's P V)
        ok = ok && mbar_wait(&s.full[n % NSTAGE], (n / NSTAGE) & 1, p.err, 11);
        // x = scl s + (A_i + R) log2(e) + r_j log2(e), two keys per paired instruction
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
        // the TMEM load and store of O are warp-wide instructions: a warp with any row to rescale
        // rescales all 32 of its rows, by 1 where the reference stays
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
          uint32_t ob[32];
          tmem_ld32(c_o, ob);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) ob[j] = __float_as_uint(__uint_as_float(ob[j]) * corr);
          tmem_st32(c_o, ob);
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
        if (FOX && !BLOCK) R += p.ft[(size_t)bh * p.nc + c];
      } else {
#pragma unroll
        for (int j = 0; j < 16; ++j) pk[j] = 0u;
      }
      // P(n-1) has been consumed by its MMA before P(n) replaces it
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
    if constexpr (BLOCK) {  // the merged state goes back where it came from (rows padded to Lp)
      if (nsteps > 0) {
        tmem_ld32(c_o, x);
        tmem_ld_wait();
        float4* dst = reinterpret_cast<float4*>(p.dacc + wrow * D + 32 * h);
#pragma unroll
        for (int q = 0; q < 8; ++q)
          dst[q] = make_float4(__uint_as_float(x[4 * q]), __uint_as_float(x[4 * q + 1]),
                               __uint_as_float(x[4 * q + 2]), __uint_as_float(x[4 * q + 3]));
        if (h == 0) {
          p.dm[wrow] = m;
          p.dl[wrow] = lt;
        }
      }
    } else {
      const float inv = 1.f / lt;
      if (nsteps > 0) {
        tmem_ld32(c_o, x);
        tmem_ld_wait();
      } else {
#pragma unroll
        for (int j = 0; j < 32; ++j) x[j] = __float_as_uint(p.dacc[wrow * D + h * 32 + j]);
      }
      if (grow < p.L) {
        uint4* dst = reinterpret_cast<uint4*>(p.o + ((size_t)bh * p.L + grow) * D + 32 * h);
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 pk;
          pk.x = pack_bf16(__uint_as_float(x[8 * q]) * inv, __uint_as_float(x[8 * q + 1]) * inv);
          pk.y = pack_bf16(__uint_as_float(x[8 * q + 2]) * inv, __uint_as_float(x[8 * q + 3]) * inv);
          pk.z = pack_bf16(__uint_as_float(x[8 * q + 4]) * inv, __uint_as_float(x[8 * q + 5]) * inv);
          pk.w = pack_bf16(__uint_as_float(x[8 * q + 6]) * inv, __uint_as_float(x[8 * q + 7]) * inv);
          dst[q] = pk;
        }
        if (h == 0) p.lse[(size_t)bh * p.L + grow] = (m + log2f(lt)) * kLn2;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
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

// [rows][64] fp32 matrix seen in 64-row x 32-column boxes with 128-byte swizzle (targets of the
// backward's bulk reductions).
bool make_map_f32_rows64(CUtensorMap* m, const void* base, uint64_t rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {64, rows};
  cuuint64_t strides[1] = {256};
  cuuint32_t box[2] = {32, 64};
  cuuint32_t es[2] = {1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// [heads][L][64] bf16 tensor (head_rows rows between heads) seen in 64-row boxes of one head; rows
// >= L read as zero and are not written by stores.
bool make_map_head_rows64_pitch(CUtensorMap* m, const void* base, uint64_t L, uint64_t heads, uint64_t head_rows) {
  auto enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[3] = {64, L, heads};
  cuuint64_t strides[2] = {128, head_rows * 128};
  cuuint32_t box[3] = {64, 64, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides, box, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}
bool make_map_head_rows64(CUtensorMap* m, const void* base, uint64_t L, uint64_t heads) {
  return make_map_head_rows64_pitch(m, base, L, heads, L);
}

cudaError_t launch_scan_tc(const Geom& g, const void* v, const float* logf, char* ws,
                           const FwdWs& lay, void* o, float* lse, void* zstore, cudaStream_t st) {
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
  p.Lk = g.Lp;
  p.nkc = 0;
  p.scl = g.scale * kLog2e;
  p.dm = (float*)(ws + lay.dm);
  p.dl = (float*)(ws + lay.dl);
  p.dacc = (float*)(ws + lay.dacc);
  p.fa = (const float*)(ws + lay.fa);
  p.fr = (const float*)(ws + lay.fr);
  p.ft = (const float*)(ws + lay.ft);
  p.o = (__nv_bfloat16*)o;
  p.lse = lse;
  p.zs = (uint8_t*)zstore;
  p.err = (int*)(ws + lay.err);
  const size_t smem = scan_smem_bytes(p.zs != nullptr);  // the attribute below is the maximum of both
  auto kern = logf ? fwd_scan_tc_kernel<true, false> : fwd_scan_tc_kernel<false, false>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem_bytes(true));
  if (e != cudaSuccess) return e;
  const long ntiles = (long)p.ntiles * g.BH;
  kern<<<(unsigned)ntiles, NTHREADS, smem, st>>>(m_ql, m_kr, m_f, m_v, p);
  return cudaGetLastError();
}

cudaError_t launch_scan_block(const Geom& g, int Lb, const void* zq, const void* kb, const void* vb,
                              const float* aq, const float* bk, char* ws, const FwdWs& lay, cudaStream_t st) {
  if (g.B != BK || g.Lp != g.L || (g.L % BQ) || Lb <= 0 || (Lb % BK) || ((aq == nullptr) != (bk == nullptr)))
    return cudaErrorInvalidValue;
  CUtensorMap m_ql, m_kr, m_f, m_v;
  if (!make_map_rows64(&m_ql, zq, (uint64_t)g.BH * g.Lp, BQ) || !make_map_rows64(&m_kr, kb, (uint64_t)g.BH * Lb, BK) ||
      !make_map_rows64(&m_f, kb, (uint64_t)g.BH * Lb, BK) ||  // not read in block mode
      !make_map_rows64(&m_v, vb, (uint64_t)g.BH * Lb, BK))
    return cudaErrorInvalidValue;
  ScanParams p{};
  p.L = g.L;
  p.Lp = g.Lp;
  p.nc = g.nc;
  p.BH = g.BH;
  p.ntiles = g.Lp / BQ;
  p.Lk = Lb;
  p.nkc = Lb / BK;
  p.scl = g.scale * kLog2e;
  p.dm = (float*)(ws + lay.dm);
  p.dl = (float*)(ws + lay.dl);
  p.dacc = (float*)(ws + lay.dacc);
  p.fa = aq;
  p.fr = bk;
  p.err = (int*)(ws + lay.err);
  const size_t smem = scan_smem_bytes(p.zs != nullptr);  // the attribute below is the maximum of both
  auto kern = aq ? fwd_scan_tc_kernel<true, true> : fwd_scan_tc_kernel<false, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)scan_smem_bytes(true));
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)((long)p.ntiles * g.BH), NTHREADS, smem, st>>>(m_ql, m_kr, m_f, m_v, p);
  return cudaGetLastError();
}

}  // namespace pathattn
