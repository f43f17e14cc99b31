// CUDA-core backward of PaTH attention: plain fp32 loops for fp32 inputs; for bf16 inputs (head
// dim 128, and chunk 32 at head dim 64) the same kernels run their small products as TF32 warp
// MMAs (smem_mm.cuh) with fp32 accumulation.
//
// The pages give no backward; this is the exact derivative of the blockwise forward of the
// PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.6–§2.7.  With Z_{b,c} the query chunk b
// transported to the right edge of key chunk c (Z_{b,b-1} = Q<-_b, Z_{b,c-1} = Z_{b,c} F_c^T):
//   dV_c  += P^T dO_b,   dK->_c += scale dS^T Z_{b,c},
//   G_{b,c} = scale dS K->_c + G_{b,c-1} F_c  (ascending c, G_{b,-1} = 0),
//   dF_c  += G_{b,c-1}^T Z_{b,c},   dQ<-_b = G_{b,b-1},
// followed per chunk by the chain rule through the diagonal-chunk logits and the UT quantities
// (Q<-, K->, F, X = U strictLower(W K^T), U = (I + strictLower(D W W^T))^{-1} D).
// PaTH-FoX (§2.5): the logit of (i, j) gains A_i - A_j (A = prefix sums of log f, formed over the
// whole sequence by fox_bwd.cu); both scans add colsum_m - rowsum_m of the logit gradient
// dS' = P (dP - D) into fxcs, from which fox_bwd.cu forms dlog f.
#include "internal.h"
#include "dev_common.cuh"
#include "smem_mm.cuh"
#include "tc_common.cuh"

#include <type_traits>

namespace pathattn {
namespace {

constexpr int NT = 256;
constexpr int NTM = 512;  // threads of the backward scan (one CTA per SM: 16 warps hide the latencies)
// D (template parameter): head dim, 64 or 128; DS is the padded shared-memory row stride (D + 1,
// or D + 4 for the backward scan's TF32 products: see BwdMainSmem).

// D_i = dO_i . o_i; padded rows get 0.  A row is read by a group of D / VEC lanes with 16-byte
// loads (VEC elements each), a warp covers DOT_PASSES row groups with all loads issued before the
// products, so that every thread keeps DOT_PASSES * 32 bytes in flight (the kernel is bound by
// HBM reads of o and dO).
constexpr int DOT_PASSES = 2;
template <typename T>
__device__ __forceinline__ float dot16(const uint4& a, const uint4& b) {
  if constexpr (std::is_same<T, float>::value) {
    return __uint_as_float(a.x) * __uint_as_float(b.x) + __uint_as_float(a.y) * __uint_as_float(b.y) +
           __uint_as_float(a.z) * __uint_as_float(b.z) + __uint_as_float(a.w) * __uint_as_float(b.w);
  } else {
    const __nv_bfloat162* x = reinterpret_cast<const __nv_bfloat162*>(&a);
    const __nv_bfloat162* y = reinterpret_cast<const __nv_bfloat162*>(&b);
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 u = __bfloat1622float2(x[j]), v = __bfloat1622float2(y[j]);
      acc = fmaf(u.x, v.x, acc);
      acc = fmaf(u.y, v.y, acc);
    }
    return acc;
  }
}
template <typename T, int D>
__global__ void __launch_bounds__(NT) bwd_dot_kernel(Geom g, const T* __restrict__ o,
                                                     const T* __restrict__ dO, float* __restrict__ Dv) {
  constexpr int VEC = 16 / (int)sizeof(T);
  constexpr int LPR = D / VEC;   // lanes per row
  constexpr int RPW = 32 / LPR;  // rows per warp and pass
  const long warp = ((long)blockIdx.x * NT + threadIdx.x) / 32;
  const int lane = threadIdx.x % 32, sub = lane / LPR, l = lane % LPR;
  const long rows = (long)g.BH * g.Lp;
  const long row0 = warp * (RPW * DOT_PASSES) + sub;
  uint4 a[DOT_PASSES], b[DOT_PASSES];
  bool ok[DOT_PASSES];
#pragma unroll
  for (int k = 0; k < DOT_PASSES; ++k) {
    const long row = row0 + (long)k * RPW;
    const int bh = (int)(row / g.Lp), i = (int)(row % g.Lp);
    ok[k] = row < rows && i < g.L;
    a[k] = b[k] = make_uint4(0u, 0u, 0u, 0u);
    if (ok[k]) {
      const size_t off = ((size_t)bh * g.L + i) * D + (size_t)l * VEC;
      a[k] = __ldg(reinterpret_cast<const uint4*>(o + off));
      b[k] = __ldg(reinterpret_cast<const uint4*>(dO + off));
    }
  }
#pragma unroll
  for (int k = 0; k < DOT_PASSES; ++k) {
    const long row = row0 + (long)k * RPW;
    const float acc = group_sum<LPR>(ok[k] ? dot16<T>(a[k], b[k]) : 0.f);
    if (l == 0 && row < rows) Dv[row] = acc;
  }
}
template <typename T, int D>
unsigned dot_blocks(const Geom& g) {
  constexpr int rows_per_block = (NT / 32) * (32 / (D / (16 / (int)sizeof(T)))) * DOT_PASSES;
  const long rows = (long)g.BH * g.Lp;
  return (unsigned)((rows + rows_per_block - 1) / rows_per_block);
}

// Row strides padded for the products' operand reads: + 4 floats (stride = 4 mod 32 banks) for
// the TF32 warp MMAs, whose fragment loads then hit 32 distinct banks in either operand
// orientation; + 1 for the plain fp32 loops, whose threads walk a row or a column.
// K, V, dO and G are adjacent: the Z-chain pass, in which all four are dead, holds its second F
// buffer there.  With the TF32 padding every buffer starts on a 16-byte boundary and every row
// is 16-byte aligned, so the fp32 operands arrive by asynchronous 16-byte copies.
template <int B, int D, bool TC>
struct BwdMainSmem {
  static constexpr int PAD = TC ? 4 : 1;
  static constexpr int DS = D + PAD;
  static constexpr int BS = B + PAD;
  static constexpr int kZ = 0, kF = kZ + B * DS, kK = kF + D * DS, kV = kK + B * DS;
  static constexpr int kdO = kV + B * DS, kG = kdO + B * DS, kGn = kG + B * DS;
  static constexpr int kP = kGn + B * DS, kdS = kP + B * BS, kLse = kdS + B * BS, kDv = kLse + B;
  static constexpr int kAk = kDv + B;  // PaTH-FoX: A_j log2(e) of the key chunk
  static constexpr int total = kAk + B;
  static constexpr size_t bytes = (size_t)total * 4;
  static_assert(D * DS <= kGn - kK, "the second F buffer fits over K, V, dO and G");
  static_assert(!TC || (DS % 4 == 0 && BS % 4 == 0), "16-byte aligned rows");
};

// A 16-byte global -> shared copy that bypasses the registers; cp_async_wait_all() waits for the
// calling thread's copies (a barrier then publishes them to the block).
__device__ __forceinline__ void cp_async16(float* sdst, const float* gsrc) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(tc::smem_u32(sdst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// `rows` fp32 rows of D (global row stride D) into shared rows of stride DS: asynchronous 16-byte
// copies (ASYNC, 16-byte aligned rows) or plain loads and stores.
template <int D, int DS, bool ASYNC>
__device__ __forceinline__ void load_rows(float* dst, const float* src, int rows, int tid) {
  if constexpr (ASYNC) {
    constexpr int Q = D / 4;
    for (int idx = tid; idx < rows * Q; idx += NTM) {
      const int r = idx / Q, q = idx % Q;
      cp_async16(dst + r * DS + 4 * q, src + (size_t)r * D + 4 * q);
    }
  } else {
    for (int idx = tid; idx < rows * D; idx += NTM) dst[(idx / D) * DS + idx % D] = src[idx];
  }
}

// Persistent CTAs; tile n (heaviest first) is query chunk b = nc-1 - n/BH of head n%BH.
template <typename T, int B, bool FOX, int D>
__global__ void __launch_bounds__(NTM, 1) bwd_main_simt_kernel(
    Geom g, const T* __restrict__ v, const float* __restrict__ lse, const T* __restrict__ dO,
    const float* __restrict__ Dv, const float* __restrict__ ql, const float* __restrict__ kr,
    const float* __restrict__ f, float* __restrict__ dql, float* __restrict__ dkr,
    float* __restrict__ dvacc, float* __restrict__ dfacc, float* __restrict__ zs,
    const float* __restrict__ fxa, float* __restrict__ fxcs) {
  extern __shared__ float sm[];
  // bf16 inputs: the products run as TF32 warp MMAs (fp32 accumulation); fp32 inputs: plain fp32
  constexpr bool TC = std::is_same<T, __nv_bfloat16>::value;
  using S = BwdMainSmem<B, D, TC>;
  constexpr int BS = S::BS, DS = S::DS;
  float* sZ = sm + S::kZ;
  float* sK = sm + S::kK;
  float* sV = sm + S::kV;
  float* sF = sm + S::kF;
  float* sdO = sm + S::kdO;
  float* sG = sm + S::kG;
  float* sGn = sm + S::kGn;
  float* sP = sm + S::kP;
  float* sdS = sm + S::kdS;
  float* sLse = sm + S::kLse;
  float* sDv = sm + S::kDv;
  float* sAk = sm + S::kAk;

  const int tid = threadIdx.x;
  float* myz = zs + (size_t)blockIdx.x * g.Lp * D;
  const long ntiles = (long)g.BH * g.nc;
  const float scl2 = g.scale * kLog2e;

  for (long n = blockIdx.x; n < ntiles; n += gridDim.x) {
    const int b = g.nc - 1 - (int)(n / g.BH);
    const int bh = (int)(n % g.BH);
    const size_t brow = (size_t)bh * g.Lp + (size_t)b * B;
    if (b == 0) {
      for (int idx = tid; idx < B * D; idx += NTM) dql[brow * D + idx] = 0.f;
      continue;
    }
    // ---- pass 1: Z_{b,c} for c = b-1 .. 0, stored in this CTA's scratch slab; F_{c-1} arrives
    // during the product with F_c (two F buffers), the two Z buffers alternate ----
    {
      float* za = sm + S::kZ;   // Z_{b,c}
      float* zb = sm + S::kGn;  // Z_{b,c-1}
      float* fa = sm + S::kF;  // F_c
      float* fn = sm + S::kK;  // F_{c-1}
      load_rows<D, DS, TC>(za, ql + brow * D, B, tid);
      if (b >= 2) load_rows<D, DS, TC>(fa, f + ((size_t)bh * g.nc + (b - 1)) * D * D, D, tid);
      if constexpr (TC) cp_async_wait_all();
      __syncthreads();
      for (int c = b - 1; c >= 0; --c) {
        for (int idx = tid; idx < B * D; idx += NTM) myz[(size_t)c * B * D + idx] = za[(idx / D) * DS + idx % D];
        if (c == 0) break;
        if (c >= 2) load_rows<D, DS, TC>(fn, f + ((size_t)bh * g.nc + (c - 1)) * D * D, D, tid);
        smem_mm<B, D, D, false, true, TC>(za, DS, fa, DS, [&](int i, int nn, float x) { zb[i * DS + nn] = x; });
        if constexpr (TC) cp_async_wait_all();
        __syncthreads();
        float* t = za;
        za = zb;
        zb = t;
        t = fa;
        fa = fn;
        fn = t;
      }
      __syncthreads();  // the last Z has been stored before its buffer (possibly G's) is reused
    }
    // ---- pass 2: ascending adjoint scan ----
    for (int idx = tid; idx < B * D; idx += NTM) {
      const int i = idx / D, cc = idx % D, gi = b * B + i;
      sdO[i * DS + cc] = gi < g.L ? to_f(dO[((size_t)bh * g.L + gi) * D + cc]) : 0.f;
      sG[i * DS + cc] = 0.f;
    }
    for (int i = tid; i < B; i += NTM) {
      const int gi = b * B + i;
      float l2 = gi < g.L ? lse[(size_t)bh * g.L + gi] * kLog2e : INFINITY;  // padded rows: P = 0
      if constexpr (FOX) l2 = fmaf(-fxa[brow + i], kLog2e, l2);                 // the + A_i of the bias
      sLse[i] = l2;
      sDv[i] = Dv[brow + i];
    }
    float fox_rowsum = 0.f;  // PaTH-FoX: row tid's sum of dS' over the off-diagonal key chunks
    __syncthreads();  // also orders pass-1 scratch writes before the reads below
    // F_c (read by step c > 0 only) is fetched during step c - 1, once that step's G product has
    // read F_{c-1}; Z_c and K_c are fetched at the step's start (their buffers serve until the
    // previous step's end)
    for (int c = 0; c < b; ++c) {
      const size_t crow = (size_t)bh * g.Lp + (size_t)c * B;
      const size_t vrow = (size_t)bh * g.L + (size_t)c * B;  // rows of chunk c < b are all < L
      load_rows<D, DS, TC>(sZ, myz + (size_t)c * B * D, B, tid);
      load_rows<D, DS, TC>(sK, kr + crow * D, B, tid);
      if constexpr (TC) {  // bf16 V: 8 values per 16-byte load (tensor pointers are 16-byte aligned)
        for (int idx = tid; idx < B * D / 8; idx += NTM) {
          const int r = idx / (D / 8), q = idx % (D / 8);
          const uint4 u = *reinterpret_cast<const uint4*>(v + (vrow + r) * D + 8 * q);
          const __nv_bfloat162* h2 = reinterpret_cast<const __nv_bfloat162*>(&u);
          const float2 a0 = __bfloat1622float2(h2[0]), a1 = __bfloat1622float2(h2[1]);
          const float2 a2 = __bfloat1622float2(h2[2]), a3 = __bfloat1622float2(h2[3]);
          float4* dst = reinterpret_cast<float4*>(sV + r * DS + 8 * q);
          dst[0] = make_float4(a0.x, a0.y, a1.x, a1.y);
          dst[1] = make_float4(a2.x, a2.y, a3.x, a3.y);
        }
      } else {
        for (int idx = tid; idx < B * D; idx += NTM) sV[(idx / D) * DS + idx % D] = to_f(v[vrow * D + idx]);
      }
      if constexpr (FOX)
        for (int j = tid; j < B; j += NTM) sAk[j] = fxa[crow + j] * kLog2e;
      if constexpr (TC) cp_async_wait_all();
      __syncthreads();
      // P and dS (the two products share their output mapping: the thread that writes P(i, j)
      // reads it back)
      smem_mm<B, B, D, false, true, TC>(sZ, DS, sK, DS, [&](int i, int j, float x) {
        sP[i * BS + j] = fast_exp2(x * scl2 - sLse[i] - (FOX ? sAk[j] : 0.f));
      });
      smem_mm<B, B, D, false, true, TC>(sdO, DS, sV, DS, [&](int i, int j, float x) {
        sdS[i * BS + j] = sP[i * BS + j] * (x - sDv[i]);
      });
      __syncthreads();
      if constexpr (FOX) {  // dS' row sums kept per thread; column sums of key chunk c into fxcs
        if (tid < B) {
          for (int j = 0; j < B; ++j) fox_rowsum += sdS[tid * BS + j];
        } else if (tid < 2 * B) {
          const int j = tid - B;
          float cs = 0.f;
          for (int i = 0; i < B; ++i) cs += sdS[i * BS + j];
          atomicAdd(fxcs + crow + j, cs);
        }
      }
      // G_new = scale dS K + G F_c first (the last read of K), then dV_c += P^T dO and
      // dK->_c += scale dS^T Z into the dead K and V buffers as dense 32 x D fp32 blocks, added to
      // the accumulators by one bulk reduction each (contiguous rows of chunk c), and dF_c +=
      // G_{b,c-1}^T Z_{b,c} in 32-row pieces through the same two buffers.  One thread issues the
      // reductions; it waits for a buffer's previous reduction to have read it before the buffer
      // is written again.
      smem_mm<B, D, B, false, false, TC>(sdS, BS, sK, DS, [&](int i, int nn, float x) { sGn[i * DS + nn] = g.scale * x; });
      if (c > 0)
        smem_mm<B, D, D, false, false, TC>(sG, DS, sF, DS, [&](int i, int nn, float x) { sGn[i * DS + nn] += x; });
      __syncthreads();  // K, V and F are dead
      if (c + 1 < b) load_rows<D, DS, TC>(sF, f + ((size_t)bh * g.nc + c + 1) * D * D, D, tid);
      smem_mm<B, D, B, true, false, TC>(sP, BS, sdO, DS, [&](int j, int cc, float x) { sV[j * D + cc] = x; });
      smem_mm<B, D, B, true, false, TC>(sdS, BS, sZ, DS, [&](int j, int cc, float x) { sK[j * D + cc] = g.scale * x; });
      tc::fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0) {
        tc::bulk_reduce_add_f32(dvacc + crow * D, sV, B * D * 4);
        tc::bulk_reduce_add_f32(dkr + crow * D, sK, B * D * 4);
        tc::bulk_commit();
      }
      if (c > 0) {  // dF_c += G_{b,c-1}^T Z_{b,c}, rows 32 q .. 32 q + 31 per piece
        float* dfc = dfacc + ((size_t)bh * g.nc + c) * D * D;
        for (int q = 0; q < D / 32; ++q) {
          float* buf = (q & 1) ? sK : sV;
          if (tid == 0) tc::bulk_wait_read0();  // every earlier reduction has read its buffer
          __syncthreads();
          smem_mm<32, D, B, true, false, TC>(sG + 32 * q, DS, sZ, DS, [&](int r, int cc, float x) { buf[r * D + cc] = x; });
          tc::fence_proxy_async_smem();
          __syncthreads();
          if (tid == 0) {
            tc::bulk_reduce_add_f32(dfc + (size_t)32 * q * D, buf, 32 * D * 4);
            tc::bulk_commit();
          }
        }
      }
      if (tid == 0) tc::bulk_wait_read0();  // K and V are reloaded next step
      __syncthreads();
      float* t = sG; sG = sGn; sGn = t;
    }
    for (int idx = tid; idx < B * D; idx += NTM) dql[brow * D + idx] = sG[(idx / D) * DS + idx % D];
    if (FOX && tid < B) atomicAdd(fxcs + brow + tid, -fox_rowsum);
    __syncthreads();
  }
  if (tid == 0) tc::bulk_wait0();  // the reductions are complete before the CTA exits
}

template <int B, int D>
struct PrepBwdSmem {
  static constexpr int DS = D + 1;
  static constexpr int BS = B + 1;
  static constexpr int nBD = 8, nBB = 11;
  static constexpr int kBD = 0, kBB = kBD + nBD * B * DS;
  static constexpr int kVec = kBB + nBB * B * BS;
  static constexpr int total = kVec + 7 * B;  // beta, lse, D, dbeta; PaTH-FoX: A, dS' row / column sums
  static constexpr size_t bytes = (size_t)total * 4;
};

// One CTA per (chunk c, head bh): diagonal-chunk attention backward and the chain rule through
// Q<- = Q - lower(QW^T) U W, K-> = K - X^T W, F = I - W^T U^T W, X = U strictLower(W K^T),
// S_d = lower(QK^T) - lower(QW^T) X, U = Y D with Y = (I + strictLower(D W W^T))^{-1}.
template <typename T, int B, bool FOX, int D>
__global__ void __launch_bounds__(NT) prep_bwd_simt_kernel(
    Geom g, const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const T* __restrict__ w, const float* __restrict__ beta, const float* __restrict__ lse,
    const T* __restrict__ dO, const float* __restrict__ Dv, const float* __restrict__ dql,
    const float* __restrict__ dkr, const float* __restrict__ dvacc, const float* __restrict__ dfacc,
    T* __restrict__ dq, T* __restrict__ dk, T* __restrict__ dv, T* __restrict__ dw,
    float* __restrict__ dbeta, const float* __restrict__ fxa, float* __restrict__ fxcs) {
  extern __shared__ float sm[];
  using S = PrepBwdSmem<B, D>;
  constexpr int BS = S::BS, DS = S::DS;
  float* bd = sm + S::kBD;
  float* sW = bd + 0 * B * DS;
  float* sQ = bd + 1 * B * DS;
  float* sK = bd + 2 * B * DS;
  float* sV = bd + 3 * B * DS;    // V, then Y1 = U W (step 4), then diag(beta) W (step 10)
  float* sdO = bd + 4 * B * DS;   // dO, then E3 = M1^T dQ<- + W dF^T (step 7a)
  float* sgQ = bd + 5 * B * DS;
  float* sgK = bd + 6 * B * DS;
  float* sgW = bd + 7 * B * DS;
  float* sY1 = sV;
  float* sE3 = sdO;
  float* bb = sm + S::kBB;
  float* sY = bb + 0 * B * BS;    // T^{-1}
  float* sU = bb + 1 * B * BS;
  float* sM1 = bb + 2 * B * BS;
  float* sN2 = bb + 3 * B * BS;
  float* sX = bb + 4 * B * BS;
  float* sG = bb + 5 * B * BS;
  float* sdS = bb + 6 * B * BS;
  float* sgU = bb + 7 * B * BS;
  float* sgX = bb + 8 * B * BS;   // later gN = strictLower(gT)
  float* sT1 = bb + 9 * B * BS;   // QK^T -> P -> gN2
  float* sT2 = bb + 10 * B * BS;  // dP -> gM1 -> gY Y^T
  float* sBeta = sm + S::kVec;
  float* sLse = sBeta + B;
  float* sDv = sLse + B;
  float* sgB = sDv + B;
  float* sFa = sgB + B;  // PaTH-FoX: A_i log2(e)
  float* sFr = sFa + B;  // PaTH-FoX: row sums of dS'
  float* sFc = sFr + B;  // PaTH-FoX: column sums of dS'

  const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int row0 = c * B;
  const size_t in_row = (size_t)bh * g.L;
  const size_t ws_row = (size_t)bh * g.Lp + row0;
  const float scl2 = g.scale * kLog2e;

  // 1. loads
  for (int idx = tid; idx < B * D; idx += NT) {
    const int r = idx / D, cc = idx % D, gi = row0 + r;
    const bool ok = gi < g.L;
    const size_t off = (in_row + gi) * D + cc;
    sW[r * DS + cc] = ok ? to_f(w[off]) : 0.f;
    sQ[r * DS + cc] = ok ? to_f(q[off]) : 0.f;
    sK[r * DS + cc] = ok ? to_f(k[off]) : 0.f;
    sV[r * DS + cc] = ok ? to_f(v[off]) : 0.f;
    sdO[r * DS + cc] = ok ? to_f(dO[off]) : 0.f;
  }
  // dQ<-, dK-> rows and dF of this chunk are read in place (global, row stride D)
  const float* gdQl = dql + ws_row * D;
  const float* gdKr = dkr + ws_row * D;
  const float* gdF = dfacc + ((size_t)bh * g.nc + c) * D * D;
  for (int r = tid; r < B; r += NT) {
    const int gi = row0 + r;
    const bool ok = gi < g.L;
    sBeta[r] = ok ? clamp_beta(beta[in_row + gi]) : 0.f;
    sLse[r] = ok ? lse[in_row + gi] * kLog2e : INFINITY;
    sDv[r] = Dv[ws_row + r];
    sgB[r] = 0.f;
    if constexpr (FOX) {
      sFa[r] = fxa[ws_row + r] * kLog2e;
      sFr[r] = sFc[r] = 0.f;
    }
  }
  __syncthreads();

  // bf16 inputs: products on TF32 tensor cores; fp32 inputs: exact fp32 loops
  constexpr bool TC = std::is_same<T, __nv_bfloat16>::value;
  // P2. G = strictLower(WW^T), M1 = lower(QW^T), N2 = strictLower(WK^T), QK^T (sT1), dP = dO V^T (sT2)
  smem_mm<B, B, D, false, true, TC>(sW, DS, sW, DS, [&](int i, int j, float x) { sG[i * BS + j] = j < i ? x : 0.f; });
  smem_mm<B, B, D, false, true, TC>(sQ, DS, sW, DS, [&](int i, int j, float x) { sM1[i * BS + j] = j <= i ? x : 0.f; });
  smem_mm<B, B, D, false, true, TC>(sW, DS, sK, DS, [&](int i, int j, float x) { sN2[i * BS + j] = j < i ? x : 0.f; });
  smem_mm<B, B, D, false, true, TC>(sQ, DS, sK, DS, [&](int i, int j, float x) { sT1[i * BS + j] = x; });
  smem_mm<B, B, D, false, true, TC>(sdO, DS, sV, DS, [&](int i, int j, float x) { sT2[i * BS + j] = x; });
  __syncthreads();

  // P3. Y = T^{-1} by forward substitution: Y_i = e_i - beta_i sum_{m<i} G_im Y_m ; U = Y diag(beta)
  if constexpr (B == 32) {
    // one warp, lane = column: the column of Y lives in registers
    if (tid < 32) {
      const int cc = tid;
      float y[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m + 1 < i; m += 2) {
          a0 += sG[i * BS + m] * y[m];
          a1 += sG[i * BS + m + 1] * y[m + 1];
        }
        if (i & 1) a0 += sG[i * BS + i - 1] * y[i - 1];
        y[i] = (cc == i ? 1.f : 0.f) - sBeta[i] * (a0 + a1);
      }
      const float bc = sBeta[cc];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        sY[i * BS + cc] = y[i];
        sU[i * BS + cc] = y[i] * bc;
      }
    }
  } else {
    for (int i = 0; i < B; ++i) {
      if (tid < B) {
        const int cc = tid;
        float val = 0.f;
        if (cc <= i) {
          float acc = 0.f;
          for (int m = cc; m < i; ++m) acc += sG[i * BS + m] * sY[m * BS + cc];
          val = (cc == i ? 1.f : 0.f) - sBeta[i] * acc;
        }
        sY[i * BS + cc] = val;
      }
      __syncthreads();
    }
    for (int idx = tid; idx < B * B; idx += NT) {
      const int i = idx / B, j = idx % B;
      sU[i * BS + j] = sY[i * BS + j] * sBeta[j];
    }
  }
  __syncthreads();

  // P4. X = U N2 ; Y1 = U W (into V's slot) ; E3 = M1^T dQ<- + W dF^T (into dO's slot needs dO
  //     until P6, so E3 waits); then the diagonal logits and, in the same epilogue, P and dS
  smem_mm<B, B, B, false, false, TC>(sU, BS, sN2, BS, [&](int i, int j, float x) { sX[i * BS + j] = x; });
  smem_mm<B, D, B, false, false, TC>(sU, BS, sW, DS, [&](int i, int cc, float x) { sY1[i * DS + cc] = x; });
  __syncthreads();

  // P5. S_d = QK^T - M1 X ; P = exp(scale S_d (+ A_i - A_j) - lse) on j <= i ; dS = scale P (dP - D)
  smem_mm<B, B, B, false, false, TC>(sM1, BS, sX, BS, [&](int i, int j, float x) {
    float p = 0.f;
    const bool live = j <= i && row0 + i < g.L;
    if (live) p = fast_exp2((sT1[i * BS + j] - x) * scl2 - sLse[i] + (FOX ? sFa[i] - sFa[j] : 0.f));
    const float ds = p * (sT2[i * BS + j] - sDv[i]);
    sT1[i * BS + j] = p;
    sdS[i * BS + j] = g.scale * ds;
    if (FOX && live) {
      atomicAdd(&sFr[i], ds);
      atomicAdd(&sFc[j], ds);
    }
  });
  __syncthreads();
  if constexpr (FOX)
    for (int r = tid; r < B; r += NT) atomicAdd(fxcs + ws_row + r, sFc[r] - sFr[r]);

  // P6. dv (final) = dV acc + P^T dO ; gQ = dQ<- + dS K ; gK = dK-> + dS^T Q ;
  //     gM1 = lower(-dS X^T - dQ<- Y1^T) (sT2) ; gX = -M1^T dS - W dK->^T
  smem_mm<B, D, B, true, false, TC>(sT1, BS, sdO, DS, [&](int r, int cc, float x) {
    if (row0 + r < g.L) dv[(in_row + row0 + r) * D + cc] = from_f<T>(dvacc[(ws_row + r) * D + cc] + x);
  });
  smem_mm<B, D, B, false, false, TC>(sdS, BS, sK, DS, [&](int r, int cc, float x) { sgQ[r * DS + cc] = gdQl[r * D + cc] + x; });
  smem_mm<B, D, B, true, false, TC>(sdS, BS, sQ, DS, [&](int r, int cc, float x) { sgK[r * DS + cc] = gdKr[r * D + cc] + x; });
  smem_mm<B, B, B, false, true, TC>(sdS, BS, sX, BS, [&](int i, int m, float x) { sT2[i * BS + m] = -x; });
  smem_mm<B, B, B, true, false, TC>(sM1, BS, sdS, BS, [&](int i, int m, float x) { sgX[i * BS + m] = -x; });
  smem_mm<B, B, D, false, true, TC>(gdQl, D, sY1, DS, [&](int i, int m, float x) {
    sT2[i * BS + m] = m <= i ? sT2[i * BS + m] - x : 0.f;
  });
  smem_mm<B, B, D, false, true, TC>(sW, DS, gdKr, D, [&](int i, int m, float x) { sgX[i * BS + m] -= x; });
  __syncthreads();

  // P7. E3 = M1^T dQ<- + W dF^T (into dO's slot, free now); gN2 = strictLower(U^T gX) (sT1, P free)
  smem_mm<B, D, B, true, false, TC>(sM1, BS, gdQl, D, [&](int m, int cc, float x) { sE3[m * DS + cc] = x; });
  smem_mm<B, D, D, false, true, TC>(sW, DS, gdF, D, [&](int m, int cc, float x) { sE3[m * DS + cc] += x; });
  smem_mm<B, B, B, true, false, TC>(sU, BS, sgX, BS, [&](int i, int j, float x) { sT1[i * BS + j] = j < i ? x : 0.f; });
  // gW = -X dK-> - Y1 dF + gM1^T Q (the -U^T E3 term follows in P8) ; gQ += gM1 W
  smem_mm<B, D, B, false, false, TC>(sX, BS, gdKr, D, [&](int r, int cc, float x) { sgW[r * DS + cc] = -x; });
  smem_mm<B, D, D, false, false, TC>(sY1, DS, gdF, D, [&](int r, int cc, float x) { sgW[r * DS + cc] -= x; });
  smem_mm<B, D, B, true, false, TC>(sT2, BS, sQ, DS, [&](int r, int cc, float x) { sgW[r * DS + cc] += x; });
  smem_mm<B, D, B, false, false, TC>(sT2, BS, sW, DS, [&](int r, int cc, float x) { sgQ[r * DS + cc] += x; });
  __syncthreads();

  // P8. gU = lower(-E3 W^T + gX N2^T); gW -= U^T E3; gW += gN2 K; gK += gN2^T W
  smem_mm<B, B, D, false, true, TC>(sE3, DS, sW, DS, [&](int i, int j, float x) { sgU[i * BS + j] = -x; });
  smem_mm<B, B, B, false, true, TC>(sgX, BS, sN2, BS, [&](int i, int j, float x) {
    sgU[i * BS + j] = j <= i ? sgU[i * BS + j] + x : 0.f;
  });
  smem_mm<B, D, B, true, false, TC>(sU, BS, sE3, DS, [&](int r, int cc, float x) { sgW[r * DS + cc] -= x; });
  smem_mm<B, D, B, false, false, TC>(sT1, BS, sK, DS, [&](int r, int cc, float x) { sgW[r * DS + cc] += x; });
  smem_mm<B, D, B, true, false, TC>(sT1, BS, sW, DS, [&](int r, int cc, float x) { sgK[r * DS + cc] += x; });
  __syncthreads();

  // P9. dbeta_j += sum_i gU_ij Y_ij ; A1 = gY Y^T = gU diag(beta) Y^T = gU U^T (into sT2)
  if (tid < B) {
    float a = 0.f;
    for (int i = tid; i < B; ++i) a += sgU[i * BS + tid] * sY[i * BS + tid];
    sgB[tid] += a;
  }
  smem_mm<B, B, B, false, true, TC>(sgU, BS, sU, BS, [&](int i, int j, float x) { sT2[i * BS + j] = x; });
  // diag(beta) W into Y1's slot (free now)
  for (int idx = tid; idx < B * D; idx += NT) {
    const int r = idx / D, cc = idx % D;
    sY1[r * DS + cc] = sBeta[r] * sW[r * DS + cc];
  }
  __syncthreads();

  // P10. gN = strictLower(-Y^T A1) into sgX
  smem_mm<B, B, B, true, false, TC>(sY, BS, sT2, BS, [&](int i, int j, float x) { sgX[i * BS + j] = j < i ? -x : 0.f; });
  __syncthreads();

  // P11. N = strictLower(D G): dbeta_i += sum_{j<i} gN_ij G_ij ; gG = D gN ;
  //      gW += gG W + gG^T W = diag(beta) (gN W) + gN^T (diag(beta) W)
  if (tid < B) {
    float a = 0.f;
    for (int j = 0; j < tid; ++j) a += sgX[tid * BS + j] * sG[tid * BS + j];
    sgB[tid] += a;
  }
  smem_mm<B, D, B, false, false, TC>(sgX, BS, sW, DS, [&](int r, int cc, float x) { sgW[r * DS + cc] += sBeta[r] * x; });
  smem_mm<B, D, B, true, false, TC>(sgX, BS, sY1, DS, [&](int r, int cc, float x) { sgW[r * DS + cc] += x; });
  __syncthreads();

  // 12. outputs
  for (int idx = tid; idx < B * D; idx += NT) {
    const int r = idx / D, cc = idx % D, gi = row0 + r;
    if (gi < g.L) {
      const size_t off = (in_row + gi) * D + cc;
      dq[off] = from_f<T>(sgQ[r * DS + cc]);
      dk[off] = from_f<T>(sgK[r * DS + cc]);
      dw[off] = from_f<T>(sgW[r * DS + cc]);
    }
  }
  for (int r = tid; r < B; r += NT)
    if (row0 + r < g.L) dbeta[in_row + row0 + r] = sgB[r];
}

template <typename T, int B, int D>
cudaError_t bwd_t(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                  const float* beta, const void* o, const float* lse, const void* dO, void* dq,
                  void* dk, void* dv, void* dw, float* dbeta, char* ws, const BwdWs& lay,
                  int phases, cudaStream_t st, const float* logf, float* dlogf) {
  cudaError_t e;
  const size_t rows = (size_t)g.BH * g.Lp;
  float* fxa = (float*)(ws + lay.fxa);
  float* fxcs = (float*)(ws + lay.fxcs);
  if (phases & 1) {
  if (logf) {  // PaTH-FoX: prefix sums of log f, zeroed dS' sums
    if ((e = launch_fox_prefix(g, logf, fxa, st)) != cudaSuccess) return e;
    if ((e = cudaMemsetAsync(fxcs, 0, rows * 4, st)) != cudaSuccess) return e;
  }
  if ((e = cudaMemsetAsync(ws + lay.dkr, 0, rows * D * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(ws + lay.dv, 0, rows * D * 4, st)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(ws + lay.df, 0, (size_t)g.BH * g.nc * D * D * 4, st)) != cudaSuccess) return e;
  bwd_dot_kernel<T, D><<<dot_blocks<T, D>(g), NT, 0, st>>>(g, (const T*)o, (const T*)dO, (float*)(ws + lay.Dv));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  if ((e = launch_prep_simt(std::is_same<T, __nv_bfloat16>::value, g, q, k, v, w, beta, nullptr, ws,
                            lay.fw, false, st)) != cudaSuccess)
    return e;
  }
  if (phases & 2) {
    auto kern = logf ? bwd_main_simt_kernel<T, B, true, D> : bwd_main_simt_kernel<T, B, false, D>;
    const size_t smem = BwdMainSmem<B, D, std::is_same<T, __nv_bfloat16>::value>::bytes;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) return e;
    kern<<<lay.nctas, NTM, smem, st>>>(g, (const T*)v, lse, (const T*)dO, (const float*)(ws + lay.Dv),
                                      (const float*)(ws + lay.fw.ql), (const float*)(ws + lay.fw.kr),
                                      (const float*)(ws + lay.fw.f), (float*)(ws + lay.dql),
                                      (float*)(ws + lay.dkr), (float*)(ws + lay.dv), (float*)(ws + lay.df),
                                      (float*)(ws + lay.zs), fxa, fxcs);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (phases & 4) {
    auto kern = logf ? prep_bwd_simt_kernel<T, B, true, D> : prep_bwd_simt_kernel<T, B, false, D>;
    const size_t smem = PrepBwdSmem<B, D>::bytes;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess) return e;
    kern<<<dim3(g.nc, g.BH), NT, smem, st>>>(
        g, (const T*)q, (const T*)k, (const T*)v, (const T*)w, beta, lse, (const T*)dO,
        (const float*)(ws + lay.Dv), (const float*)(ws + lay.dql), (const float*)(ws + lay.dkr),
        (const float*)(ws + lay.dv), (const float*)(ws + lay.df), (T*)dq, (T*)dk, (T*)dv, (T*)dw, dbeta,
        fxa, fxcs);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
    if (dlogf && (e = launch_fox_dlogf(g, fxcs, dlogf, st)) != cudaSuccess) return e;
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_bwd_dot(const Geom& g, const void* o, const void* dO, float* Dv, cudaStream_t st) {
  bwd_dot_kernel<__nv_bfloat16, kHeadDim><<<dot_blocks<__nv_bfloat16, kHeadDim>(g), NT, 0, st>>>(
      g, (const __nv_bfloat16*)o, (const __nv_bfloat16*)dO, Dv);
  return cudaGetLastError();
}

cudaError_t launch_bwd_simt(bool is_bf16, const Geom& g, const void* q, const void* k,
                            const void* v, const void* w, const float* beta, const void* o,
                            const float* lse, const void* dO, void* dq, void* dk, void* dv,
                            void* dw, float* dbeta, char* ws, const BwdWs& lay, int phases,
                            cudaStream_t st, const float* logf, float* dlogf) {
  if (g.B != 32 || (dlogf && !logf)) return cudaErrorInvalidValue;
  if (g.D == kHeadDimWide)
    return is_bf16 ? bwd_t<__nv_bfloat16, 32, kHeadDimWide>(g, q, k, v, w, beta, o, lse, dO, dq, dk, dv, dw, dbeta, ws,
                                                            lay, phases, st, logf, dlogf)
                   : bwd_t<float, 32, kHeadDimWide>(g, q, k, v, w, beta, o, lse, dO, dq, dk, dv, dw, dbeta, ws, lay,
                                                    phases, st, logf, dlogf);
  if (g.D != kHeadDim) return cudaErrorInvalidValue;
  return is_bf16 ? bwd_t<__nv_bfloat16, 32, kHeadDim>(g, q, k, v, w, beta, o, lse, dO, dq, dk, dv, dw, dbeta, ws, lay,
                                                      phases, st, logf, dlogf)
                 : bwd_t<float, 32, kHeadDim>(g, q, k, v, w, beta, o, lse, dO, dq, dk, dv, dw, dbeta, ws, lay, phases,
                                              st, logf, dlogf);
}

}  // namespace pathattn
