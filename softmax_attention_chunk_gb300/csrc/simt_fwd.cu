// SIMT (fp32 CUDA-core) forward of PaTH attention: per-chunk UT preparation and the
// right-to-left chunk scan.  Used for the fp32 mode and as the correctness path.
//
// Method: PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.6 (UT representation,
// full-matrix logits) and §2.7 (boundary-adjusted Q/K, chunk transforms, right-to-left scan).
#include "internal.h"
#include "dev_common.cuh"
#include "smem_mm.cuh"

#include <type_traits>

namespace pathattn {
namespace {

constexpr int NT = 256;

// D: head dim (64 or 128); DS = D + 1 is the padded smem row stride of [rows][D] matrices.
template <int B, int D>
struct PrepSmem {
  static constexpr int DS = D + 1;
  static constexpr int BS = B + 1;
  static constexpr int kW = 0, kQ = kW + B * DS, kK = kQ + B * DS, kV = kK + B * DS;
  static constexpr int kU = kV + B * DS, kM1 = kU + B * BS, kX = kM1 + B * BS, kT = kX + B * BS;
  static constexpr int kR = kT + B * BS;
  static constexpr int kG = kR + B * DS, kN2 = kG + B * BS, kAM = kN2 + B * BS;
  static constexpr int kBeta = kAM + B * BS, kLf = kBeta + B, kA = kLf + B;
  static constexpr int total = kA + B;
  static constexpr size_t bytes = (size_t)total * 4;
};

// One CTA per (chunk c, head bh).  Writes Q<-, K->, F, the diagonal-chunk softmax state and
// the chunk-local forget-gate sums.  Rows beyond L are padding with q=k=v=w=0, beta=0
// (H = I), log f = 0.
template <typename T, int B, typename OutT, int D>
__global__ void __launch_bounds__(NT) prep_simt_kernel(
    Geom g, const T* __restrict__ q, const T* __restrict__ k, const T* __restrict__ v,
    const T* __restrict__ w, const float* __restrict__ beta, const float* __restrict__ logf,
    OutT* __restrict__ ql, OutT* __restrict__ kr, OutT* __restrict__ f, float* __restrict__ dm,
    float* __restrict__ dl, float* __restrict__ dacc, float* __restrict__ fa,
    float* __restrict__ fr, float* __restrict__ ft, int with_diag) {
  extern __shared__ float sm[];
  using S = PrepSmem<B, D>;
  constexpr int BS = S::BS, DS = S::DS;
  float* sW = sm + S::kW;
  float* sQ = sm + S::kQ;
  float* sK = sm + S::kK;
  float* sV = sm + S::kV;
  float* sU = sm + S::kU;
  float* sM1 = sm + S::kM1;
  float* sX = sm + S::kX;
  float* sT = sm + S::kT;
  float* sR = sm + S::kR;
  float* sG = sm + S::kG;
  float* sN2 = sm + S::kN2;
  float* sAM = sm + S::kAM;
  float* sBeta = sm + S::kBeta;
  float* sLf = sm + S::kLf;
  float* sA = sm + S::kA;
  // bf16 inputs: products on TF32 tensor cores; fp32 inputs: exact fp32 loops
  constexpr bool TC = std::is_same<T, __nv_bfloat16>::value;

  const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int row0 = c * B;
  const size_t in_row = (size_t)bh * g.L;
  const size_t ws_row = (size_t)bh * g.Lp + row0;

  for (int idx = tid; idx < B * D; idx += NT) {
    const int r = idx / D, cc = idx % D, gi = row0 + r;
    const bool ok = gi < g.L;
    const size_t off = (in_row + gi) * D + cc;
    sW[r * DS + cc] = ok ? to_f(w[off]) : 0.f;
    sQ[r * DS + cc] = ok ? to_f(q[off]) : 0.f;
    sK[r * DS + cc] = ok ? to_f(k[off]) : 0.f;
    if (with_diag) sV[r * DS + cc] = ok ? to_f(v[off]) : 0.f;
  }
  for (int r = tid; r < B; r += NT) {
    const int gi = row0 + r;
    const bool ok = gi < g.L;
    sBeta[r] = ok ? clamp_beta(beta[in_row + gi]) : 0.f;
    sLf[r] = (ok && logf) ? logf[in_row + gi] : 0.f;
  }
  __syncthreads();

  // Phase 1 (independent products of the inputs): G = strictLower(W W^T), M1 = lower(Q W^T),
  // N2 = strictLower(W K^T), Q K^T (start of the diagonal logits); chunk-local forget prefix.
  smem_mm<B, B, D, false, true, TC>(sW, DS, sW, DS, [&](int i, int j, float x) { sG[i * BS + j] = j < i ? x : 0.f; });
  smem_mm<B, B, D, false, true, TC>(sQ, DS, sW, DS, [&](int i, int j, float x) { sM1[i * BS + j] = j <= i ? x : 0.f; });
  smem_mm<B, B, D, false, true, TC>(sW, DS, sK, DS, [&](int i, int j, float x) { sN2[i * BS + j] = j < i ? x : 0.f; });
  smem_mm<B, B, D, false, true, TC>(sQ, DS, sK, DS, [&](int i, int j, float x) { sT[i * BS + j] = x; });
  if (tid == NT - 1) {
    float a = 0.f;
    for (int r = 0; r < B; ++r) { a += sLf[r]; sA[r] = a; }
  }
  __syncthreads();

  // Phase 2: U = (I + strictLower(D G))^{-1} D by forward substitution:
  // row i of U = beta_i (e_i - sum_{m<i} G_im U_m).  U is lower triangular.
  if constexpr (B == 32) {
    // one warp, lane = column: the column of U lives in registers
    if (tid < 32) {
      const int cc = tid;
      float u[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float a0 = (cc == i) ? 1.f : 0.f, a1 = 0.f;
#pragma unroll
        for (int m = 0; m + 1 < i; m += 2) {
          a0 -= sG[i * BS + m] * u[m];
          a1 -= sG[i * BS + m + 1] * u[m + 1];
        }
        if (i & 1) a0 -= sG[i * BS + i - 1] * u[i - 1];
        u[i] = sBeta[i] * (a0 + a1);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) sU[i * BS + cc] = u[i];
    }
    __syncthreads();
  } else {
    for (int i = 0; i < B; ++i) {
      if (tid < B) {
        const int cc = tid;
        float val = 0.f;
        if (cc <= i) {
          float acc = (cc == i) ? 1.f : 0.f;
          for (int m = cc; m < i; ++m) acc -= sG[i * BS + m] * sU[m * BS + cc];
          val = sBeta[i] * acc;
        }
        sU[i * BS + cc] = val;
      }
      __syncthreads();
    }
  }

  // Phase 3: A = M1 U, X = U N2, Y = U^T W
  smem_mm<B, B, B, false, false, TC>(sM1, BS, sU, BS, [&](int i, int j, float x) { sAM[i * BS + j] = x; });
  smem_mm<B, B, B, false, false, TC>(sU, BS, sN2, BS, [&](int i, int j, float x) { sX[i * BS + j] = x; });
  smem_mm<B, D, B, true, false, TC>(sU, BS, sW, DS, [&](int m, int n, float x) { sR[m * DS + n] = x; });
  __syncthreads();

  // Phase 4: Q<- = Q - A W (left edge), K-> = K - X^T W (right edge),
  //          S_d = lower(Q K^T) - M1 X (same element owners as Q K^T), F = I - W^T Y
  smem_mm<B, D, B, false, false, TC>(sAM, BS, sW, DS, [&](int i, int j, float x) {
    ql[(ws_row + i) * D + j] = from_f<OutT>(sQ[i * DS + j] - x);
  });
  smem_mm<B, D, B, true, false, TC>(sX, BS, sW, DS, [&](int j, int n, float x) {
    kr[(ws_row + j) * D + n] = from_f<OutT>(sK[j * DS + n] - x);
  });
  smem_mm<B, B, B, false, false, TC>(sM1, BS, sX, BS, [&](int i, int j, float x) { sT[i * BS + j] -= x; });
  {
    OutT* fout = f + ((size_t)bh * g.nc + c) * D * D;
    smem_mm<D, D, B, true, false, TC>(sW, DS, sR, DS, [&](int n, int kk, float x) {
      fout[n * D + kk] = from_f<OutT>((n == kk ? 1.f : 0.f) - x);
    });
  }
  __syncthreads();

  if (with_diag) {
    // Diagonal-chunk attention partial state per row (log2 domain).
    constexpr int NSUB = NT / B;
    const int r = tid / NSUB, sub = tid % NSUB;
    const float scl = g.scale * kLog2e;
    float mx = -INFINITY;
    for (int j = sub; j < B; j += NSUB) {
      float s = -INFINITY;
      if (j <= r && row0 + j < g.L) s = sT[r * BS + j] * scl + (sA[r] - sA[j]) * kLog2e;
      sT[r * BS + j] = s;
      mx = fmaxf(mx, s);
    }
    mx = group_max<NSUB>(mx);
    float l = 0.f;
    for (int j = sub; j < B; j += NSUB) {
      const float s = sT[r * BS + j];
      const float p = (s == -INFINITY) ? 0.f : fast_exp2(s - mx);
      sT[r * BS + j] = p;
      l += p;
    }
    l = group_sum<NSUB>(l);
    if (sub == 0) {
      dm[ws_row + r] = mx;
      dl[ws_row + r] = l;
    }
    __syncthreads();
    smem_mm<B, D, B, false, false, TC>(sT, BS, sV, DS, [&](int i, int cc, float x) { dacc[(ws_row + i) * D + cc] = x; });
  }

  if (logf) {
    const float tot = sA[B - 1];
    for (int r = tid; r < B; r += NT) {
      fa[ws_row + r] = sA[r];
      fr[ws_row + r] = tot - sA[r];
    }
    if (tid == 0) ft[(size_t)bh * g.nc + c] = tot;
  }
}

template <int B, int D>
struct MainSmem {
  static constexpr int DS = D + 1;
  static constexpr int BS = B + 1;
  static constexpr int kZ = 0, kZn = kZ + B * DS, kK = kZn + B * DS, kV = kK + B * DS;
  static constexpr int kF = kV + B * DS, kP = kF + D * DS, kR = kP + B * BS;
  static constexpr int total = kR + B;
  static constexpr size_t bytes = (size_t)total * 4;
};

// One CTA per (query chunk b, head bh): starts from the diagonal-chunk state and scans the
// earlier chunks right to left: S = Z K->_c^T, online softmax, O += P V_c, Z <- Z F_c^T.
template <typename T, int B, int D>
__global__ void __launch_bounds__(NT) main_simt_kernel(
    Geom g, const T* __restrict__ v, const float* __restrict__ ql, const float* __restrict__ kr,
    const float* __restrict__ f, const float* __restrict__ dm, const float* __restrict__ dl,
    const float* __restrict__ dacc, const float* __restrict__ fa, const float* __restrict__ fr,
    const float* __restrict__ ft, int fox, T* __restrict__ o, float* __restrict__ lse) {
  extern __shared__ float sm[];
  using S = MainSmem<B, D>;
  constexpr int BS = S::BS, DS = S::DS;
  constexpr int NSUB = NT / B;
  constexpr int OC = D / NSUB;
  constexpr int SC = B / NSUB;
  float* sZ = sm + S::kZ;
  float* sZn = sm + S::kZn;
  float* sK = sm + S::kK;
  float* sV = sm + S::kV;
  float* sF = sm + S::kF;
  float* sP = sm + S::kP;
  float* sR = sm + S::kR;

  const int b = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int r = tid / NSUB, sub = tid % NSUB;
  const size_t wrow = (size_t)bh * g.Lp + (size_t)b * B;
  const float scl = g.scale * kLog2e;

  for (int idx = tid; idx < B * D; idx += NT) sZ[(idx / D) * DS + idx % D] = ql[wrow * D + idx];
  float m = dm[wrow + r];
  float l = (sub == 0) ? dl[wrow + r] : 0.f;
  float acc[OC];
#pragma unroll
  for (int u = 0; u < OC; ++u) acc[u] = dacc[(wrow + r) * D + sub + NSUB * u];
  const float arow = fox ? fa[wrow + r] : 0.f;
  float Rsum = 0.f;
  __syncthreads();

  for (int c = b - 1; c >= 0; --c) {
    const size_t crow = (size_t)bh * g.Lp + (size_t)c * B;
    const size_t vrow = (size_t)bh * g.L + (size_t)c * B;  // chunk c < b is always full
    for (int idx = tid; idx < B * D; idx += NT) {
      const int rr = idx / D, cc = idx % D;
      sK[rr * DS + cc] = kr[crow * D + idx];
      sV[rr * DS + cc] = to_f(v[vrow * D + idx]);
    }
    const float* fc = f + ((size_t)bh * g.nc + c) * D * D;
    for (int idx = tid; idx < D * D; idx += NT) sF[(idx / D) * DS + idx % D] = fc[idx];
    for (int j = tid; j < B; j += NT) sR[j] = fox ? fr[crow + j] : 0.f;
    const float Tc = fox ? ft[(size_t)bh * g.nc + c] : 0.f;
    __syncthreads();

    float s[SC];
    float mx = -INFINITY;
    const float rowbias = (arow + Rsum) * kLog2e;
#pragma unroll
    for (int u = 0; u < SC; ++u) {
      const int j = sub + NSUB * u;
      float dot = 0.f;
#pragma unroll 16
      for (int kk = 0; kk < D; ++kk) dot += sZ[r * DS + kk] * sK[j * DS + kk];
      s[u] = dot * scl + rowbias + sR[j] * kLog2e;
      mx = fmaxf(mx, s[u]);
    }
    mx = group_max<NSUB>(mx);
    const float mnew = fmaxf(m, mx);
    const float corr = fast_exp2(m - mnew);
    m = mnew;
    l *= corr;
#pragma unroll
    for (int u = 0; u < OC; ++u) acc[u] *= corr;
#pragma unroll
    for (int u = 0; u < SC; ++u) {
      const float p = fast_exp2(s[u] - m);
      l += p;
      sP[r * BS + sub + NSUB * u] = p;
    }
    // Z' = Z F_c^T
#pragma unroll
    for (int u = 0; u < OC; ++u) {
      const int n = sub + NSUB * u;
      float dot = 0.f;
#pragma unroll 16
      for (int kk = 0; kk < D; ++kk) dot += sZ[r * DS + kk] * sF[n * DS + kk];
      sZn[r * DS + n] = dot;
    }
    __syncwarp();
#pragma unroll
    for (int u = 0; u < OC; ++u) {
      const int cc = sub + NSUB * u;
      float a = 0.f;
#pragma unroll 8
      for (int j = 0; j < B; ++j) a += sP[r * BS + j] * sV[j * DS + cc];
      acc[u] += a;
    }
    Rsum += Tc;
    __syncthreads();
    float* t = sZ; sZ = sZn; sZn = t;
  }

  l = group_sum<NSUB>(l);
  const int gi = b * B + r;
  if (gi < g.L) {
    const float inv = 1.f / l;
    const size_t orow = (size_t)bh * g.L + gi;
#pragma unroll
    for (int u = 0; u < OC; ++u) o[orow * D + sub + NSUB * u] = from_f<T>(acc[u] * inv);
    if (sub == 0) lse[orow] = (m + log2f(l)) * kLn2;
  }
}

template <typename T, int B, int D, typename OutT = float>
cudaError_t prep_t(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                   const float* beta, const float* logf, char* ws, const FwdWs& lay,
                   bool with_diag, cudaStream_t st) {
  auto kern = prep_simt_kernel<T, B, OutT, D>;
  const size_t smem = PrepSmem<B, D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(g.nc, g.BH);
  kern<<<grid, NT, smem, st>>>(g, (const T*)q, (const T*)k, (const T*)v, (const T*)w, beta, logf,
                               (OutT*)(ws + lay.ql), (OutT*)(ws + lay.kr), (OutT*)(ws + lay.f),
                               (float*)(ws + lay.dm), (float*)(ws + lay.dl), (float*)(ws + lay.dacc),
                               (float*)(ws + lay.fa), (float*)(ws + lay.fr), (float*)(ws + lay.ft),
                               with_diag ? 1 : 0);
  return cudaGetLastError();
}

template <typename T, int B, int D>
cudaError_t main_t(const Geom& g, const void* v, const float* logf, char* ws, const FwdWs& lay,
                   void* o, float* lse, cudaStream_t st) {
  auto kern = main_simt_kernel<T, B, D>;
  const size_t smem = MainSmem<B, D>::bytes;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  dim3 grid(g.nc, g.BH);
  kern<<<grid, NT, smem, st>>>(g, (const T*)v, (const float*)(ws + lay.ql), (const float*)(ws + lay.kr),
                               (const float*)(ws + lay.f), (const float*)(ws + lay.dm),
                               (const float*)(ws + lay.dl), (const float*)(ws + lay.dacc),
                               (const float*)(ws + lay.fa), (const float*)(ws + lay.fr),
                               (const float*)(ws + lay.ft), logf ? 1 : 0, (T*)o, lse);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_prep_simt(bool is_bf16, const Geom& g, const void* q, const void* k,
                             const void* v, const void* w, const float* beta, const float* logf,
                             char* ws, const FwdWs& lay, bool with_diag, cudaStream_t st) {
  if (g.D == kHeadDimWide) {
    if (g.B != 32) return cudaErrorInvalidValue;
    return is_bf16 ? prep_t<__nv_bfloat16, 32, kHeadDimWide>(g, q, k, v, w, beta, logf, ws, lay, with_diag, st)
                   : prep_t<float, 32, kHeadDimWide>(g, q, k, v, w, beta, logf, ws, lay, with_diag, st);
  }
  if (g.D != kHeadDim) return cudaErrorInvalidValue;
  if (g.B == 32)
    return is_bf16 ? prep_t<__nv_bfloat16, 32, kHeadDim>(g, q, k, v, w, beta, logf, ws, lay, with_diag, st)
                   : prep_t<float, 32, kHeadDim>(g, q, k, v, w, beta, logf, ws, lay, with_diag, st);
  if (g.B == 64)
    return is_bf16 ? prep_t<__nv_bfloat16, 64, kHeadDim>(g, q, k, v, w, beta, logf, ws, lay, with_diag, st)
                   : prep_t<float, 64, kHeadDim>(g, q, k, v, w, beta, logf, ws, lay, with_diag, st);
  return cudaErrorInvalidValue;
}

cudaError_t launch_main_simt(bool is_bf16, const Geom& g, const void* v, const float* logf,
                             char* ws, const FwdWs& lay, void* o, float* lse, cudaStream_t st) {
  if (g.D == kHeadDimWide) {
    if (g.B != 32) return cudaErrorInvalidValue;
    return is_bf16 ? main_t<__nv_bfloat16, 32, kHeadDimWide>(g, v, logf, ws, lay, o, lse, st)
                   : main_t<float, 32, kHeadDimWide>(g, v, logf, ws, lay, o, lse, st);
  }
  if (g.D != kHeadDim) return cudaErrorInvalidValue;
  if (g.B == 32)
    return is_bf16 ? main_t<__nv_bfloat16, 32, kHeadDim>(g, v, logf, ws, lay, o, lse, st)
                   : main_t<float, 32, kHeadDim>(g, v, logf, ws, lay, o, lse, st);
  if (g.B == 64)
    return is_bf16 ? main_t<__nv_bfloat16, 64, kHeadDim>(g, v, logf, ws, lay, o, lse, st)
                   : main_t<float, 64, kHeadDim>(g, v, logf, ws, lay, o, lse, st);
  return cudaErrorInvalidValue;
}

}  // namespace pathattn
