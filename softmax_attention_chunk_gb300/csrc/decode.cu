// Decode step of PaTH attention: in-place rewrite of every cached key with the new token's
// transition, append, and single-query softmax attention, in one streaming pass over the cache.
//
// Method: PaTH reading notes (cc.laoqi.cc/papers/2505.16381), §2.8 Eq. (1):
//   k_j <- k_j - beta_t w_t (w_t^T k_j) for j < t, then k_t appended unchanged, so that
//   (k_j^(t))^T q_t = k_j^T H_{j+1} ... H_t q_t.
// The score of the rewritten key needs no second pass: q.k_new = q.k - beta (w.k)(q.w), so both
// dot products come from the key as loaded.  The cache is split along the sequence into
// independent CTAs (a split-KV decode); a second kernel merges the per-split softmax states.
#include "internal.h"
#include "dev_common.cuh"

namespace pathattn {
namespace {

constexpr int NT = 256;          // key groups x (head dim / 8) lanes
constexpr int UNROLL = 4;        // keys in flight per group

template <typename T> struct Vec8;
template <> struct Vec8<__nv_bfloat16> {
  uint4 raw;
  __device__ __forceinline__ void load(const __nv_bfloat16* p) { raw = *reinterpret_cast<const uint4*>(p); }
  __device__ __forceinline__ void store(__nv_bfloat16* p) const { *reinterpret_cast<uint4*>(p) = raw; }
  __device__ __forceinline__ void to_float(float* f) const {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      float2 t = __bfloat1622float2(h[i]);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
  __device__ __forceinline__ void from_float(const float* f) {
    __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&raw);
#pragma unroll
    for (int i = 0; i < 4; ++i) h[i] = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
  }
};
template <> struct Vec8<float> {
  float4 a, b;
  __device__ __forceinline__ void load(const float* p) {
    a = reinterpret_cast<const float4*>(p)[0];
    b = reinterpret_cast<const float4*>(p)[1];
  }
  __device__ __forceinline__ void store(float* p) const {
    reinterpret_cast<float4*>(p)[0] = a;
    reinterpret_cast<float4*>(p)[1] = b;
  }
  __device__ __forceinline__ void to_float(float* f) const {
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
  __device__ __forceinline__ void from_float(const float* f) {
    a = make_float4(f[0], f[1], f[2], f[3]);
    b = make_float4(f[4], f[5], f[6], f[7]);
  }
};

// grid (nsplit, BH).  Split s covers rows [s*per, min((s+1)*per, t+1)) of its head.  A key is
// read by D / 8 lanes, each owning 8 consecutive elements (one 16-byte vector in bf16), so the
// CTA streams 256 / (D / 8) keys at a time (32 at D = 64, 16 at D = 128).
// Writes partial (m [log2 domain], l, acc[D]) to partials[(bh*kDecodeMaxSplits + s)*(D+2)].
// FOX (PaTH-FoX, notes §2.5): the logit of key j gains sum_{s=j+1..t} log f_s = A_t - a_j, with
// ac[bh][j] = a_j the prefix sums of log f kept beside the cache; A_t = a_{t-1} + log f_t is
// stored as row t.
template <typename T, bool FOX, int D>
__global__ void __launch_bounds__(NT) decode_split_kernel(
    int cap, int t, int per, float scale, T* __restrict__ kc, T* __restrict__ vc,
    const T* __restrict__ qt, const T* __restrict__ kt, const T* __restrict__ vt,
    const T* __restrict__ wt, const float* __restrict__ beta_t, float* __restrict__ partials,
    float* __restrict__ ac, const float* __restrict__ logf_t) {
  constexpr int LANES = D / 8;  // lanes per key; each owns 8 consecutive elements
  constexpr int GROUPS = NT / LANES;
  __shared__ float s_m[GROUPS], s_l[GROUPS];
  __shared__ float s_acc[GROUPS][D + 1];

  const int split = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int lane8 = tid % LANES, grp = tid / LANES;
  const int j0 = split * per;
  const int j1 = min(j0 + per, t + 1);
  const size_t hrow = (size_t)bh * cap;
  const int e0 = lane8 * 8;

  float qf[8], wf[8];
  {
    Vec8<T> a, b;
    a.load(qt + (size_t)bh * D + e0);
    b.load(wt + (size_t)bh * D + e0);
    a.to_float(qf);
    b.to_float(wf);
  }
  float qw = 0.f;
#pragma unroll
  for (int i = 0; i < 8; ++i) qw += qf[i] * wf[i];
  qw = group_sum<LANES>(qw);
  const float bt = clamp_beta(beta_t[bh]);
  const float scl = scale * kLog2e;
  float At = 0.f;
  if constexpr (FOX) At = (t > 0 ? ac[hrow + t - 1] : 0.f) + logf_t[bh];

  float m = -INFINITY, l = 0.f, acc[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) acc[i] = 0.f;

  // Trip count is uniform over the CTA so that every lane reaches the group shuffles.
  for (int base = j0; base < j1; base += GROUPS * UNROLL) {
    Vec8<T> kv[UNROLL], vv[UNROLL];
    float aj[UNROLL];  // prefix sums a_j of the keys (FOX), used once the key is consumed
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int j = base + grp + u * GROUPS;
      aj[u] = 0.f;
      if (j < t) {
        kv[u].load(kc + (hrow + j) * D + e0);
        vv[u].load(vc + (hrow + j) * D + e0);
        if constexpr (FOX) aj[u] = ac[hrow + j];
      } else if (j == t) {
        kv[u].load(kt + (size_t)bh * D + e0);
        vv[u].load(vt + (size_t)bh * D + e0);
      } else {
        const float z[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        kv[u].from_float(z);
        vv[u].from_float(z);
      }
    }
#pragma unroll
    for (int u = 0; u < UNROLL; ++u) {
      const int j = base + grp + u * GROUPS;
      const bool valid = j < j1;  // uniform within the lane group
      float kf[8];
      kv[u].to_float(kf);
      float a = 0.f, qk = 0.f;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        a += wf[i] * kf[i];
        qk += qf[i] * kf[i];
      }
      a = group_sum<LANES>(a);
      qk = group_sum<LANES>(qk);
      if (valid) {
        float s;
        if (j < t) {
          const float ba = bt * a;
#pragma unroll
          for (int i = 0; i < 8; ++i) kf[i] -= ba * wf[i];
          Vec8<T> kn;
          kn.from_float(kf);
          kn.store(kc + (hrow + j) * D + e0);
          s = (qk - ba * qw) * scl;
          if constexpr (FOX) s += (At - aj[u]) * kLog2e;
        } else {  // j == t: append the new key and value unchanged
          kv[u].store(kc + (hrow + j) * D + e0);
          vv[u].store(vc + (hrow + j) * D + e0);
          if constexpr (FOX) {
            if (lane8 == 0) ac[hrow + t] = At;
          }
          s = qk * scl;
        }
        float vf[8];
        vv[u].to_float(vf);
        const float mn = fmaxf(m, s);
        const float corr = fast_exp2(m - mn);
        const float p = fast_exp2(s - mn);
        l = l * corr + p;
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = acc[i] * corr + p * vf[i];
        m = mn;
      }
    }
  }

  if (lane8 == 0) {
    s_m[grp] = m;
    s_l[grp] = l;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) s_acc[grp][e0 + i] = acc[i];
  __syncthreads();
  float* out = partials + ((size_t)bh * kDecodeMaxSplits + split) * (D + 2);
  if (tid < D) {
    float M = -INFINITY;
    for (int g2 = 0; g2 < GROUPS; ++g2) M = fmaxf(M, s_m[g2]);
    float a = 0.f, ls = 0.f;
    for (int g2 = 0; g2 < GROUPS; ++g2) {
      const float sc = (s_m[g2] == -INFINITY) ? 0.f : fast_exp2(s_m[g2] - M);
      a += s_acc[g2][tid] * sc;
      ls += s_l[g2] * sc;
    }
    out[2 + tid] = a;
    if (tid == 0) {
      out[0] = M;
      out[1] = ls;
    }
  }
}

// grid BH, block D: merge the per-split states of one head and write o_t.
template <typename T, int D>
__global__ void __launch_bounds__(D) decode_combine_kernel(int nsplit, const float* __restrict__ partials,
                                                           T* __restrict__ o) {
  const int bh = blockIdx.x, c = threadIdx.x;
  const float* p = partials + (size_t)bh * kDecodeMaxSplits * (D + 2);
  float M = -INFINITY;
  for (int s = 0; s < nsplit; ++s) M = fmaxf(M, p[s * (D + 2)]);
  float a = 0.f, l = 0.f;
  for (int s = 0; s < nsplit; ++s) {
    const float ms = p[s * (D + 2)];
    const float sc = (ms == -INFINITY) ? 0.f : fast_exp2(ms - M);
    l += p[s * (D + 2) + 1] * sc;
    a += p[s * (D + 2) + 2 + c] * sc;
  }
  o[(size_t)bh * D + c] = from_f<T>(a / l);
}

template <typename T, int D>
cudaError_t decode_t(int BH, int cap, int t, float scale, void* kc, void* vc, const void* q,
                     const void* k, const void* v, const void* w, const float* beta, void* o,
                     float* partials, float* ac, const float* logf_t, cudaStream_t st) {
  const int n = t + 1;
  // Aim for >= ~4 waves of CTAs over 152 SMs while keeping >= 256 rows per split.
  int nsplit = (n + 1023) / 1024;
  const int want = (4 * 152 * 8 + BH - 1) / BH;
  while (nsplit < want && (n + nsplit) / (nsplit + 1) >= 256) ++nsplit;
  if (nsplit > kDecodeMaxSplits) nsplit = kDecodeMaxSplits;
  if (nsplit < 1) nsplit = 1;
  const int per = (n + nsplit - 1) / nsplit;
  nsplit = (n + per - 1) / per;
  if (ac)
    decode_split_kernel<T, true, D><<<dim3(nsplit, BH), NT, 0, st>>>(
        cap, t, per, scale, (T*)kc, (T*)vc, (const T*)q, (const T*)k, (const T*)v, (const T*)w, beta,
        partials, ac, logf_t);
  else
    decode_split_kernel<T, false, D><<<dim3(nsplit, BH), NT, 0, st>>>(
        cap, t, per, scale, (T*)kc, (T*)vc, (const T*)q, (const T*)k, (const T*)v, (const T*)w, beta,
        partials, nullptr, nullptr);
  decode_combine_kernel<T, D><<<BH, D, 0, st>>>(nsplit, partials, (T*)o);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode(bool is_bf16, int BH, int cap, int t, float scale, void* kc, void* vc,
                          const void* q, const void* k, const void* v, const void* w,
                          const float* beta, void* o, float* partials, cudaStream_t st, float* ac,
                          const float* logf_t, int D) {
  if (D == kHeadDim)
    return is_bf16 ? decode_t<__nv_bfloat16, kHeadDim>(BH, cap, t, scale, kc, vc, q, k, v, w, beta, o, partials, ac, logf_t, st)
                   : decode_t<float, kHeadDim>(BH, cap, t, scale, kc, vc, q, k, v, w, beta, o, partials, ac, logf_t, st);
  if (D == kHeadDimWide)
    return is_bf16 ? decode_t<__nv_bfloat16, kHeadDimWide>(BH, cap, t, scale, kc, vc, q, k, v, w, beta, o, partials, ac,
                                                           logf_t, st)
                   : decode_t<float, kHeadDimWide>(BH, cap, t, scale, kc, vc, q, k, v, w, beta, o, partials, ac, logf_t, st);
  return cudaErrorInvalidValue;
}

}  // namespace pathattn
