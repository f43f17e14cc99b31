// Merge of two adjacent chunk-32 UT results (a = earlier, b = later) into the chunk-64
// operands the tensor-core kernels consume.  With F_a, F_b the chunk transforms
// (products of the chunk's H in time order) and row-vector conventions:
//   F64        = F_a F_b
//   K->64 rows = [K->32_a F_b ; K->32_b]      (keys moved to the right edge of the 64-chunk)
//   Q<-64 rows = [Q<-32_a ; Q<-32_b F_a^T]    (queries moved to its left edge)
// The diagonal 64-chunk adds one block to the chunk-32 diagonal blocks: rows of b against keys
// of a, whose logits are Q<-32_b K->32_a^T (adjacent chunks: nothing in between), merged into
// the rows' softmax state.  Forget-gate sums: local prefixes of b gain T_a, local suffixes of a
// gain T_b.  (PaTH reading notes, cc.laoqi.cc/papers/2505.16381, §2.6 interval form and §2.7.)
#include "internal.h"
#include "dev_common.cuh"
#include "smem_mm.cuh"

namespace pathattn {
namespace {

constexpr int NT = 256;
constexpr int D = kHeadDim;
constexpr int DS = D + 1;
constexpr int H32 = 32;

struct MergeSmem {
  float fa[D * DS], fb[D * DS];
  float qb[H32 * DS], ka[H32 * DS], va[H32 * DS];
  float p[H32 * (H32 + 1)];
  float corr[H32];
};

template <typename T>
__global__ void __launch_bounds__(NT) merge64_kernel(
    Geom g, const T* __restrict__ v, const float* __restrict__ ql32, const float* __restrict__ kr32,
    const float* __restrict__ f32, const float* __restrict__ dm32, const float* __restrict__ dl32,
    const float* __restrict__ dacc32, const float* __restrict__ fa32, const float* __restrict__ fr32,
    const float* __restrict__ ft32, __nv_bfloat16* __restrict__ ql64, __nv_bfloat16* __restrict__ kr64,
    __nv_bfloat16* __restrict__ f64, float* __restrict__ dm64, float* __restrict__ dl64,
    float* __restrict__ dacc64, float* __restrict__ fa64, float* __restrict__ fr64, float* __restrict__ ft64,
    int fox, int with_diag) {
  extern __shared__ float smraw[];
  MergeSmem& s = *reinterpret_cast<MergeSmem*>(smraw);
  const int c = blockIdx.x, bh = blockIdx.y, tid = threadIdx.x;
  const int nc32 = g.Lp / 32, nc64 = g.Lp / 64;
  const size_t row0 = (size_t)bh * g.Lp + (size_t)c * 64;  // first row of the 64-chunk
  const float* Fa = f32 + ((size_t)bh * nc32 + 2 * c) * D * D;
  const float* Fb = Fa + D * D;
  for (int idx = tid; idx < D * D; idx += NT) {
    s.fa[(idx / D) * DS + idx % D] = Fa[idx];
    s.fb[(idx / D) * DS + idx % D] = Fb[idx];
  }
  for (int idx = tid; idx < H32 * D; idx += NT) {
    const int r = idx / D, cc = idx % D;
    s.qb[r * DS + cc] = ql32[(row0 + 32 + r) * D + cc];
    s.ka[r * DS + cc] = kr32[(row0 + r) * D + cc];
    if (with_diag) {
      const int gi = c * 64 + r;  // key row of chunk a
      s.va[r * DS + cc] = gi < g.L ? to_f(v[((size_t)bh * g.L + gi) * D + cc]) : 0.f;
    }
  }
  __syncthreads();

  // F64 = F_a F_b
  __nv_bfloat16* fo = f64 + ((size_t)bh * nc64 + c) * D * D;
  smem_mm<D, D, D, false, false, true>(s.fa, DS, s.fb, DS, [&](int n, int k, float x) { fo[n * D + k] = __float2bfloat16_rn(x); });
  // Q<-64 = [Q<-32_a ; Q<-32_b F_a^T],  K->64 = [K->32_a F_b ; K->32_b]
  for (int idx = tid; idx < 32 * D; idx += NT) {
    const int r = idx / D, cc = idx % D;
    ql64[(row0 + r) * D + cc] = __float2bfloat16_rn(ql32[(row0 + r) * D + cc]);
    kr64[(row0 + 32 + r) * D + cc] = __float2bfloat16_rn(kr32[(row0 + 32 + r) * D + cc]);
  }
  smem_mm<H32, D, D, false, true, true>(s.qb, DS, s.fa, DS, [&](int r, int n, float x) {
    ql64[(row0 + 32 + r) * D + n] = __float2bfloat16_rn(x);
  });
  smem_mm<H32, D, D, false, false, true>(s.ka, DS, s.fb, DS, [&](int r, int n, float x) {
    kr64[(row0 + r) * D + n] = __float2bfloat16_rn(x);
  });
  const float Ta = fox ? ft32[(size_t)bh * nc32 + 2 * c] : 0.f;
  const float Tb = fox ? ft32[(size_t)bh * nc32 + 2 * c + 1] : 0.f;
  if (fox) {
    for (int r = tid; r < 64; r += NT) {
      fa64[row0 + r] = fa32[row0 + r] + (r < 32 ? 0.f : Ta);
      fr64[row0 + r] = fr32[row0 + r] + (r < 32 ? Tb : 0.f);
    }
    if (tid == 0) ft64[(size_t)bh * nc64 + c] = Ta + Tb;
  }
  if (!with_diag) return;
  // rows of a keep their chunk-32 diagonal state
  for (int idx = tid; idx < 32 * D; idx += NT) dacc64[row0 * D + idx] = dacc32[row0 * D + idx];
  for (int r = tid; r < 32; r += NT) {
    dm64[row0 + r] = dm32[row0 + r];
    dl64[row0 + r] = dl32[row0 + r];
  }
  // rows of b: merge the block against the keys of a
  smem_mm<H32, H32, D, false, true, true>(s.qb, DS, s.ka, DS, [&](int i, int j, float x) { s.p[i * (H32 + 1) + j] = x; });
  __syncthreads();
  constexpr int NSUB = NT / H32;  // 8 threads per row
  const int r = tid / NSUB, sub = tid % NSUB;
  const size_t wr = row0 + 32 + r;
  const float scl = g.scale * kLog2e;
  const float arow = fox ? fa32[wr] : 0.f;
  float sv[H32 / NSUB];
  float mx = -INFINITY;
#pragma unroll
  for (int u = 0; u < H32 / NSUB; ++u) {
    const int j = sub + NSUB * u;
    float x = s.p[r * (H32 + 1) + j] * scl;
    if (fox) x += (arow + fr32[row0 + j]) * kLog2e;
    if (c * 64 + j >= g.L) x = -INFINITY;  // (never: chunk a is full when b has rows)
    sv[u] = x;
    mx = fmaxf(mx, x);
  }
  mx = group_max<NSUB>(mx);
  const float m0 = dm32[wr];
  const float mnew = fmaxf(m0, mx);
  const float corr = (m0 == -INFINITY) ? 0.f : fast_exp2(m0 - mnew);
  float ls = 0.f;
#pragma unroll
  for (int u = 0; u < H32 / NSUB; ++u) {
    const float pj = (sv[u] == -INFINITY) ? 0.f : fast_exp2(sv[u] - mnew);
    s.p[r * (H32 + 1) + sub + NSUB * u] = pj;
    ls += pj;
  }
  ls = group_sum<NSUB>(ls);
  if (sub == 0) {
    s.corr[r] = corr;
    dm64[wr] = mnew;
    dl64[wr] = dl32[wr] * corr + ls;
  }
  __syncthreads();
  smem_mm<H32, D, H32, false, false, true>(s.p, H32 + 1, s.va, DS, [&](int i, int cc, float x) {
    const size_t w2 = row0 + 32 + i;
    dacc64[w2 * D + cc] = dacc32[w2 * D + cc] * s.corr[i] + x;
  });
}

}  // namespace

cudaError_t launch_merge64(const TcWs& w, const void* v, const float* logf, char* ws, bool with_diag,
                           cudaStream_t st) {
  const Geom& g = w.g64;
  const size_t smem = sizeof(MergeSmem);
  auto kern = merge64_kernel<__nv_bfloat16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
  if (e != cudaSuccess) return e;
  const FwdWs& a = w.p32;
  const FwdWs& b = w.p64;
  kern<<<dim3(g.nc, g.BH), NT, smem, st>>>(
      g, (const __nv_bfloat16*)v, (const float*)(ws + a.ql), (const float*)(ws + a.kr), (const float*)(ws + a.f),
      (const float*)(ws + a.dm), (const float*)(ws + a.dl), (const float*)(ws + a.dacc), (const float*)(ws + a.fa),
      (const float*)(ws + a.fr), (const float*)(ws + a.ft), (__nv_bfloat16*)(ws + b.ql), (__nv_bfloat16*)(ws + b.kr),
      (__nv_bfloat16*)(ws + b.f), (float*)(ws + b.dm), (float*)(ws + b.dl), (float*)(ws + b.dacc),
      (float*)(ws + b.fa), (float*)(ws + b.fr), (float*)(ws + b.ft), logf ? 1 : 0, with_diag ? 1 : 0);
  return cudaGetLastError();
}

}  // namespace pathattn
