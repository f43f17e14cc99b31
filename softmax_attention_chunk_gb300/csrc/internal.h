// Internal declarations shared by the library's translation units (not part of the ABI).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

namespace pathattn {

constexpr int kHeadDim = 64;      // head dim of the tensor-core path (and the default)
constexpr int kHeadDimWide = 128;  // the other head dim: fp32 SIMT kernels and decode
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// Largest number of persistent CTAs the backward main kernel runs (each owns a slab of
// transported-query scratch).  8 per SM on a 152-SM GB300.
constexpr int kBwdMaxCtas = 1216;
// Largest number of sequence splits of one decode step.
constexpr int kDecodeMaxSplits = 128;

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Problem geometry derived from a descriptor.
struct Geom {
  int BH;       // batch * heads
  int L;        // sequence length
  int B;        // chunk size
  int nc;       // number of chunks = ceil(L / B)
  int Lp;       // padded length nc * B
  float scale;
  int D = kHeadDim;  // head dim (kHeadDim or kHeadDimWide)
};

// Byte offsets of the forward workspace.  Element type "E" of ql/kr/f is float32 for the SIMT
// path and bf16 for the tensor-core path (esize).
struct FwdWs {
  size_t ql, kr, f;            // Q<- [BH][Lp][64], K-> [BH][Lp][64], F [BH][nc][64][64]
  size_t dm, dl, dacc;         // diagonal-chunk softmax state: max (log2 domain), sum, acc[64]
  size_t fa, fr, ft;           // forget gate: local inclusive prefix, local exclusive suffix, chunk total
  size_t err;                  // int: first timeout code of a tensor-core kernel (0 = none)
  size_t total;
};

inline FwdWs fwd_ws_layout(const Geom& g, size_t esize, size_t base = 0) {
  FwdWs w{};
  size_t off = base;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  const size_t rows = (size_t)g.BH * g.Lp;
  w.ql = take(rows * g.D * esize);
  w.kr = take(rows * g.D * esize);
  w.f = take((size_t)g.BH * g.nc * g.D * g.D * esize);
  w.dm = take(rows * 4);
  w.dl = take(rows * 4);
  w.dacc = take(rows * g.D * 4);
  w.fa = take(rows * 4);
  w.fr = take(rows * 4);
  w.ft = take((size_t)g.BH * g.nc * 4);
  w.err = take(4);
  w.total = off;
  return w;
}

// Backward workspace: the forward layout (fp32 elements) followed by fp32 gradient
// accumulators and the per-CTA transported-query scratch.
struct BwdWs {
  FwdWs fw;
  size_t Dv;                   // D_i = dO_i . o_i            [BH][Lp]
  size_t dql, dkr, dv;         // dQ<-, dK->, dV accumulators [BH][Lp][64] fp32
  size_t df;                   // dF accumulators             [BH][nc][64][64] fp32
  size_t zs;                   // Z scratch                   [nctas][Lp][64] fp32
  size_t fxa, fxcs;            // PaTH-FoX: prefix sums of log f, colsum - rowsum of dS' [BH][Lp]
  int nctas;
  size_t total;
};

inline int bwd_num_ctas(const Geom& g) {
  const long tiles = (long)g.BH * g.nc;
  return (int)(tiles < kBwdMaxCtas ? tiles : kBwdMaxCtas);
}

inline BwdWs bwd_ws_layout(const Geom& g) {
  BwdWs w{};
  w.fw = fwd_ws_layout(g, 4);
  size_t off = w.fw.total;
  auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
  const size_t rows = (size_t)g.BH * g.Lp;
  w.Dv = take(rows * 4);
  w.dql = take(rows * g.D * 4);
  w.dkr = take(rows * g.D * 4);
  w.dv = take(rows * g.D * 4);
  w.df = take((size_t)g.BH * g.nc * g.D * g.D * 4);
  w.nctas = bwd_num_ctas(g);
  w.zs = take((size_t)w.nctas * g.Lp * g.D * 4);
  w.fxa = take(rows * 4);
  w.fxcs = take(rows * 4);
  w.total = off;
  return w;
}

// Workspace of the bf16 tensor-core path (Lp a multiple of 128).  p64: chunk-64 operands of the
// tcgen05 kernels (bf16 Q<-, K->, F; fp32 diagonal-chunk softmax and forget-gate state).
struct TcWs {
  Geom g64;
  FwdWs p64;
  // backward only
  size_t Dv;                       // D_i                                [BH][Lp]
  size_t dql64, dkr64, dv, df64;   // chunk-64 gradients (fp32; dkr64/dv/df64 accumulate)
  size_t zs;                       // transported queries Z, bf16 swizzled 128x64 tiles
  size_t fxa, fxcs;                // PaTH-FoX: prefix sums of log f, column sums of dS' [BH][Lp]
  size_t total;
};

inline Geom tc_geom(int BH, int L, float scale, int B) {
  Geom g;
  g.BH = BH;
  g.L = L;
  g.Lp = (L + 127) / 128 * 128;
  g.B = B;
  g.nc = g.Lp / B;
  g.scale = scale;
  return g;
}

inline TcWs tc_ws_layout(int BH, int L, float scale, bool for_backward) {
  TcWs w{};
  w.g64 = tc_geom(BH, L, scale, 64);
  // p64 first: the forward and backward layouts place it at the same offsets
  w.p64 = fwd_ws_layout(w.g64, 2, 0);
  size_t off = w.p64.total;
  if (for_backward) {
    auto take = [&](size_t bytes) { size_t o = off; off = align_up(off + bytes, 256); return o; };
    const size_t rows = (size_t)BH * w.g64.Lp;
    const size_t nt = (size_t)w.g64.Lp / 128;
    w.Dv = take(rows * 4);
    w.dql64 = take(rows * kHeadDim * 4);
    w.dkr64 = take(rows * kHeadDim * 4);
    w.dv = take(rows * kHeadDim * 4);
    w.df64 = take((size_t)BH * w.g64.nc * kHeadDim * kHeadDim * 4);
    // tile T of a head has at most 2T+1 steps: sum over tiles <= nt^2 tiles of 16 KB
    w.zs = take((size_t)BH * nt * nt * 128 * 128);
    w.fxa = take(rows * 4);
    w.fxcs = take(rows * 4);
  }
  w.total = off;
  return w;
}

inline size_t decode_ws_bytes(int BH, int D = kHeadDim) {
  return align_up((size_t)BH * kDecodeMaxSplits * (D + 2) * 4, 256);
}

// ---- launchers (return cudaGetLastError() of their launches) ----

// PaTH-FoX backward helpers (one CTA per head): A[bh][i] = sum_{s<=i} log f_s over [0, Lp) (rows
// >= L keep the total), and dlog f_s = -sum_{m>=s} cs[bh][m] for s < L.
cudaError_t launch_fox_prefix(const Geom& g, const float* logf, float* A, cudaStream_t st);
cudaError_t launch_fox_dlogf(const Geom& g, const float* cs, float* dlogf, cudaStream_t st);

// SIMT (fp32 arithmetic) forward.  is_bf16 selects the input element type; g.D is 64 (chunk 32
// or 64) or 128 (chunk 32).
cudaError_t launch_prep_simt(bool is_bf16, const Geom& g, const void* q, const void* k,
                             const void* v, const void* w, const float* beta, const float* logf,
                             char* ws, const FwdWs& lay, bool with_diag, cudaStream_t st);
cudaError_t launch_main_simt(bool is_bf16, const Geom& g, const void* v, const float* logf,
                             char* ws, const FwdWs& lay, void* o, float* lse, cudaStream_t st);

// Prefill -> decode hand-off: rows 0..g.L-1 of the caches ([g.BH][cap][64]) get the prompt keys
// transported to the prompt end and the prompt values; g.B must be 64; ws holds at least
// prefill_ws_bytes(g, is_bf16) bytes.
// With logf and a_cache set (PaTH-FoX), rows 0..g.L-1 of a_cache ([g.BH][cap] fp32) get the
// inclusive prefix sums of logf ([g.BH][g.L]).
size_t prefill_ws_bytes(const Geom& g, bool is_bf16);
// Byte offset in that workspace of the int error word of the tcgen05 preparation (bf16 caches at
// head dim 64), or (size_t)-1 when the hand-off runs no kernel with bounded waits.
size_t prefill_err_offset(const Geom& g, bool is_bf16);
cudaError_t launch_prefill(bool is_bf16, const Geom& g, int cap, const void* k, const void* v, const void* w,
                           const float* beta, void* k_cache, void* v_cache, char* ws, cudaStream_t st,
                           const float* logf = nullptr, float* a_cache = nullptr);

// tcgen05 UT preparation at chunk 64 (bf16 inputs): writes the chunk-64 operands of the
// tensor-core scans (bf16 Q<-, K->, F) and, with_diag, the diagonal softmax state.  With f32_f
// (and no diagonal state) F is written split, F = F_hi + F_lo, as two bf16 64 x 64 tiles in the
// 128-byte swizzled layout per chunk ([BH][nc][2][64 x 64], 16 KB per chunk) at lay.f, which must
// then have room for it, from products whose bf16 operands U and U^T W are split into high and
// low bf16 parts (about 16 significant bits).  with_q = false (with f32_f) runs the keys-only
// instance of the hand-off: Q<- is not written, q is not read, and rows 0..g.L-1 of v are copied
// to v_cache ([g.BH][cap][64] bf16, cap >= g.L).  stall_ns (test hook of the failure path): nonzero makes every CTA give
// up a wait on a barrier nothing arrives at after that many ns, recording code 99 in lay.err, and
// end without writing anything.
cudaError_t launch_ut_prep64(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                             const float* beta, const float* logf, char* ws, const FwdWs& lay, bool with_diag,
                             cudaStream_t st, bool f32_f = false, uint32_t stall_ns = 0, bool with_q = true,
                             void* v_cache = nullptr, int cap = 0);

// Chunk walk on tcgen05 at head dim 64 over 64-row chunks, one CTA per head: with M = I at the
// first chunk visited, out_c = X_c M_c^T for every chunk and the next M = M_c F_c^T (right to
// left, asc = false: M_c = S_c, the suffix product) or M_c F_c (left to right, asc = true:
// M_c = P_c^T), M held as a bf16 high/low pair and every product split-precision.  x: chunk-aligned
// bf16 rows [g.BH][g.Lp][64]; fs: the split chunk transforms of launch_ut_prep64 with f32_f; out:
// rows [g.BH][out_head][64] (fp32 with out_f32, else bf16), rows >= g.L not written; t_out (right to
// left only, may be null): the final M = S_{-1} [g.BH][64][64] fp32.  err: the int that a wait
// that gives up records its code in.
cudaError_t launch_walk_tc(const Geom& g, bool asc, bool out_f32, const void* x, const void* fs, void* out,
                           size_t out_head, float* t_out, int* err, cudaStream_t st);
// Both walks of a context-parallel shard in one launch: xk (K->) right to left into fp32 k_out and
// t_out, xq (Q<-) left to right into bf16 q_out (both [g.BH][out_head][64]).
cudaError_t launch_walk_tc_pair(const Geom& g, const void* xk, const void* xq, const void* fs, float* k_out,
                                void* q_out, size_t out_head, float* t_out, int* err, cudaStream_t st);
// Head dim 128 (bf16): the tcgen05 UT preparation of every 64-row chunk (Q<-, K->, F = 128 x 128
// in bf16, the diagonal softmax state) into lay = fwd_ws_layout(g, 2) with g.D = 128, g.B = 64, and
// the tcgen05 forward scan over 128-row query tiles from it (g.nc even).
cudaError_t launch_ut_prep128(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                              const float* beta, const float* logf, char* ws, const FwdWs& lay, cudaStream_t st);
cudaError_t launch_scan128_tc(const Geom& g, const void* v, const float* logf, char* ws, const FwdWs& lay, void* o,
                              float* lse, cudaStream_t st);
// tcgen05 forward scan over 128-row query tiles (pairs of 64-row chunks); g.nc must be even.
cudaError_t launch_scan_tc(const Geom& g, const void* v, const float* logf, char* ws,
                           const FwdWs& lay, void* o, float* lse, void* zstore, cudaStream_t st);

// SIMT backward.  phases: bit 0 = prepare (zero accumulators, D_i, recomputed UT quantities),
// bit 1 = adjoint chunk scan, bit 2 = per-chunk UT backward writing the gradients.  With logf
// (PaTH-FoX, [BH][L]) the logits carry the forget-gate bias; dlogf (needs logf) receives its
// gradient at the end of bit 2.
cudaError_t launch_bwd_simt(bool is_bf16, const Geom& g, const void* q, const void* k,
                            const void* v, const void* w, const float* beta, const void* o,
                            const float* lse, const void* dO, void* dq, void* dk, void* dv,
                            void* dw, float* dbeta, char* ws, const BwdWs& lay, int phases,
                            cudaStream_t st, const float* logf = nullptr, float* dlogf = nullptr);

// D_i = dO_i . o_i for the bf16 tensor-core backward.
cudaError_t launch_bwd_dot(const Geom& g, const void* o, const void* dO, float* Dv, cudaStream_t st);
// tcgen05 UT backward at chunk 64: diagonal-chunk attention backward and the chain rule through
// the per-chunk UT quantities, writing dq, dk, dv, dw, dbeta.
cudaError_t launch_ut_bwd64(const Geom& g, const void* q, const void* k, const void* v, const void* w,
                            const float* beta, const float* lse, const void* dO, const float* Dv, const float* dql,
                            const float* dkr, const float* dvacc, const float* df, void* dq, void* dk, void* dv,
                            void* dw, float* dbeta, int* err, cudaStream_t st, const float* logf = nullptr,
                            float* fxcs = nullptr);
// Tensor-core backward (bf16).  phases: 1 = prepare (accumulators, D_i, chunk-32 UT quantities,
// chunk-64 merge, Z chain), 2 = adjoint scan, 4 = chunk conversion + UT backward; with bit 8
// the prepare phase keeps the forward's preparation found in ws.
cudaError_t launch_bwd_tc(const TcWs& w, const void* q, const void* k, const void* v, const void* wv,
                          const float* beta, const void* o, const float* lse, const void* dO, void* dq, void* dk,
                          void* dv, void* dw, float* dbeta, char* ws, int phases, cudaStream_t st, const float* logf = nullptr,
                          float* dlogf = nullptr);

// Decode step.
// ac / logf_t (PaTH-FoX, both set or both null): prefix sums of log f beside the cache
// ([BH][cap] fp32, rows 0..t-1 valid, row t written) and this step's log f ([BH]).
// D: head dim (kHeadDim or kHeadDimWide); partials hold decode_ws_bytes(BH, D) bytes.
cudaError_t launch_decode(bool is_bf16, int BH, int cap, int t, float scale, void* kc, void* vc,
                          const void* q, const void* k, const void* v, const void* w,
                          const float* beta, void* o, float* partials, cudaStream_t st, float* ac = nullptr,
                          const float* logf_t = nullptr, int D = kHeadDim);

}  // namespace pathattn
