/*
 * path_attn.h — C ABI of the GB300 (sm_103a) PaTH attention library.
 *
 * PaTH attention (Yang et al., "PaTH Attention: Position Encoding via Accumulating Householder
 * Transformations", arXiv 2505.16381v2; reading notes at cc.laoqi.cc/papers/2505.16381/v2/r1):
 *
 *   H_t        = I - beta_t w_t w_t^T                          (notes §2.1)
 *   logit(i,j) = scale * k_j^T H_{j+1} H_{j+2} ... H_i q_i       (j <= i; H_j excluded, H_i included)
 *              + sum_{s=j+1..i} log f_s                         (optional PaTH-FoX gate, notes §2.5)
 *   o_i        = sum_{j<=i} softmax_j(logit(i,.)) v_j,  lse_i = log sum_{j<=i} exp(logit(i,j))
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - All tensor arguments are DEVICE pointers into memory the caller owns (cudaMalloc, PyTorch,
 *    ...).  The library allocates nothing, frees nothing, and keeps no state between calls
 *    other than a per-device attribute cache.  Calls are reentrant.
 *  - Layouts are dense row-major: q,k,v,w,o,dO,dq,dk,dv,dw are [batch][heads][seqlen][head_dim];
 *    beta, log_f, lse, dbeta are [batch][heads][seqlen].  Decode vectors are
 *    [batch][heads][head_dim], beta_t is [batch][heads], caches are
 *    [batch][heads][capacity][head_dim].
 *  - Element type of q,k,v,w,o,dO,dq,dk,dv,dw and of the caches: the descriptor's dtype
 *    (PATH_BF16 or PATH_FP32).  beta, log_f, lse, dbeta are always float32.  Arithmetic
 *    accumulates in fp32.
 *  - Every tensor pointer must be 16-byte aligned.  Workspace ("ws") pointers must be 256-byte
 *    aligned and hold at least the size returned by the matching *_workspace_size function.
 *  - beta is clamped to [0, 2] inside the kernels (the range of the 2*sigmoid parameterisation,
 *    notes §2.1/§2.2).  Inputs already in range are used unchanged; dbeta is the gradient with
 *    respect to the clamped value.  w is used as given (it is not renormalised).
 *  - "stream" is a cudaStream_t passed as void* (NULL = legacy default stream).  Work is
 *    enqueued asynchronously; faults inside kernels surface at the caller's next sync, and a
 *    tensor-core kernel whose internal wait gave up is reported by path_attn_workspace_status.
 *  - Errors: every argument is validated before any CUDA call; on a validation error nothing
 *    is launched and a status below is returned.  Launch failures return PATH_ERR_CUDA.
 *    No exception crosses the ABI.
 */
#ifndef PATH_ATTN_H
#define PATH_ATTN_H

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PATH_OK = 0,
  PATH_ERR_INVALID_ARG = 1,  /* null pointer, non-positive size, misaligned pointer, bad enum */
  PATH_ERR_UNSUPPORTED = 2,  /* valid but not implemented (head_dim not 64 or 128, chunk value, ...) */
  PATH_ERR_WORKSPACE = 3,    /* ws_bytes smaller than the required workspace */
  PATH_ERR_CAPACITY = 4,     /* decode: t + 1 > capacity */
  PATH_ERR_CUDA = 5,         /* a CUDA runtime call or kernel launch failed */
  PATH_ERR_INTERNAL = 6
} path_status_t;

typedef enum { PATH_BF16 = 0, PATH_FP32 = 1 } path_dtype_t;

typedef struct {
  int batch;      /* > 0 */
  int heads;      /* > 0 */
  int seqlen;     /* L > 0 */
  int head_dim;   /* d: 64 or 128.  bf16 at 64 runs the tcgen05 kernels (chunk 64); the bf16
                     forward at 128 runs the head-dim-128 tcgen05 kernels (chunk 0 or 64: 64-row
                     chunks); fp32 and the backward at 128 run the fp32 CUDA-core kernels with
                     32-row chunks (fp32 chunk 64 at 128 is PATH_ERR_UNSUPPORTED) */
  int dtype;      /* path_dtype_t of q,k,v,w,o (and dO,dq,dk,dv,dw in the backward) */
  float scale;    /* multiplies the Householder-path logit; the forget bias is added unscaled */
  int chunk;      /* UT chunk size B; 0 lets the library choose (see path_attn_chunk) */
} path_attn_desc_t;

typedef struct {
  int batch;       /* > 0 */
  int heads;       /* > 0 */
  int head_dim;    /* 64 or 128 (path_decode_step_noalloc: 64 only) */
  int capacity;    /* rows allocated per (batch, head) in each cache */
  int cache_dtype; /* path_dtype_t of the caches and of q_t,k_t,v_t,w_t,o_t */
  float scale;     /* logit multiplier */
} path_decode_desc_t;

/* Human-readable name of a status code (static string, never NULL). */
const char* path_status_string(int status);

/* Chunk size B used by the forward (for_backward = 0) or backward (1) pass for this
 * descriptor, or minus a path_status_t if the descriptor is invalid/unsupported. Host only. */
int path_attn_chunk(const path_attn_desc_t* desc, int for_backward);

/* Bytes of workspace path_attn_fwd (for_backward = 0) or path_attn_bwd (for_backward = 1)
 * needs for this descriptor; 0 if the descriptor is invalid.  Host only, no CUDA call. */
size_t path_attn_workspace_size(const path_attn_desc_t* desc, int for_backward);

/*
 * Forward pass: o and lse for every (batch, head, row).
 *
 * Steps (notes §2.6–§2.7): per chunk of B positions, the UT transform
 * U = (I + strictLower(D W W^T))^{-1} D by forward substitution; the boundary-adjusted queries
 * Q<- = Q - lower(Q W^T) U W, keys K-> = K - (U strictLower(W K^T))^T W and chunk transform
 * F = I - W^T U^T W; the diagonal chunk from lower(Q K^T) - lower(Q W^T) U strictLower(W K^T);
 * then, per query chunk, a right-to-left scan over earlier chunks (scores Z K->^T, online
 * softmax, O += P V, Z <- Z F^T).
 *
 * log_f: forget-gate log values (<= 0) or NULL for plain PaTH.
 * o: output, desc dtype.  lse: float32 natural-log log-sum-exp per row (the backward needs it).
 * ws/ws_bytes: scratch of at least path_attn_workspace_size(desc, 0) bytes; its contents on
 * entry are ignored and on exit are unspecified.
 */
int path_attn_fwd(const path_attn_desc_t* desc, const void* q, const void* k, const void* v,
                  const void* w, const float* beta, const float* log_f, void* o, float* lse,
                  void* ws, size_t ws_bytes, void* stream);

/*
 * Backward pass: gradients of sum(dO * o) with respect to q, k, v, w and beta, given the
 * forward's o and lse for the same inputs.  The pages give no backward; this is the exact
 * derivative of the forward definition, evaluated blockwise: recomputed per-chunk UT
 * quantities, a descending scan that stores the transported queries Z_c, an ascending adjoint
 * scan G_c = dS_c K->_c + G_{c-1} F_c with dF_c += G_{c-1}^T Z_c, then the chain rule through
 * the per-chunk UT quantities.
 *
 * dq,dk,dv,dw: desc dtype outputs (overwritten).  dbeta: float32 (overwritten).
 * PaTH-FoX (forget gate, notes §2.5): pass the forward's log_f; dlog_f (float32, same shape,
 * may be NULL) receives dL/dlog f.  dlog_f without log_f is PATH_ERR_INVALID_ARG.  Both paths
 * take the forget gate; the bf16 tensor-core path recovers the logit gradient from the scaled
 * one, so there log_f with scale == 0 returns PATH_ERR_UNSUPPORTED (the fp32 path accepts it).
 * ws: at least path_attn_workspace_size(desc, 1) bytes.
 */
int path_attn_bwd(const path_attn_desc_t* desc, const void* q, const void* k, const void* v,
                  const void* w, const float* beta, const float* log_f, const void* o,
                  const float* lse, const void* dO, void* dq, void* dk, void* dv, void* dw,
                  float* dbeta, float* dlog_f, void* ws, size_t ws_bytes, void* stream);

/*
 * The same two passes split into their phases, so that a caller can time or overlap them.
 * path_attn_fwd(...) is path_attn_fwd_phases(PATH_FWD_ALL, ...); path_attn_bwd likewise.
 * Phases must run in the listed order on one stream with the same arguments and the same
 * workspace, and nothing else may use that workspace in between.  Arguments, validation and
 * errors are those of the full call (every pointer is checked whatever the phase);
 * phases == 0 or an unknown bit gives PATH_ERR_INVALID_ARG.
 *   forward:  PREPARE = per-chunk UT transform, Q<-, K->, F and diagonal-chunk softmax state
 *             into ws;  SCAN = right-to-left chunk scan writing o and lse.
 *   backward: PREPARE = zero the accumulators, D_i = dO_i . o_i, recompute the per-chunk UT
 *             quantities;  SCAN = descending Z pass and ascending adjoint scan (accumulates
 *             dV, dK->, dF, writes dQ<- in ws);  FINISH = diagonal-chunk and UT backward
 *             writing dq, dk, dv, dw, dbeta.
 */
enum { PATH_FWD_PREPARE = 1, PATH_FWD_SCAN = 2, PATH_FWD_ALL = 3 };
enum { PATH_BWD_PREPARE = 1, PATH_BWD_SCAN = 2, PATH_BWD_FINISH = 4, PATH_BWD_ALL = 7 };
/* Optional bit for path_attn_bwd_phases(PREPARE): the workspace already holds the forward's
 * per-chunk preparation for exactly these inputs and descriptor, because path_attn_fwd was run
 * with this same workspace (sized by path_attn_workspace_size(desc, 1)) and nothing used it since.
 * PREPARE then skips recomputing it (the bf16 tensor-core path; ignored by the fp32 path).  If the
 * statement is false the gradients are wrong; nothing detects it. */
enum { PATH_BWD_REUSE_FWD = 8 };
/* Optional bit for path_attn_fwd_phases(SCAN), for a forward that a backward will follow (a
 * training step): ws must be backward-sized (path_attn_workspace_size(desc, 1), else
 * PATH_ERR_WORKSPACE), and the scan also stores every transported query tile Z_n (§2.7: the
 * queries carried across earlier chunks) in ws, which the backward needs.  The bf16
 * tensor-core path at head_dim 64 only; ignored otherwise. */
enum { PATH_FWD_STORE_Z = 4 };
/* Optional bit for path_attn_bwd_phases(PREPARE): the workspace already holds the transported
 * query tiles because the forward ran with PATH_FWD_STORE_Z on it (same inputs, descriptor and
 * workspace, nothing used it since); PREPARE then skips recomputing them.  Same caveat and scope
 * as PATH_BWD_REUSE_FWD. */
enum { PATH_BWD_Z_FROM_FWD = 16 };

int path_attn_fwd_phases(int phases, const path_attn_desc_t* desc, const void* q, const void* k,
                         const void* v, const void* w, const float* beta, const float* log_f,
                         void* o, float* lse, void* ws, size_t ws_bytes, void* stream);

int path_attn_bwd_phases(int phases, const path_attn_desc_t* desc, const void* q, const void* k,
                         const void* v, const void* w, const float* beta, const float* log_f,
                         const void* o, const float* lse, const void* dO, void* dq, void* dk,
                         void* dv, void* dw, float* dbeta, float* dlog_f, void* ws,
                         size_t ws_bytes, void* stream);

/* Bytes of workspace path_decode_step needs for any t < capacity; 0 if invalid. Host only. */
size_t path_decode_workspace_size(const path_decode_desc_t* desc);

/*
 * One decode step at position t (notes §2.8, Eq. (1)).  On entry rows 0..t-1 of each cache
 * hold the keys/values of earlier positions, keys already transported to position t-1.
 * The step
 *   1. rewrites every cached key in place: k_j <- k_j - beta_t (w_t . k_j) w_t   (j < t),
 *   2. appends k_t and v_t unchanged at row t,
 *   3. writes o_t = sum_j softmax_j(scale k_j . q_t) v_j over j = 0..t.
 * Requires 0 <= t and t + 1 <= capacity (else PATH_ERR_CAPACITY).
 * q_t,k_t,v_t,w_t,o_t: [batch][heads][head_dim] in cache_dtype; beta_t: [batch][heads] float32.
 * ws: at least path_decode_workspace_size(desc) bytes (per-split partial softmax states).
 */
int path_decode_step(const path_decode_desc_t* desc, void* k_cache, void* v_cache, int t,
                     const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                     const float* beta_t, void* o_t, void* ws, size_t ws_bytes, void* stream);

/* Bytes of workspace path_decode_prefill needs for a prompt of prompt_len tokens (the fp32
 * chunk transforms of the prompt); 0 if the descriptor or prompt_len is invalid. Host only. */
size_t path_decode_prefill_workspace_size(const path_decode_desc_t* desc, int prompt_len);

/*
 * Prefill -> decode hand-off (notes §2.8, last paragraph: after a prefill every key must be
 * aligned to the prompt end, by the block suffix products).  Fills rows 0..prompt_len-1 of each
 * cache so that path_decode_step can continue at t = prompt_len:
 *   k_cache row j = H_{L-1} ... H_{j+1} k_j   (H_t = I - beta_t w_t w_t^T, L = prompt_len),
 *   v_cache row j = v_j,
 * i.e. exactly what prompt_len calls of path_decode_step from an empty cache would leave there.
 * Computed blockwise in fp32 (64-row chunks: each key moved to its chunk's end, then through the
 * later chunks' transforms right to left; 32-row chunks at head_dim 128) and rounded once to
 * cache_dtype.
 * k, v, w: [batch][heads][prompt_len][head_dim] in cache_dtype; beta: [batch][heads][prompt_len]
 * float32 (clamped to [0, 2]).  Caches: [batch][heads][capacity][head_dim]; rows >= prompt_len
 * are not touched.  Requires 0 <= prompt_len <= capacity (else PATH_ERR_CAPACITY); prompt_len = 0
 * does nothing.  PaTH-FoX: with log_f ([batch][heads][prompt_len] float32) and a_cache
 * ([batch][heads][capacity] float32) both given, rows 0..prompt_len-1 of a_cache get the inclusive
 * prefix sums of log_f, as path_decode_step_fox expects; both NULL for plain PaTH (one without the
 * other is PATH_ERR_INVALID_ARG).  ws: at least path_decode_prefill_workspace_size(desc, prompt_len) bytes,
 * 256-byte aligned.  Asynchronous on stream.
 */
int path_decode_prefill(const path_decode_desc_t* desc, void* k_cache, void* v_cache, int prompt_len,
                        const void* k, const void* v, const void* w, const float* beta, const float* log_f,
                        float* a_cache, void* ws, size_t ws_bytes, void* stream);

/*
 * One PaTH-FoX decode step (notes §2.8 Eq. (1) with the forget gate of §2.5): the key rewrite
 * and append of path_decode_step, and the logit of cached key j gains
 *   sum_{s=j+1..t} log f_s = a_t - a_j,
 * where a_cache ([batch][heads][capacity] float32) holds the prefix sums a_j = sum_{s<=j} log f_s
 * of the cached rows (rows 0..t-1 on entry; path_decode_prefill with log_f fills them for a
 * prompt).  The step stores a_t = a_{t-1} + log_f_t (a_{-1} = 0) in row t, then
 *   o_t = sum_j softmax_j(scale k_j . q_t + a_t - a_j) v_j   over j = 0..t.
 * log_f_t: [batch][heads] float32 (log of the forget gate, <= 0).  Other arguments, requirements
 * and errors as path_decode_step (same workspace size).
 */
int path_decode_step_fox(const path_decode_desc_t* desc, void* k_cache, void* v_cache, float* a_cache, int t,
                         const void* q_t, const void* k_t, const void* v_t, const void* w_t, const float* beta_t,
                         const float* log_f_t, void* o_t, void* ws, size_t ws_bytes, void* stream);

#define PATH_DECODE_NOALLOC_MAX_HEADS 496
/*
 * path_decode_step without a workspace argument.  The paper has no counterpart: this exists
 * for callers that cannot allocate device memory when they decode — code running inside
 * another runtime's memory pool without access to its allocator, plugins that may only use
 * the buffers handed to them, or serving loops that forbid allocation after start-up.
 *
 * Same arguments, semantics and results as path_decode_step, minus ws/ws_bytes.  The per-split
 * partial softmax states live in a fixed 16 MiB array inside the library, present on every
 * GPU that loads it until the process exits.  Limit: batch * heads <= PATH_DECODE_NOALLOC_MAX_HEADS,
 * otherwise PATH_ERR_WORKSPACE is returned and nothing runs.  The call itself allocates
 * nothing (no cudaMalloc, no library allocator).
 *  - The first call made with a given device current looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call before any stream capture.
 *    The cached address belongs to that device's current context: after cudaDeviceReset (or
 *    anything else that destroys the primary context) it is stale, and this entry point must
 *    not be called again in that process.
 *  - All calls on a device share the one array: calls that may overlap on the GPU (different
 *    streams without ordering between them) race and give wrong results.  Calls ordered on one
 *    stream are safe.  Nothing in the array needs to start at zero: each call overwrites the
 *    parts it reads.
 */
int path_decode_step_noalloc(const path_decode_desc_t* desc, void* k_cache, void* v_cache, int t,
                             const void* q_t, const void* k_t, const void* v_t, const void* w_t,
                             const float* beta_t, void* o_t, void* stream);

/*
 * Device-side status of the passes that ran on a workspace.  (The pages have no failure
 * machinery; this is the library's own.)  Every wait of the tensor-core kernels on their internal
 * pipeline barriers is bounded (about 2 s); a wait that gives up writes a nonzero code into an int
 * inside the workspace (the first code wins) and its kernel ends early, so the outputs of that
 * call are incomplete even though the call returned PATH_OK (kernels run after it returns).
 * This call waits for all work queued on `stream` (it synchronises the stream), then reads that
 * word through a 4-byte copy into host memory.
 *   desc, for_backward: the descriptor and the pass the workspace was sized for (they fix where the
 *     word lives); ws, ws_bytes: that workspace.
 * Returns PATH_OK (no wait gave up), PATH_ERR_INTERNAL (one did; *code, when code is not NULL,
 * receives the first recorded code), PATH_ERR_CUDA (the synchronisation or the copy failed, e.g.
 * after a kernel fault), or an argument error as the passes would return it.  Passes that run the
 * fp32 CUDA-core kernels have no such waits: the call returns PATH_OK for them without touching
 * the device.
 * The word is cleared by the forward's PREPARE phase and by the backward's PREPARE phase (except
 * with PATH_BWD_REUSE_FWD or PATH_BWD_Z_FROM_FWD, where it keeps the forward's code), so it covers
 * every tensor-core kernel since the last clearing.
 * Test hook: with the environment variable PATH_ATTN_DEBUG_STALL_NS set to n > 0 at the time of
 * a call, the forward's PREPARE phase on the tensor-core path makes every CTA wait on a barrier
 * that nothing arrives at, give up after n ns (at most 1 s), record code 99 and end without
 * writing anything; the workspace status then reads PATH_ERR_INTERNAL with code 99.  The context
 * stays usable: a later call without the variable runs normally.
 */
int path_attn_workspace_status(const path_attn_desc_t* desc, int for_backward, const void* ws, size_t ws_bytes,
                               int* code, void* stream);

/* The same for the workspace of path_decode_prefill (desc and prompt_len as given to it): the
 * tcgen05 preparation of bf16 caches at head dim 64 has bounded waits; the other hand-off paths
 * have none (PATH_OK).  Synchronises `stream`. */
int path_decode_prefill_status(const path_decode_desc_t* desc, int prompt_len, const void* ws, size_t ws_bytes,
                               int* code, void* stream);

/*
 * Context parallelism (sequence sharding) of the forward pass.  The reading notes §2.8, last
 * paragraph (the paper's Sec. 3.5), sketch it: pass the transported keys and values and the block
 * transforms between devices and accumulate right to left.  The sequence of L tokens is cut into
 * consecutive shards, one per device, each a multiple of 128 tokens.  For a query i of shard r and
 * a key j of an earlier shard r':
 *   logit(i, j) = scale * k~_j^T (M_{r'+1} ... M_{r-1}) z^_i + a_i + b_j
 * with k~_j = H_{e(r')} ... H_{j+1} k_j (the key moved to the end of its shard), z^_i =
 * H_{s(r)} ... H_i q_i (the query moved to the start of its shard), M_s = H_{s(s)} ... H_{e(s)}
 * (the product over shard s) and, with a forget gate, a_i = sum_{t=s(r)..i} log f_t and
 * b_j = sum_{t=j+1..e(r')} log f_t plus the totals of the shards in between.  Each device then:
 *   1. runs path_attn_fwd_phases(PATH_FWD_PREPARE) on its shard (fwd_ws) and
 *      path_cp_shard_prepare (its keys moved to its end, its queries moved to its start, M^T, and
 *      the forget-gate terms);
 *   2. for every earlier shard, receives that shard's key block (already moved to the end of the
 *      previous shard), its values and key biases, merges them into its queries' softmax state
 *      with path_cp_attend_block, moves the block through its own shard with path_cp_pass_block
 *      and sends it on to the next device;
 *   3. runs path_attn_fwd_phases(PATH_FWD_SCAN): o and lse over the whole prefix.
 * The order in which blocks are merged does not change the result (up to rounding).  Scope: bf16
 * at head dim 64 (the tensor-core path), seqlen and block_len multiples of 128, forward only (the
 * backward is not sharded).  desc is always the local shard's descriptor (seqlen = its length).
 */

/* Bytes of workspace path_cp_shard_prepare needs; 0 if desc is invalid or outside the scope. */
size_t path_cp_prepare_workspace_size(const path_attn_desc_t* desc);

/*
 * Per-shard transports.  Inputs q, k, w ([batch][heads][seqlen][64] bf16), beta (fp32), log_f
 * (fp32 or NULL).  Outputs (caller-owned device memory):
 *   k_end   [batch][heads][seqlen][64] fp32: row j = k~_j, the key moved to the shard's end;
 *   q_start [batch][heads][seqlen][64] bf16: row i = z^_i, the query moved to the shard's start;
 *   t_shard [batch][heads][64][64] fp32: M^T, the transpose of the shard's product (row-major);
 *   with log_f (all three or none): a_q [batch][heads][seqlen] = inclusive prefix sums of log f,
 *   b_k = total - a_q, f_tot [batch][heads] = the total.
 * Computed from the UT preparation (split-precision fp32 chunk transforms, as the prefill hand-off)
 * by two fp32 walks over the chunks.  ws: path_cp_prepare_workspace_size bytes, 256-byte aligned,
 * contents unspecified on exit (a bounded wait of its preparation that gives up is recorded there
 * but not reported by a status call).
 * Errors: PATH_ERR_UNSUPPORTED outside the scope above; argument errors as elsewhere.
 */
int path_cp_shard_prepare(const path_attn_desc_t* desc, const void* q, const void* k, const void* w,
                          const float* beta, const float* log_f, float* k_end, void* q_start, float* t_shard,
                          float* a_q, float* b_k, float* f_tot, void* ws, size_t ws_bytes, void* stream);

/* Bytes of block scratch path_cp_attend_block needs for blocks of block_len keys; 0 if invalid. */
size_t path_cp_block_workspace_size(const path_attn_desc_t* desc, int block_len);

/*
 * Merges one earlier shard's key block into the softmax state that the forward's PREPARE phase left
 * in fwd_ws (path_attn_workspace_size(desc, 0 or 1) bytes, the same workspace the later SCAN phase
 * uses): for every local query i (row of q_start) and every block key j,
 *   s_ij = scale * k_block_j . q_start_i (+ a_q_i + b_k_j),
 * added to the query's running maximum, sum and weighted values with v_block_j.  k_block
 * [batch][heads][block_len][64] fp32 (rounded to bf16 for the tensor-core product), v_block the
 * same shape in bf16, a_q [..][seqlen] and b_k [..][block_len] fp32 or both NULL.  blk_ws:
 * path_cp_block_workspace_size bytes, 256-byte aligned.  Runs the forward scan kernel in its block
 * mode (tcgen05); its bounded waits report through path_attn_workspace_status on fwd_ws.
 */
int path_cp_attend_block(const path_attn_desc_t* desc, int block_len, const void* q_start, const float* k_block,
                         const void* v_block, const float* a_q, const float* b_k, void* fwd_ws, size_t fwd_ws_bytes,
                         void* blk_ws, size_t blk_ws_bytes, void* stream);

/*
 * Moves a key block through the local shard, in place: rows k_block <- k_block M (k_block
 * [batch][heads][block_len][64] fp32, t_shard = M^T from path_cp_shard_prepare), and with a forget
 * gate b_k += f_tot (b_k [batch][heads][block_len], f_tot [batch][heads]; both or neither).
 */
int path_cp_pass_block(const path_attn_desc_t* desc, int block_len, float* k_block, float* b_k,
                       const float* t_shard, const float* f_tot, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PATH_ATTN_H */
