/*
 * PaTH attention — plain fp64 CPU oracle.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, __graft_entry__.smoke() and the cpu_baseline /
 * reference arm of bench.py may load this file's library.  It shares no code, header, table
 * or helper with the CUDA library; the product path never calls it.
 *
 * What it computes is the plain definition, one query row at a time, with no blocking, no
 * UT transform and no online softmax:
 *
 *   H_t = I - beta_t w_t w_t^T                      (reading notes cc.laoqi.cc 2505.16381, §2.1)
 *   logit(i,j) = scale * k_j^T H_{j+1} ... H_i q_i  (+ sum_{s=j+1..i} log f_s with PaTH-FoX, §2.5)
 *   A = causal softmax over j <= i,  o_i = sum_j A_ij v_j,  lse_i = log sum_j exp(logit(i,j))
 *
 * The product is evaluated right to left by walking j = i, i-1, ..., 0 with z = q_i:
 * score k_j . z, then z <- H_j z (H_j joins the path of every key left of j).  The softmax is
 * an exact two-pass one over the stored scores of the row.
 *
 * Readings of points the pages leave open:
 *   - scale multiplies the Householder-path logit only; the forget-gate bias is added unscaled
 *     (the notes omit the attention scale, §2.1);
 *   - beta is clamped to [0, 2] (the parameterisation's range, §2.1/2.2); values inside pass
 *     unchanged and the gradient returned is the one with respect to the clamped value;
 *   - w is used as given (not renormalised).
 *
 * Backward (absent from the pages): exact reverse-mode derivative of the same walk, per row.
 * Decode: the in-place key rewrite of the notes' §2.8 (Eq. (1)) followed by a plain
 * single-query softmax; with a forget gate the bias sum_{s=j+1..t} log f_s is carried as prefix
 * sums per cache row.  Prefill hand-off: the same rewrite applied to the prompt tokens in
 * order, so that every prompt key ends up transported to the prompt end (§2.8, last paragraph).
 *
 * Parallelism: OpenMP over independent query rows (and heads); no reduction order depends on
 * the thread count except the final sum of per-thread gradient buffers in oracle_bwd.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double clamp_beta(double b) { return b < 0.0 ? 0.0 : (b > 2.0 ? 2.0 : b); }

static double dot(const double* a, const double* b, int d) {
  double s = 0.0;
  for (int n = 0; n < d; ++n) s += a[n] * b[n];
  return s;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* Scores of row i of one head: s[j] for j = 0..i (scale and forget bias applied).
 * If zs != NULL it receives z_j = H_{j+1}...H_i q_i (the vector scored against k_j), [i+1][d]. */
static void row_scores(int d, const double* q, const double* k, const double* w,
                       const double* beta, const double* logf, double scale, int i,
                       double* s, double* z, double* zs) {
  memcpy(z, q + (size_t)i * d, sizeof(double) * d);
  double g = 0.0;
  for (int j = i; j >= 0; --j) {
    const double* kj = k + (size_t)j * d;
    const double* wj = w + (size_t)j * d;
    if (zs) memcpy(zs + (size_t)j * d, z, sizeof(double) * d);
    s[j] = scale * dot(kj, z, d) + g;
    const double c = clamp_beta(beta[j]) * dot(wj, z, d);
    for (int n = 0; n < d; ++n) z[n] -= c * wj[n];
    if (logf) g += logf[j];
  }
}

/* exact two-pass softmax of s[0..i]; writes p[0..i]; returns lse */
static double row_softmax(const double* s, int i, double* p) {
  double m = -INFINITY;
  for (int j = 0; j <= i; ++j) m = s[j] > m ? s[j] : m;
  double l = 0.0;
  for (int j = 0; j <= i; ++j) l += exp(s[j] - m);
  for (int j = 0; j <= i; ++j) p[j] = exp(s[j] - m) / l;
  return m + log(l);
}

/* Forward for selected rows of one head.  q,k,v,w: [L][d]; beta, logf: [L] (logf may be NULL).
 * rows: nrows indices (NULL = all rows 0..L-1, nrows ignored).  o: [nrows][d], lse: [nrows]. */
int oracle_fwd_head_rows(int L, int d, const double* q, const double* k, const double* v,
                         const double* w, const double* beta, const double* logf, double scale,
                         int nrows, const int* rows, double* o, double* lse) {
  if (L <= 0 || d <= 0) return 0;
  const int n = rows ? nrows : L;
  int bad = 0;
#pragma omp parallel
  {
    double* s = (double*)malloc(sizeof(double) * L);
    double* p = (double*)malloc(sizeof(double) * L);
    double* z = (double*)malloc(sizeof(double) * d);
    if (!s || !p || !z) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int r = 0; r < n; ++r) {
        const int i = rows ? rows[r] : r;
        if (i < 0 || i >= L) continue;
        row_scores(d, q, k, w, beta, logf, scale, i, s, z, NULL);
        lse[r] = row_softmax(s, i, p);
        double* orow = o + (size_t)r * d;
        for (int c = 0; c < d; ++c) orow[c] = 0.0;
        for (int j = 0; j <= i; ++j) {
          const double* vj = v + (size_t)j * d;
          for (int c = 0; c < d; ++c) orow[c] += p[j] * vj[c];
        }
      }
    }
    free(s); free(p); free(z);
  }
  return bad ? -1 : 0;
}

/* Forward for nheads independent heads laid out [nheads][L][d] (beta/logf [nheads][L]). */
int oracle_fwd(int nheads, int L, int d, const double* q, const double* k, const double* v,
               const double* w, const double* beta, const double* logf, double scale,
               double* o, double* lse) {
  for (int h = 0; h < nheads; ++h) {
    const size_t off = (size_t)h * L * d;
    int rc = oracle_fwd_head_rows(L, d, q + off, k + off, v + off, w + off, beta + (size_t)h * L,
                                  logf ? logf + (size_t)h * L : NULL, scale, L, NULL, o + off,
                                  lse + (size_t)h * L);
    if (rc) return rc;
  }
  return 0;
}

/* Full logit matrix of one head, S[i][j] (scale and bias applied), -INFINITY for j > i. */
int oracle_logits(int L, int d, const double* q, const double* k, const double* w,
                  const double* beta, const double* logf, double scale, double* S) {
  double* z = (double*)malloc(sizeof(double) * d);
  if (!z) return -1;
  for (int i = 0; i < L; ++i) {
    double* row = S + (size_t)i * L;
    row_scores(d, q, k, w, beta, logf, scale, i, row, z, NULL);
    for (int j = i + 1; j < L; ++j) row[j] = -INFINITY;
  }
  free(z);
  return 0;
}

/* Backward of one head.  Inputs as oracle_fwd_head_rows plus dO [L][d].  Outputs (overwritten):
 * dq, dk, dv, dw [L][d], dbeta [L], dlogf [L] (dlogf may be NULL; then not computed).
 *
 * Per row i (reverse mode of the walk):
 *   z_j = H_{j+1}..H_i q_i, s_j = scale k_j.z_j + g_ij, p = softmax(s), o_i = sum p_j v_j
 *   ds_j = p_j (dO_i.v_j - dO_i.o_i)
 *   dv_j += p_j dO_i;  dk_j += scale ds_j z_j
 *   zeta_{-1} = 0;  zeta_j = scale ds_j k_j + H_j zeta_{j-1}   (j = 0..i, gradient of z_j)
 *   dbeta_j -= (w_j.z_j)(w_j.zeta_{j-1});  dw_j -= beta_j[(w_j.z_j) zeta_{j-1} + (w_j.zeta_{j-1}) z_j]
 *   dq_i = zeta_i;   dlogf_s += sum_{j<s} ds_j for s = 1..i (bias sums log f over j < s <= i).
 */
int oracle_bwd_head(int L, int d, const double* q, const double* k, const double* v,
                    const double* w, const double* beta, const double* logf, double scale,
                    const double* dO, double* dq, double* dk, double* dv, double* dw,
                    double* dbeta, double* dlogf) {
  if (L <= 0 || d <= 0) return 0;
  memset(dq, 0, sizeof(double) * L * d);
  memset(dk, 0, sizeof(double) * L * d);
  memset(dv, 0, sizeof(double) * L * d);
  memset(dw, 0, sizeof(double) * L * d);
  memset(dbeta, 0, sizeof(double) * L);
  if (dlogf) memset(dlogf, 0, sizeof(double) * L);
  int bad = 0;
#pragma omp parallel
  {
    const size_t Ld = (size_t)L * d;
    double* s = (double*)malloc(sizeof(double) * L);
    double* p = (double*)malloc(sizeof(double) * L);
    double* ds = (double*)malloc(sizeof(double) * L);
    double* z = (double*)malloc(sizeof(double) * d);
    double* zeta = (double*)malloc(sizeof(double) * d);
    double* zs = (double*)malloc(sizeof(double) * Ld);
    double* o = (double*)malloc(sizeof(double) * d);
    double* tdk = (double*)calloc(Ld, sizeof(double));
    double* tdv = (double*)calloc(Ld, sizeof(double));
    double* tdw = (double*)calloc(Ld, sizeof(double));
    double* tdb = (double*)calloc(L, sizeof(double));
    double* tdf = (double*)calloc(L, sizeof(double));
    if (!s || !p || !ds || !z || !zeta || !zs || !o || !tdk || !tdv || !tdw || !tdb || !tdf) {
#pragma omp atomic write
      bad = 1;
    } else {
#pragma omp for schedule(dynamic, 4)
      for (int i = 0; i < L; ++i) {
        row_scores(d, q, k, w, beta, logf, scale, i, s, z, zs);
        (void)row_softmax(s, i, p);
        const double* dOi = dO + (size_t)i * d;
        for (int c = 0; c < d; ++c) o[c] = 0.0;
        for (int j = 0; j <= i; ++j)
          for (int c = 0; c < d; ++c) o[c] += p[j] * v[(size_t)j * d + c];
        const double Di = dot(dOi, o, d);
        for (int j = 0; j <= i; ++j) {
          const double dpj = dot(dOi, v + (size_t)j * d, d);
          ds[j] = p[j] * (dpj - Di);
          for (int c = 0; c < d; ++c) tdv[(size_t)j * d + c] += p[j] * dOi[c];
          const double* zj = zs + (size_t)j * d;
          for (int c = 0; c < d; ++c) tdk[(size_t)j * d + c] += scale * ds[j] * zj[c];
        }
        /* adjoint of the walk, ascending j */
        for (int c = 0; c < d; ++c) zeta[c] = 0.0;
        for (int j = 0; j <= i; ++j) {
          const double* wj = w + (size_t)j * d;
          const double* kj = k + (size_t)j * d;
          const double* zj = zs + (size_t)j * d;
          const double bj = clamp_beta(beta[j]);
          /* zeta currently holds zeta_{j-1} (gradient w.r.t. H_j z_j) */
          const double a = dot(wj, zj, d);
          const double b = dot(wj, zeta, d);
          tdb[j] -= a * b;
          for (int c = 0; c < d; ++c) tdw[(size_t)j * d + c] -= bj * (a * zeta[c] + b * zj[c]);
          /* zeta_j = H_j zeta_{j-1} + scale ds_j k_j */
          for (int c = 0; c < d; ++c) zeta[c] = zeta[c] - bj * b * wj[c] + scale * ds[j] * kj[c];
        }
        for (int c = 0; c < d; ++c) dq[(size_t)i * d + c] = zeta[c];
        if (dlogf) {
          double acc = 0.0;
          for (int sidx = 1; sidx <= i; ++sidx) {
            acc += ds[sidx - 1];
            tdf[sidx] += acc;
          }
        }
      }
#pragma omp critical
      {
        for (size_t n = 0; n < Ld; ++n) {
          dk[n] += tdk[n];
          dv[n] += tdv[n];
          dw[n] += tdw[n];
        }
        for (int n = 0; n < L; ++n) {
          dbeta[n] += tdb[n];
          if (dlogf) dlogf[n] += tdf[n];
        }
      }
    }
    free(s); free(p); free(ds); free(z); free(zeta); free(zs); free(o);
    free(tdk); free(tdv); free(tdw); free(tdb); free(tdf);
  }
  return bad ? -1 : 0;
}

/* One decode step for nheads heads (reading notes §2.8, Eq. (1)).
 * kc, vc: caches [nheads][cap][d], rows 0..t-1 valid; they are modified in place:
 *   k_j <- k_j - beta_t (w_t . k_j) w_t for j < t, then slot t <- (k_t, v_t) unchanged.
 * q_t,k_t,v_t,w_t: [nheads][d]; beta_t: [nheads]; o_t: [nheads][d]; lse_t: [nheads] or NULL. */
int oracle_decode_step(int nheads, int d, int cap, int t, double* kc, double* vc,
                       const double* q_t, const double* k_t, const double* v_t,
                       const double* w_t, const double* beta_t, double scale, double* o_t,
                       double* lse_t) {
  if (t < 0 || t + 1 > cap) return -2;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < nheads; ++h) {
    double* K = kc + (size_t)h * cap * d;
    double* V = vc + (size_t)h * cap * d;
    const double* w = w_t + (size_t)h * d;
    const double* q = q_t + (size_t)h * d;
    const double b = clamp_beta(beta_t[h]);
    for (int j = 0; j < t; ++j) {
      double* kj = K + (size_t)j * d;
      const double a = dot(w, kj, d);
      for (int n = 0; n < d; ++n) kj[n] -= b * a * w[n];
    }
    memcpy(K + (size_t)t * d, k_t + (size_t)h * d, sizeof(double) * d);
    memcpy(V + (size_t)t * d, v_t + (size_t)h * d, sizeof(double) * d);
    double* s = (double*)malloc(sizeof(double) * (t + 1));
    double* p = (double*)malloc(sizeof(double) * (t + 1));
    if (!s || !p) {
#pragma omp atomic write
      bad = 1;
    } else {
      for (int j = 0; j <= t; ++j) s[j] = scale * dot(K + (size_t)j * d, q, d);
      const double l = row_softmax(s, t, p);
      if (lse_t) lse_t[h] = l;
      double* o = o_t + (size_t)h * d;
      for (int n = 0; n < d; ++n) o[n] = 0.0;
      for (int j = 0; j <= t; ++j)
        for (int n = 0; n < d; ++n) o[n] += p[j] * V[(size_t)j * d + n];
    }
    free(s); free(p);
  }
  return bad ? -1 : 0;
}

/* Prefill -> decode hand-off for nheads heads (reading notes §2.8, last paragraph: after a
 * prefill every key is aligned to the prompt end).  The decode rewrite applied to the L prompt
 * tokens in order: for t = 0..L-1, k_j <- k_j - beta_t (w_t . k_j) w_t for every j < t, then
 * row t <- (k_t, v_t).  On return row j of kc holds H_{L-1} ... H_{j+1} k_j.
 * kc, vc: caches [nheads][cap][d] (rows 0..L-1 written, the rest untouched);
 * k, v, w: [nheads][L][d]; beta: [nheads][L] (clamped to [0, 2] like everywhere else). */
int oracle_prefill_cache(int nheads, int d, int cap, int L, double* kc, double* vc,
                         const double* k, const double* v, const double* w, const double* beta) {
  if (L < 0 || L > cap) return -2;
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < nheads; ++h) {
    double* K = kc + (size_t)h * cap * d;
    double* V = vc + (size_t)h * cap * d;
    for (int t = 0; t < L; ++t) {
      const double* wt = w + ((size_t)h * L + t) * d;
      const double b = clamp_beta(beta[(size_t)h * L + t]);
      for (int j = 0; j < t; ++j) {
        double* kj = K + (size_t)j * d;
        const double a = dot(wt, kj, d);
        for (int n = 0; n < d; ++n) kj[n] -= b * a * wt[n];
      }
      memcpy(K + (size_t)t * d, k + ((size_t)h * L + t) * d, sizeof(double) * d);
      memcpy(V + (size_t)t * d, v + ((size_t)h * L + t) * d, sizeof(double) * d);
    }
  }
  return 0;
}

/* Selected rows of the prefill hand-off, one key at a time (same rewrite as above, restricted to
 * the keys asked for): out[h][r] = H_{L-1} ... H_{j+1} k_j with j = rows[r], for every head h.
 * k, w: [nheads][L][d]; beta: [nheads][L]; rows: nrows indices in [0, L); out: [nheads][nrows][d]. */
int oracle_transport_keys(int nheads, int d, int L, int nrows, const int* rows, const double* k,
                          const double* w, const double* beta, double* out) {
  for (int r = 0; r < nrows; ++r)
    if (rows[r] < 0 || rows[r] >= L) return -2;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
  for (int h = 0; h < nheads; ++h) {
    for (int r = 0; r < nrows; ++r) {
      const int j = rows[r];
      double* o = out + ((size_t)h * nrows + r) * d;
      memcpy(o, k + ((size_t)h * L + j) * d, sizeof(double) * d);
      for (int t = j + 1; t < L; ++t) {
        const double* wt = w + ((size_t)h * L + t) * d;
        const double b = clamp_beta(beta[(size_t)h * L + t]);
        const double a = dot(wt, o, d);
        for (int n = 0; n < d; ++n) o[n] -= b * a * wt[n];
      }
    }
  }
  return 0;
}

/* One PaTH-FoX decode step for nheads heads (reading notes §2.8 Eq. (1) with the forget-gate bias
 * of §2.5): the keys are rewritten exactly as in oracle_decode_step, and the logit of cached key j
 * gains sum_{s=j+1..t} log f_s.  That sum is carried as prefix sums: ac[h][j] = sum_{s<=j} log f_s,
 * so the bias is ac[t] - ac[j]; the step stores ac[t] = ac[t-1] + log f_t (ac[-1] = 0).
 * ac: [nheads][cap] fp64, rows 0..t-1 valid on entry; logf_t: [nheads]; other arguments as in
 * oracle_decode_step. */
int oracle_decode_step_fox(int nheads, int d, int cap, int t, double* kc, double* vc, double* ac,
                           const double* q_t, const double* k_t, const double* v_t, const double* w_t,
                           const double* beta_t, const double* logf_t, double scale, double* o_t,
                           double* lse_t) {
  if (t < 0 || t + 1 > cap) return -2;
  int bad = 0;
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < nheads; ++h) {
    double* K = kc + (size_t)h * cap * d;
    double* V = vc + (size_t)h * cap * d;
    double* A = ac + (size_t)h * cap;
    const double* w = w_t + (size_t)h * d;
    const double* q = q_t + (size_t)h * d;
    const double b = clamp_beta(beta_t[h]);
    for (int j = 0; j < t; ++j) {
      double* kj = K + (size_t)j * d;
      const double a = dot(w, kj, d);
      for (int n = 0; n < d; ++n) kj[n] -= b * a * w[n];
    }
    memcpy(K + (size_t)t * d, k_t + (size_t)h * d, sizeof(double) * d);
    memcpy(V + (size_t)t * d, v_t + (size_t)h * d, sizeof(double) * d);
    A[t] = (t > 0 ? A[t - 1] : 0.0) + logf_t[h];
    double* s = (double*)malloc(sizeof(double) * (t + 1));
    double* p = (double*)malloc(sizeof(double) * (t + 1));
    if (!s || !p) {
#pragma omp atomic write
      bad = 1;
    } else {
      for (int j = 0; j <= t; ++j) s[j] = scale * dot(K + (size_t)j * d, q, d) + (A[t] - A[j]);
      const double l = row_softmax(s, t, p);
      if (lse_t) lse_t[h] = l;
      double* o = o_t + (size_t)h * d;
      for (int n = 0; n < d; ++n) o[n] = 0.0;
      for (int j = 0; j <= t; ++j)
        for (int n = 0; n < d; ++n) o[n] += p[j] * V[(size_t)j * d + n];
    }
    free(s); free(p);
  }
  return bad ? -1 : 0;
}
