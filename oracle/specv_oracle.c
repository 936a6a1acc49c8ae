/*
 * specv_oracle.c -- plain, slow, double-precision CPU statement of batched
 * speculative-sampling verification and SSD (Saguaro) outcome prediction.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or calls
 * this file: only the test suite, the smoke check and the benchmark's CPU
 * baseline leg do.  It shares no source, header, table or helper with the CUDA
 * library; the two meet only in the seeded input arrays.
 *
 * Sources (page title -- section):
 *   [SSD]  "Speculative Speculative Decoding" (Kumar, Dao, May) -- §2.1
 *          (accept rule, residual, bonus token, outcome v_T = (k, t*)),
 *          §3.1 Alg. 1 and the cache hit/miss definition, §4.1.1 (top-F_k
 *          outcome prediction excluding the sent draft token).
 *   [DLN]  "Speculative Decoding" (dl-note) -- §2.2 (accept probability),
 *          §2.3 (residual distribution), §3 (exactness), Appendix (vLLM
 *          convention: accept iff draft prob > 0 and p/q >= u).
 *   [CS349D] "Lecture 5 - Speculative Decoding and SpecInfer" -- §2.1
 *          (greedy and temperature as adjusted distributions), §2.2 (the rule
 *          u <= p(x)/q(x)), §2.7 (greedy special case), §3.1 (one iteration:
 *          residual at the first rejection, or a sample from p_{gamma+1}),
 *          §6.4 (multi-step speculative sampling over several candidates at
 *          one token-tree node, and naive sampling).
 *
 * Readings where the pages leave a step open (each one is listed in the
 * design notes):
 *   - temperature: p = softmax(z/T) computed as exp((z - max z)/T)/sum; the
 *     same T for target and draft of a batch row; T = 0 is greedy (one-hot at
 *     the FIRST maximum).
 *   - accept test at position i: accept iff q_i(x_i) > 0 and
 *     p_i(x_i)/q_i(x_i) >= U[i].  q_i(x_i) > 0 holds exactly when the draft
 *     logit of x_i is finite; the ratio is evaluated as exp(log p - log q) so
 *     that neither factor underflows.  Greedy rows do not consult U: with
 *     one-hot p and q the ratio is 1 iff x_i is the argmax of both rows.
 *   - bonus: r = max(p_n - q_n, 0) after a rejection at n, r = p_K if all K
 *     drafts are accepted; t* = the smallest v whose running sum of r in
 *     index order exceeds U[K] * sum(r).  If sum(r) is 0 the draw falls back
 *     to r = p_n; if rounding leaves no v, t* is the last v with r(v) > 0.
 *     Both fallbacks set ROW_FALLBACK.  Greedy bonus = argmax of p_n.
 *   - outcome prediction: keys at lookahead k are the F largest draft logits
 *     of draft row k, ordered by (logit descending, index ascending), with the
 *     token x_{k+1} that was sent for verification at that position removed
 *     (k < K); nothing is removed at k = K.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { OR_BF16 = 0, OR_FP32 = 1 };

/* Per-batch-row status bits (same meaning as the library's, defined here
 * independently). */
enum {
  ROW_BAD_TOKEN = 1,  /* a draft token outside [0, V) */
  ROW_NONFINITE = 2,  /* NaN or +inf logit, or a row with no finite logit */
  ROW_BAD_TEMP = 4,   /* temperature < 0, NaN or inf */
  ROW_FALLBACK = 8,   /* bonus draw used a fallback (informational) */
  ROW_BAD_COUNT = 32  /* a per-row draft or candidate count out of range */
};

/* Margin inside which an executed accept test or the bonus draw counts as a
 * boundary case: |U - p/q| < 1e-6, or U*R within 1e-6*R of a running sum. */
#define BOUNDARY_EPS 1e-6

static double load_logit(const void* base, int dtype, int64_t idx) {
  if (dtype == OR_FP32) return (double)((const float*)base)[idx];
  uint32_t bits = ((uint32_t)((const uint16_t*)base)[idx]) << 16;
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* ---------------------------------------------------------------------------
 * a1  Distribution of one vocabulary row: [CS349D] §2.1 (greedy = one-hot,
 *     temperature T = softmax(logits / T)).
 * Fills p[0..V-1], the first argmax, the max logit m and log of the softmax
 * normaliser S = sum_v exp((z_v - m)/T) (0 for greedy).  Returns status bits.
 */
static int row_distribution(const void* base, int dtype, int64_t off, int V,
                            double T, double* p, int* argmax, double* m_out,
                            double* logS_out) {
  int am = -1;
  double m = -INFINITY;
  for (int v = 0; v < V; ++v) {
    double z = load_logit(base, dtype, off + v);
    if (isnan(z) || z == INFINITY) return ROW_NONFINITE;
    if (z > m) { m = z; am = v; }
  }
  if (am < 0) return ROW_NONFINITE; /* every logit is -inf: no distribution */
  *argmax = am;
  *m_out = m;
  if (T == 0.0) {
    for (int v = 0; v < V; ++v) p[v] = (v == am) ? 1.0 : 0.0;
    *logS_out = 0.0;
    return 0;
  }
  double S = 0.0;
  for (int v = 0; v < V; ++v) {
    p[v] = exp((load_logit(base, dtype, off + v) - m) / T);
    S += p[v];
  }
  for (int v = 0; v < V; ++v) p[v] /= S;
  *logS_out = log(S);
  return 0;
}

/* Candidates of a row, ordered by (logit descending, index ascending). */
typedef struct { double z; int v; } cand_t;

static int cand_cmp(const void* a, const void* b) {
  const cand_t* x = (const cand_t*)a;
  const cand_t* y = (const cand_t*)b;
  if (x->z > y->z) return -1;
  if (x->z < y->z) return 1;
  return (x->v < y->v) ? -1 : (x->v > y->v);
}

/* ---------------------------------------------------------------------------
 * f2  Saguaro sampling scheme: [SSD] §4.2.1.  sigma_{F,C}(z) is proportional
 *     to C * exp(z_t) for the F tokens with the largest logits (top_F(z), in
 *     the key order above) and to exp(z_t) for every other token.  With a
 *     temperature the scheme applies to z / T (top_F is the same); greedy rows
 *     (T = 0) are left one-hot.  In: p[] = softmax(z/T) of the row (from
 *     row_distribution).  Out: p[] = sigma_{F,C}(z/T).  Returns 0, or
 *     ROW_NONFINITE when no mass is left (C = 0 and nothing outside top_F).
 */
static int saguaro_reweight(const void* base, int dtype, int64_t off, int V, int F, double C,
                            double* p, cand_t* c) {
  for (int v = 0; v < V; ++v) {
    c[v].z = load_logit(base, dtype, off + v);
    c[v].v = v;
  }
  qsort(c, (size_t)V, sizeof(cand_t), cand_cmp);
  for (int f = 0; f < F && f < V; ++f) p[c[f].v] *= C;
  double S = 0.0;
  for (int v = 0; v < V; ++v) S += p[v];
  if (!(S > 0.0)) return ROW_NONFINITE;
  for (int v = 0; v < V; ++v) p[v] /= S;
  return 0;
}

/* log p(v) for a temperature row, from the row's max and log-normaliser. */
static double log_prob(const void* base, int dtype, int64_t off, int v, double T,
                       double m, double logS) {
  return (load_logit(base, dtype, off + v) - m) / T - logS;
}

/* ---------------------------------------------------------------------------
 * Verification of one batch row.
 *   a2 accept scan: [DLN] §2.2 and Appendix; [CS349D] §2.2, §2.7, §3.1 step 3.
 *   a3 bonus: [SSD] §2.1 (residual r ∝ max(p_target - p_draft, 0), target
 *      itself when all drafts are accepted); [DLN] §2.3; [CS349D] §3.1 step 4.
 * Scratch: pt[(K+1)*V], qd[K*V], r[V].
 */
static void verify_row(int K, int V, int dtype, const void* target,
                       int64_t t_off, int64_t t_rs, const void* draft,
                       int64_t d_off, int64_t d_rs, const int32_t* x, double T,
                       const float* U, int no_draft, int sg_F, double sg_C,
                       int32_t* n_out, int32_t* tok_out,
                       double* p_out, double* q_out, double* alpha_out,
                       int32_t* status_out, int32_t* boundary_out, double* pt,
                       double* qd, double* r) {
  int status = 0;
  int boundary = 0;
  for (int i = 0; i <= K; ++i) tok_out[i] = -1;
  for (int i = 0; i < K; ++i) { p_out[i] = 0.0; q_out[i] = 0.0; alpha_out[i] = 0.0; }
  *n_out = 0;

  if (!(T >= 0.0) || isinf(T)) status |= ROW_BAD_TEMP;
  for (int i = 0; i < K; ++i)
    if (x[i] < 0 || x[i] >= V) status |= ROW_BAD_TOKEN;
  if (status) { *status_out = status; *boundary_out = 0; return; }

  int amt[64], amd[64];
  double mt[64], lst[64], md[64], lsd[64];
  for (int i = 0; i <= K; ++i)
    status |= row_distribution(target, dtype, t_off + (int64_t)i * t_rs, V, T,
                               pt + (int64_t)i * V, &amt[i], &mt[i], &lst[i]);
  for (int i = 0; i < K; ++i) {
    if (no_draft) {
      /* [DLN] Appendix, NO_DRAFT_PROBS: the draft probability of the sent
       * token is taken as 1, i.e. q_i is one-hot at x_i. */
      for (int v = 0; v < V; ++v) qd[(int64_t)i * V + v] = (v == x[i]) ? 1.0 : 0.0;
      amd[i] = x[i];
      continue;
    }
    status |= row_distribution(draft, dtype, d_off + (int64_t)i * d_rs, V, T,
                               qd + (int64_t)i * V, &amd[i], &md[i], &lsd[i]);
    /* Saguaro drafts were sampled from sigma_{F,C}: that is q ([SSD] §4.2.1) */
    if (sg_F > 0 && T > 0.0 && !status) {
      cand_t* cs = (cand_t*)malloc(sizeof(cand_t) * (size_t)V);
      status |= saguaro_reweight(draft, dtype, d_off + (int64_t)i * d_rs, V, sg_F, sg_C,
                                 qd + (int64_t)i * V, cs);
      free(cs);
    }
  }
  if (status) { *status_out = status; *boundary_out = 0; return; }

  /* Per-position p_i(x_i), q_i(x_i) and the overlap sum_v min(p_i, q_i)
   * ([SSD] §2.1 Theorem 1). */
  for (int i = 0; i < K; ++i) {
    const double* p = pt + (int64_t)i * V;
    const double* q = qd + (int64_t)i * V;
    p_out[i] = p[x[i]];
    q_out[i] = q[x[i]];
    double a = 0.0;
    for (int v = 0; v < V; ++v) a += (p[v] < q[v]) ? p[v] : q[v];
    alpha_out[i] = a;
  }

  /* a2: left-to-right accept test, stop at the first rejection. */
  int n = K;
  for (int i = 0; i < K; ++i) {
    int accept;
    if (T == 0.0) {
      accept = (x[i] == amd[i]) && (x[i] == amt[i]);
    } else {
      int64_t to = t_off + (int64_t)i * t_rs, dof = d_off + (int64_t)i * d_rs;
      double zdx = no_draft ? 0.0 : load_logit(draft, dtype, dof + x[i]);
      if (zdx == -INFINITY) {
        accept = 0; /* q_i(x_i) = 0: reject */
      } else {
        /* log q_i(x_i) = 0 without draft probabilities (q one-hot at x_i) */
        double lq = no_draft ? 0.0
                    : sg_F > 0 ? log(qd[(int64_t)i * V + x[i]])
                               : log_prob(draft, dtype, dof, x[i], T, md[i], lsd[i]);
        double ratio = exp(log_prob(target, dtype, to, x[i], T, mt[i], lst[i]) - lq);
        accept = ratio >= (double)U[i];
        if (fabs((double)U[i] - ratio) < BOUNDARY_EPS) boundary = 1;
      }
    }
    if (!accept) { n = i; break; }
  }

  /* a3: bonus token. */
  int tstar;
  if (T == 0.0) {
    tstar = amt[n]; /* residual of two one-hots, or p_{K+1}: argmax of p_n */
  } else {
    const double* p = pt + (int64_t)n * V;
    double R = 0.0;
    if (n < K) {
      const double* q = qd + (int64_t)n * V;
      for (int v = 0; v < V; ++v) { r[v] = p[v] > q[v] ? p[v] - q[v] : 0.0; R += r[v]; }
    } else {
      for (int v = 0; v < V; ++v) { r[v] = p[v]; R += r[v]; }
    }
    if (!(R > 0.0)) {
      status |= ROW_FALLBACK;
      R = 0.0;
      for (int v = 0; v < V; ++v) { r[v] = p[v]; R += r[v]; }
    }
    double tau = (double)U[K] * R;
    double cum = 0.0, prev = 0.0;
    tstar = -1;
    for (int v = 0; v < V; ++v) {
      prev = cum;
      cum += r[v];
      if (cum > tau) { tstar = v; break; }
    }
    if (tstar < 0) {
      status |= ROW_FALLBACK;
      for (int v = V - 1; v >= 0; --v) if (r[v] > 0.0) { tstar = v; break; }
      boundary = 1;
    } else if (fabs(tau - prev) < BOUNDARY_EPS * R || fabs(cum - tau) < BOUNDARY_EPS * R) {
      boundary = 1;
    }
  }

  *n_out = n;
  for (int i = 0; i < n; ++i) tok_out[i] = x[i];
  tok_out[n] = tstar;
  *status_out = status;
  *boundary_out = boundary;
}

/* Exported: verification of B batch rows.  Logit layouts are
 *   target[b*t_bs + i*t_rs + v], i in [0, K]     (K+1 target rows)
 *   draft [b*d_bs + i*d_rs + v], i in [0, K)     (K draft rows)
 * Outputs: accept_len[B], out_tokens[B*(K+1)] (-1 padded), p_out/q_out/
 * alpha_out[B*K], row_status[B], boundary[B].  nthreads <= 0 uses all. */
int specv_oracle_verify(int B, int K, int V, int dtype, const void* target,
                        int64_t t_bs, int64_t t_rs, const void* draft,
                        int64_t d_bs, int64_t d_rs, const int32_t* tokens,
                        const float* temperature, const float* uniforms, int no_draft,
                        int sg_F, double sg_C,
                        int32_t* accept_len, int32_t* out_tokens, double* p_out,
                        double* q_out, double* alpha_out, int32_t* row_status,
                        int32_t* boundary, int nthreads) {
  if (B < 0 || K < 1 || K > 63 || V < 1 || sg_F < 0 || !(sg_C >= 0.0 && sg_C <= 1.0)) return 1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int b = 0; b < B; ++b) {
    double* pt = (double*)malloc(sizeof(double) * (size_t)(K + 1) * V);
    double* qd = (double*)malloc(sizeof(double) * (size_t)K * V);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    verify_row(K, V, dtype, target, (int64_t)b * t_bs, t_rs, draft,
               (int64_t)b * d_bs, d_rs, tokens + (int64_t)b * K,
               (double)temperature[b], uniforms + (int64_t)b * (K + 1), no_draft, sg_F, sg_C,
               accept_len + b, out_tokens + (int64_t)b * (K + 1),
               p_out + (int64_t)b * K, q_out + (int64_t)b * K,
               alpha_out + (int64_t)b * K, row_status + b, boundary + b, pt, qd, r);
    free(pt);
    free(qd);
    free(r);
  }
  (void)nthreads;
  return 0;
}

/* Exported: verification with a per-row draft count ([DLN] Appendix,
 * cu_num_draft_tokens).  Row b has K_b = cu[b] - cu[b-1] drafts (cu[-1] = 0),
 * 0 <= K_b <= Kmax, packed along one axis:
 *   draft row (b, i)  at draft [(cu[b-1] + i) * d_rs],      i < K_b
 *   target row (b, i) at target[(cu[b-1] + b + i) * t_rs],  i <= K_b
 *   tokens x_{b,i} at tokens[cu[b-1] + i]; uniforms at uniforms[cu[b-1] + b + i],
 *   i <= K_b (the last drives the bonus).
 * Outputs: accept_len[B], out_tokens[B*(Kmax+1)] (-1 padded), p_out/q_out/
 * alpha_out[num_tokens] (packed like the tokens), row_status[B] (bit 32: K_b
 * outside [0, Kmax]), boundary[B].  cu is a host array here. */
int specv_oracle_verify_ragged(int B, int Kmax, int V, int dtype, const void* target,
                               int64_t t_rs, const void* draft, int64_t d_rs,
                               const int32_t* cu, const int32_t* tokens,
                               const float* temperature, const float* uniforms, int no_draft,
                               int32_t* accept_len, int32_t* out_tokens, double* p_out,
                               double* q_out, double* alpha_out, int32_t* row_status,
                               int32_t* boundary, int nthreads) {
  if (B < 0 || Kmax < 0 || Kmax > 63 || V < 1) return 1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int b = 0; b < B; ++b) {
    const int64_t c0 = b == 0 ? 0 : cu[b - 1];
    const int kb = (int)(cu[b] - c0);
    int32_t* ot = out_tokens + (int64_t)b * (Kmax + 1);
    for (int i = 0; i <= Kmax; ++i) ot[i] = -1;
    if (kb < 0 || kb > Kmax) {
      accept_len[b] = 0;
      row_status[b] = ROW_BAD_COUNT;
      boundary[b] = 0;
      continue;
    }
    double* pt = (double*)malloc(sizeof(double) * (size_t)(kb + 1) * V);
    double* qd = (double*)malloc(sizeof(double) * (size_t)(kb > 0 ? kb : 1) * V);
    double* r = (double*)malloc(sizeof(double) * (size_t)V);
    verify_row(kb, V, dtype, target, (c0 + b) * t_rs, t_rs, draft, c0 * d_rs, d_rs,
               tokens + c0, (double)temperature[b], uniforms + c0 + b, no_draft, 0, 1.0,
               accept_len + b, ot, p_out + c0, q_out + c0, alpha_out + c0,
               row_status + b, boundary + b, pt, qd, r);
    free(pt);
    free(qd);
    free(r);
  }
  (void)nthreads;
  return 0;
}

/* Exported: draft-side Saguaro sampling ([SSD] §4.2.1): for each of B rows
 * (z[b*z_bs + v]), the token t = the smallest v whose running sum of
 * sigma_{F,C}(z/T) exceeds U[b] (T = 0: the first argmax), and q_out[b] =
 * sigma(t).  F = 0 samples softmax(z/T) itself. */
int specv_oracle_saguaro_sample(int B, int V, int dtype, const void* z, int64_t z_bs,
                                const float* temperature, int F, double C, const float* U,
                                int32_t* tokens, double* q_out, int32_t* row_status) {
  if (B < 0 || V < 1 || F < 0 || !(C >= 0.0 && C <= 1.0)) return 1;
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1)
#endif
  for (int b = 0; b < B; ++b) {
    double* p = (double*)malloc(sizeof(double) * (size_t)V);
    cand_t* cs = (cand_t*)malloc(sizeof(cand_t) * (size_t)V);
    const double T = (double)temperature[b];
    int am;
    double m, ls;
    int st = (!(T >= 0.0) || isinf(T)) ? ROW_BAD_TEMP : 0;
    if (!st) st = row_distribution(z, dtype, (int64_t)b * z_bs, V, T, p, &am, &m, &ls);
    if (!st && F > 0 && T > 0.0) st = saguaro_reweight(z, dtype, (int64_t)b * z_bs, V, F, C, p, cs);
    tokens[b] = -1;
    q_out[b] = 0.0;
    row_status[b] = st;
    if (st || T == 0.0) {
      if (!st) {
        tokens[b] = am;
        q_out[b] = 1.0;
      }
      free(p);
      free(cs);
      continue;
    }
    double cum = 0.0;
    for (int v = 0; v < V; ++v) {
      cum += p[v];
      if (cum > (double)U[b]) { tokens[b] = v; break; }
    }
    if (tokens[b] < 0) {  /* U at the top end after rounding: the last v with mass */
      for (int v = V - 1; v >= 0; --v) if (p[v] > 0.0) { tokens[b] = v; break; }
      row_status[b] |= ROW_FALLBACK;
    }
    q_out[b] = p[tokens[b]];
    free(p);
    free(cs);
  }
  return 0;
}

/* Exported: sigma_{F,C}(z/T) of one row, for the pins. */
int specv_oracle_saguaro_probs(int V, int dtype, const void* row, double T, int F, double C,
                               double* p) {
  int am;
  double m, ls;
  int st = row_distribution(row, dtype, 0, V, T, p, &am, &m, &ls);
  if (st || T == 0.0 || F == 0) return st;
  cand_t* cs = (cand_t*)malloc(sizeof(cand_t) * (size_t)V);
  st = saguaro_reweight(row, dtype, 0, V, F, C, p, cs);
  free(cs);
  return st;
}

/* Exported: the a1 distribution of one row, for the pins. */
int specv_oracle_row_probs(int V, int dtype, const void* row, double T,
                           double* p) {
  int am;
  double m, ls;
  return row_distribution(row, dtype, 0, V, T, p, &am, &m, &ls);
}

/* ---------------------------------------------------------------------------
 * a4  Outcome prediction: [SSD] §4.1.1 ("Saguaro verification-outcome
 *     prediction"): at every lookahead k take the top-F_k tokens of the draft
 *     logits, excluding the token sent for verification at that position.
 *     Full sort of the candidates; no partial selection.
 */

int specv_oracle_predict(int B, int K, int V, int F, int dtype,
                         const void* draft, int64_t d_bs, int64_t d_rs,
                         const int32_t* tokens, const int32_t* fanout,
                         int32_t* keys, float* key_logits,
                         int32_t* row_status, int nthreads) {
  if (B < 0 || K < 1 || V < 1 || F < 1) return 1;
  if (fanout)
    for (int k = 0; k <= K; ++k)
      if (fanout[k] < 0 || fanout[k] > F) return 1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int b = 0; b < B; ++b) {
    cand_t* c = (cand_t*)malloc(sizeof(cand_t) * (size_t)V);
    int status = 0;
    for (int k = 0; k <= K; ++k) {
      int32_t* kk = keys + ((int64_t)b * (K + 1) + k) * F;
      float* kl = key_logits + ((int64_t)b * (K + 1) + k) * F;
      for (int f = 0; f < F; ++f) { kk[f] = -1; kl[f] = -INFINITY; }
      int excl = -1;
      if (k < K) {
        excl = tokens[(int64_t)b * K + k];
        if (excl < 0 || excl >= V) { status |= ROW_BAD_TOKEN; continue; }
      }
      int64_t off = (int64_t)b * d_bs + (int64_t)k * d_rs;
      int nc = 0, bad = 0;
      for (int v = 0; v < V; ++v) {
        double z = load_logit(draft, dtype, off + v);
        if (isnan(z) || z == INFINITY) { bad = 1; break; }
        if (v == excl) continue;
        c[nc].z = z;
        c[nc].v = v;
        ++nc;
      }
      if (bad) { status |= ROW_NONFINITE; continue; }
      qsort(c, (size_t)nc, sizeof(cand_t), cand_cmp);
      /* per-lookahead fan-out F_k (SSD Theorem 12) keeps the first F_k keys */
      const int Fk = fanout ? fanout[k] : F;
      for (int f = 0; f < Fk && f < nc; ++f) { kk[f] = c[f].v; kl[f] = (float)c[f].z; }
    }
    row_status[b] = status;
    free(c);
  }
  (void)nthreads;
  return 0;
}

/* ---------------------------------------------------------------------------
 * f1  Geometric fan-out: [SSD] Theorem 12 (Saguaro cache shape), proved in
 *     Appendix A.2 (Theorem 18).  For a drafter with acceptance rate a and an
 *     r-th power-law cache hit rate (miss probability F^-r), the F_k that
 *     maximise the hit rate under sum_k F_k <= budget are
 *       F_k = F_0 a^{k/(1+r)}                       for k < K,
 *       F_K = F_0 a^{K/(1+r)} (1 - a)^{-1/(1+r)},
 *       F_0 = budget / (a^{K/(1+r)} (1-a)^{-1/(1+r)}
 *                       + (1 - a^{K/(1+r)}) / (1 - a^{1/(1+r)})),
 *     so that the F_k sum to the budget.  The pages leave integer rounding
 *     open; the reading taken here: floor every F_k, give the budget left
 *     over to the lookaheads with the largest fractional parts (lower k first
 *     on ties), then cap each at max_f.  real[] (optional) receives F_k.
 *     Returns 0, or 1 on arguments outside 0 < a < 1, r > 0, K >= 1,
 *     budget >= 0, max_f >= 0.
 */
int specv_oracle_geometric_fanout(int K, double a, double r, int budget, int max_f,
                                  double* real, int32_t* fk) {
  if (K < 1 || !(a > 0.0 && a < 1.0) || !(r > 0.0) || budget < 0 || max_f < 0) return 1;
  const double g = 1.0 / (1.0 + r);
  const double aK = pow(a, K * g);
  const double F0 = budget / (aK * pow(1.0 - a, -g) + (1.0 - aK) / (1.0 - pow(a, g)));
  double* x = (double*)malloc(sizeof(double) * (size_t)(K + 1));
  int used = 0;
  for (int k = 0; k <= K; ++k) {
    x[k] = (k < K) ? F0 * pow(a, k * g) : F0 * aK * pow(1.0 - a, -g);
    if (real) real[k] = x[k];
    fk[k] = (int32_t)floor(x[k]);
    used += fk[k];
  }
  for (int left = budget - used; left > 0; --left) {
    int best = -1;
    double best_frac = -1.0;
    for (int k = 0; k <= K; ++k) {
      const double frac = x[k] - floor(x[k]);
      if (fk[k] == (int32_t)floor(x[k]) && frac > best_frac) { best = k; best_frac = frac; }
    }
    if (best < 0) break;
    fk[best] += 1;
  }
  for (int k = 0; k <= K; ++k)
    if (fk[k] > max_f) fk[k] = max_f;
  free(x);
  return 0;
}

/* ---------------------------------------------------------------------------
 * a5  Cache hit: [SSD] §3.1, hit iff the realised outcome v_T = (k, t*) is in
 *     the speculation cache S_T, i.e. t* is among the keys predicted for
 *     accept length k.
 */
void specv_oracle_check_hit(int B, int K, int F, const int32_t* keys,
                            const int32_t* accept_len, const int32_t* out_tokens,
                            uint8_t* hit) {
  for (int b = 0; b < B; ++b) {
    int n = accept_len[b];
    hit[b] = 0;
    if (n < 0 || n > K) continue;
    int t = out_tokens[(int64_t)b * (K + 1) + n];
    if (t < 0) continue;
    const int32_t* kk = keys + ((int64_t)b * (K + 1) + n) * F;
    for (int f = 0; f < F; ++f)
      if (kk[f] == t) { hit[b] = 1; break; }
  }
}

/* ---------------------------------------------------------------------------
 * a6  Multi-step speculative sampling (MSS) at one node of a token tree,
 *     [CS349D] §6.4 (SpecInfer Theorem 4.2 / 4.3).  The node's candidates
 *     x_1..x_m (children drawn independently from the draft distribution q of
 *     the node) are tested in order: x_j is accepted iff q(x_j) > 0 and
 *     p_j(x_j) / q(x_j) >= u_j, with p_1 = p (the target distribution of the
 *     node) and, after each rejection, p_{j+1} = norm(max(0, p_j - q)).  If
 *     all m are rejected the token is drawn from p_{m+1} by inverse CDF of
 *     the node's last uniform.  One candidate is plain speculative sampling.
 *     Naive sampling (NS, same section), the rule for candidates that were
 *     not drawn from q (e.g. the top-k of q): one draw y ~ p by inverse CDF of
 *     the last uniform, a candidate is accepted iff it equals y.
 *
 * Readings (listed in the design notes):
 *   - T = 0 (greedy): the first candidate equal to argmax p is accepted, else
 *     the token is argmax p ([CS349D] §6.4, greedy verification follows the
 *     target's argmax); NS gives the same result.
 *   - a residual with no mass (p_j <= q everywhere, reachable only through
 *     rounding or q(x_j) = 0) ends the testing: the token is drawn from p and
 *     ROW_FALLBACK is set, as for the single-draft bonus.
 *   - accept_prob[j] = min(1, p_j(x_j)/q(x_j)) for every tested candidate
 *     (0 when q(x_j) = 0), 0 for the untested ones and under NS.
 */

/* Inverse-CDF draw from the unnormalised r[0..V-1] with uniform U: the
 * smallest v whose running sum exceeds U*sum(r); the last v with r > 0 when
 * rounding leaves none (sets *fb).  *bd is set when U*sum(r) lies within
 * BOUNDARY_EPS*sum(r) of a running sum next to the chosen v. */
static int icdf_draw(const double* r, int V, double U, int* fb, int* bd) {
  double R = 0.0;
  for (int v = 0; v < V; ++v) R += r[v];
  double tau = U * R, cum = 0.0, prev = 0.0;
  for (int v = 0; v < V; ++v) {
    prev = cum;
    cum += r[v];
    if (cum > tau) {
      if (fabs(tau - prev) < BOUNDARY_EPS * R || fabs(cum - tau) < BOUNDARY_EPS * R) *bd = 1;
      return v;
    }
  }
  *fb = 1;
  *bd = 1;
  for (int v = V - 1; v >= 0; --v) if (r[v] > 0.0) return v;
  return -1;
}

/* One node from its distributions p, q (T > 0).  Scratch pj[V], r[V]. */
static void mss_node(int V, const double* p, const double* q, const int32_t* x, int m,
                     const float* U, int M, int naive, int32_t* acc_out, int32_t* tok_out,
                     double* aprob, int* status, int* boundary, double* pj, double* r) {
  int fb = 0;
  *acc_out = -1;
  for (int j = 0; j < M; ++j) aprob[j] = 0.0;
  if (naive) {
    *tok_out = icdf_draw(p, V, (double)U[M], &fb, boundary);
    for (int j = 0; j < m; ++j)
      if (x[j] == *tok_out) { *acc_out = j; break; }
    if (fb) *status |= ROW_FALLBACK;
    return;
  }
  memcpy(pj, p, sizeof(double) * (size_t)V);
  for (int j = 0; j < m; ++j) {
    const double qx = q[x[j]];
    const double ratio = qx > 0.0 ? pj[x[j]] / qx : 0.0;
    aprob[j] = ratio < 1.0 ? ratio : 1.0;
    if (qx > 0.0 && fabs((double)U[j] - ratio) < BOUNDARY_EPS) *boundary = 1;
    if (qx > 0.0 && ratio >= (double)U[j]) {
      *acc_out = j;
      *tok_out = x[j];
      return;
    }
    /* rejected: p_{j+1} = norm(max(0, p_j - q)) */
    double Z = 0.0;
    for (int v = 0; v < V; ++v) { r[v] = pj[v] > q[v] ? pj[v] - q[v] : 0.0; Z += r[v]; }
    if (!(Z > 0.0)) {  /* no residual mass: draw from p itself */
      *status |= ROW_FALLBACK;
      *tok_out = icdf_draw(p, V, (double)U[M], &fb, boundary);
      if (fb) *status |= ROW_FALLBACK;
      return;
    }
    for (int v = 0; v < V; ++v) pj[v] = r[v] / Z;
  }
  *tok_out = icdf_draw(pj, V, (double)U[M], &fb, boundary);
  if (fb) *status |= ROW_FALLBACK;
}

/* Exported: MSS (naive = 0) or NS (naive = 1) at B nodes.  Layouts:
 *   target[b*t_rs + v], draft[b*d_rs + v]      one row each per node
 *   cands[b*M + j], j < m_b = num_cands ? num_cands[b] : M (0 <= m_b <= M)
 *   uniforms[b*(M+1) + j]: u_j for candidate j < M, u_M for the draw
 * Outputs: accepted[B] (candidate index or -1), token[B], accept_prob[B*M],
 * row_status[B] (ROW_BAD_COUNT for a count outside [0, M]), boundary[B]. */
int specv_oracle_mss(int B, int M, int V, int dtype, const void* target, int64_t t_rs,
                     const void* draft, int64_t d_rs, const int32_t* cands,
                     const int32_t* num_cands, const float* temperature, const float* uniforms,
                     int naive, int32_t* accepted, int32_t* token, double* accept_prob,
                     int32_t* row_status, int32_t* boundary, int nthreads) {
  if (B < 0 || M < 0 || M > 32 || V < 1) return 1;
#ifdef _OPENMP
  if (nthreads <= 0) nthreads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads)
#endif
  for (int b = 0; b < B; ++b) {
    const int32_t* x = cands + (int64_t)b * M;
    const float* U = uniforms + (int64_t)b * (M + 1);
    const double T = (double)temperature[b];
    const int m = num_cands ? num_cands[b] : M;
    int st = 0, bd = 0;
    accepted[b] = -1;
    token[b] = -1;
    for (int j = 0; j < M; ++j) accept_prob[(int64_t)b * M + j] = 0.0;
    if (!(T >= 0.0) || isinf(T)) st |= ROW_BAD_TEMP;
    if (m < 0 || m > M) st |= ROW_BAD_COUNT;
    else
      for (int j = 0; j < m; ++j)
        if (x[j] < 0 || x[j] >= V) st |= ROW_BAD_TOKEN;
    double* p = (double*)malloc(sizeof(double) * (size_t)V * 4);
    double *q = p + V, *pj = p + 2 * (size_t)V, *r = p + 3 * (size_t)V;
    int amt = -1, amd = -1;
    double mt, lst, md, lsd;
    if (!st) st |= row_distribution(target, dtype, (int64_t)b * t_rs, V, T, p, &amt, &mt, &lst);
    if (!st) st |= row_distribution(draft, dtype, (int64_t)b * d_rs, V, T, q, &amd, &md, &lsd);
    if (!st) {
      if (T == 0.0) {
        token[b] = amt;
        for (int j = 0; j < m; ++j) {
          if (!naive) accept_prob[(int64_t)b * M + j] = (x[j] == amt) ? 1.0 : 0.0;
          if (x[j] == amt) { accepted[b] = j; break; }
        }
      } else {
        mss_node(V, p, q, x, m, U, M, naive, accepted + b, token + b,
                 accept_prob + (int64_t)b * M, &st, &bd, pj, r);
      }
    }
    row_status[b] = st;
    boundary[b] = bd;
    free(p);
  }
  (void)nthreads;
  return 0;
}

/* Exported, for the pins: the exact law of the node's output token given one
 * candidate tuple x[0..m-1] and the distributions p, q (not logits):
 *   law[y] = sum_j (prod_{i<j} (1 - a_i)) a_j [y = x_j] + prod_j (1 - a_j) p_{m+1}(y)
 * with a_j = min(1, p_j(x_j)/q(x_j)) (0 if q(x_j) = 0) for MSS, and
 * law = p for NS.  Also the probability that some candidate is accepted.
 * Returns 1 if a residual has no mass (the law is then undefined). */
int specv_oracle_mss_law(int V, const double* p, const double* q, const int32_t* x, int m,
                         int naive, double* law, double* p_accept) {
  if (naive) {
    double pa = 0.0;
    for (int v = 0; v < V; ++v) {
      law[v] = p[v];
      int in = 0;
      for (int j = 0; j < m; ++j) in |= (x[j] == v);
      if (in) pa += p[v];
    }
    *p_accept = pa;
    return 0;
  }
  double* pj = (double*)malloc(sizeof(double) * (size_t)V * 2);
  double* r = pj + V;
  memcpy(pj, p, sizeof(double) * (size_t)V);
  for (int v = 0; v < V; ++v) law[v] = 0.0;
  double reach = 1.0; /* probability that candidates 1..j-1 were all rejected */
  for (int j = 0; j < m; ++j) {
    const double qx = q[x[j]];
    double a = qx > 0.0 ? pj[x[j]] / qx : 0.0;
    if (a > 1.0) a = 1.0;
    law[x[j]] += reach * a;
    reach *= 1.0 - a;
    double Z = 0.0;
    for (int v = 0; v < V; ++v) { r[v] = pj[v] > q[v] ? pj[v] - q[v] : 0.0; Z += r[v]; }
    if (!(Z > 0.0)) {
      free(pj);
      *p_accept = 1.0 - reach;
      return reach > 0.0 ? 1 : 0;  /* unreachable residual: harmless */
    }
    for (int v = 0; v < V; ++v) pj[v] = r[v] / Z;
  }
  for (int v = 0; v < V; ++v) law[v] += reach * pj[v];
  *p_accept = 1.0 - reach;
  free(pj);
  return 0;
}
