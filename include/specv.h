/*
 * specv.h -- C ABI of the GB300 (sm_103a) speculative-sampling verification
 * and SSD outcome-prediction library (libspecv.so).
 *
 * Sources (page title -- section):
 *   "Speculative Speculative Decoding" (Kumar, Dao, May): §2.1 (accept test,
 *     residual r ∝ max(p_target - p_draft, 0), bonus token, verification
 *     outcome v_T = (k, t*)), §3.1 Algorithm 1 and the cache hit/miss
 *     definition, §4.1.1 (Saguaro outcome prediction: top-F_k draft tokens per
 *     lookahead k, excluding the token sent for verification there).
 *   "Speculative Decoding" (dl-note): §2.2-§2.3 (accept probability, residual
 *     distribution), Appendix (vLLM argument layout: one uniform per draft
 *     token, output [B, K+1], draft probability 0 rejects).
 *   "Lecture 5 - Speculative Decoding and SpecInfer": §2.1 (greedy and
 *     temperature sampling as adjusted distributions), §2.2 (accept iff
 *     u <= p(x)/q(x)), §2.7 (greedy special case), §3.1 (one iteration).
 *
 * Conventions shared by every entry point
 *   - All pointers are DEVICE pointers unless stated otherwise; the caller
 *     allocates and owns every buffer, including the workspace.  The library
 *     never allocates, frees or synchronises: work is enqueued on `stream`
 *     (a cudaStream_t passed as void*, NULL = legacy default stream) and the
 *     outputs are valid once the caller has synchronised that stream.
 *   - Logits are bf16 (raw 16-bit patterns) or fp32, rows contiguous along
 *     the vocabulary.  Row (b, i) starts at element b*batch_stride +
 *     i*row_stride of its tensor; strides are in elements and must be >= V
 *     (row_stride) and >= rows*row_stride (batch_stride).  A 16-byte aligned
 *     base and strides whose byte size is a multiple of 16 select the
 *     vectorised path; any other layout is accepted and read element-wise.
 *   - Argument errors are detected on the host, before any launch, and
 *     return SPECV_ERR_INVALID_ARG (nothing is written).  A failed launch
 *     returns SPECV_ERR_CUDA.  Data errors never trap: they are reported per
 *     batch row in the optional row_status output (bits below).  A flagged
 *     batch row gets accept length 0 and tokens -1 (and, in an SSD round, -1
 *     keys and no hit); specv_predict_outcomes gives -1 keys at the lookaheads
 *     whose draft row or sent token is invalid.
 *   - Launches.  specv_verify, specv_ssd_round, specv_saguaro_sample and
 *     specv_mss_verify are two kernels: one streaming pass over every logit
 *     (per-chunk statistics and candidates into the workspace), then one
 *     decision per batch row (launched as a programmatic dependent of the
 *     first).  The workspace needs no initialisation: everything a call
 *     reads from it is written earlier in the same call.  A call only
 *     enqueues kernels on the given stream, so it can be captured in a CUDA
 *     graph and replayed (on new inputs written into the same buffers).
 *   - Limits: 1 <= K <= 32, 0 <= B, 1 <= F <= 32, 1 <= V < 2^31 (in practice
 *     up to about 10^8: beyond that a CTA's table of partial sums no longer
 *     fits in shared memory and the call returns SPECV_ERR_UNSUPPORTED).
 */
#ifndef SPECV_H
#define SPECV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  SPECV_OK = 0,
  SPECV_ERR_INVALID_ARG = 1, /* bad pointer, size, stride or dtype */
  SPECV_ERR_UNSUPPORTED = 2, /* valid but outside what this build handles */
  SPECV_ERR_CUDA = 3,        /* a CUDA launch or attribute call failed */
  SPECV_ERR_WORKSPACE = 4    /* workspace NULL or smaller than required */
} specv_status;

typedef enum { SPECV_BF16 = 0, SPECV_FP32 = 1 } specv_dtype;

/* Per-batch-row status bits (row_status outputs). */
#define SPECV_ROW_BAD_TOKEN 1 /* a draft token outside [0, V) */
#define SPECV_ROW_NONFINITE 2 /* a NaN or +inf logit, or a row of all -inf */
#define SPECV_ROW_BAD_TEMP 4  /* temperature < 0, NaN or inf */
#define SPECV_ROW_FALLBACK 8  /* informational: the bonus draw fell back
                                 (zero residual mass -> drawn from p_n; or
                                 rounding left no index -> last v with r>0) */
#define SPECV_ROW_BAD_COUNT 32 /* per-row draft counts (cu_num_draft_tokens)
                                 give this row a count outside [0, K] or rows
                                 past num_draft_tokens; the row is read nowhere */
#define SPECV_ROW_DEVICE_TIMEOUT 16 /* a bulk copy of this row's logits into
                                 shared memory did not complete within about
                                 a second of device time; the kernel gave up on
                                 the row instead of waiting forever (not
                                 expected on a healthy GPU; for tests, the
                                 environment variable SPECV_TEST_STALL="A:<i>"
                                 or "B:<b>", read once per process, makes one
                                 such wait run out) */

/*
 * Verification of B independent batch rows ("Speculative Speculative
 * Decoding" §2.1; "Lecture 5" §3.1).
 *
 * For batch row b with temperature T = temperature[b] (same T for target and
 * draft; T = 0 is greedy):
 *   p_i = softmax(target row i / T), i in [0, K]     (one-hot argmax if T=0,
 *   q_i = softmax(draft row i / T),  i in [0, K)      ties -> lowest index)
 *   accept length n = the first i with NOT( q_i(x_i) > 0 and
 *       p_i(x_i) / q_i(x_i) >= uniforms[b, i] ), or K if there is none
 *       (greedy rows: accept iff x_i is the argmax of both rows i);
 *   bonus t* = the smallest v whose running sum of r in index order exceeds
 *       uniforms[b, K] * sum(r), where r = max(p_n - q_n, 0) if n < K and
 *       r = p_K if n = K (greedy rows: argmax of p_n).
 * Outputs: accept_len[b] = n; out_tokens[b, 0..K] = x_1..x_n, t*, then -1;
 *   optional p_draft[b, i] = p_i(x_i), q_draft[b, i] = q_i(x_i) for every
 *   i < K (fp32); optional row_status[b].
 */
typedef struct {
  int32_t B, K, V;
  int32_t dtype;                  /* specv_dtype */
  const void* target_logits;      /* K+1 rows per batch row */
  int64_t target_batch_stride;    /* elements */
  int64_t target_row_stride;      /* elements */
  const void* draft_logits;       /* K rows per batch row (a [B, K+1, V]
                                     SSD tensor is accepted: row K unused) */
  int64_t draft_batch_stride;
  int64_t draft_row_stride;
  const int32_t* draft_tokens;    /* [B, K] x_1..x_K */
  const float* temperature;       /* [B] */
  const float* uniforms;          /* [B, K+1] in [0,1): columns 0..K-1 drive
                                     the accept tests, column K the bonus */
  int32_t* accept_len;            /* OUT [B] */
  int32_t* out_tokens;            /* OUT [B, K+1] */
  float* p_draft;                 /* OUT, optional (NULL) [B, K] */
  float* q_draft;                 /* OUT, optional (NULL) [B, K] */
  int32_t* row_status;            /* OUT, optional (NULL) [B] */
  /* Per-row draft counts ("Speculative Decoding" dl-note, Appendix:
   * cu_num_draft_tokens).  Optional DEVICE [B]: inclusive prefix sums of the
   * draft counts K_b, 0 <= K_b <= K.  NULL: every row has K drafts in the
   * strided layout above.  When given, rows are packed along one axis and the
   * batch strides are ignored (c = cu[b-1], 0 for b = 0):
   *   target row (b, i), i <= K_b:  target_logits + (c + b + i) * target_row_stride
   *   draft row (b, i),  i <  K_b:  draft_logits + (c + i) * draft_row_stride
   *   draft_tokens[c + i], p_draft[c + i], q_draft[c + i]   (i < K_b)
   *   uniforms[c + b + i], i <= K_b (entry K_b drives the bonus);
   * accept_len and out_tokens keep their [B] and [B, K+1] shapes.  A row whose
   * counts fall outside [0, K] or past num_draft_tokens is flagged
   * SPECV_ROW_BAD_COUNT and read nowhere (its p_draft/q_draft are not
   * written).  Verification only (specv_verify, specv_verify_noalloc). */
  const int32_t* cu_num_draft_tokens;
  int32_t num_draft_tokens;       /* with cu: cu[B-1], the draft rows the packed
                                     buffers hold (target rows: that + B) */
  int32_t flags;                  /* SPECV_NO_DRAFT_PROBS or 0 */
} specv_verify_args;

/* flags: no draft distribution (dl-note Appendix, NO_DRAFT_PROBS: n-gram or
 * suffix drafts).  draft_logits must be NULL; q_i is taken one-hot at x_i, so
 * a draft is accepted iff p_i(x_i) >= uniforms[b, i] (greedy rows: iff x_i is
 * the argmax of p_i), q_draft reports 1, and after a rejection at n the bonus
 * is drawn from r = p_n with r(x_n) = 0.  Verification only. */
#define SPECV_NO_DRAFT_PROBS 1

/* Bytes of device workspace specv_verify needs for these sizes (0 if B=0). */
size_t specv_verify_workspace_bytes(int32_t B, int32_t K, int32_t V,
                                    int32_t dtype);

/* Enqueue verification.  workspace: device memory of at least
 * specv_verify_workspace_bytes(...) bytes, 256-byte aligned, owned by the
 * caller, not shared with a concurrently running call. */
specv_status specv_verify(const specv_verify_args* args, void* workspace,
                          size_t workspace_bytes, void* stream);

/*
 * Verification exactly as specv_verify, without a workspace argument.  The
 * pages have no counterpart: this entry point exists for callers that cannot
 * allocate device memory where they call the library -- a server that reserved
 * all free GPU memory for its KV cache at start-up, or a host language with no
 * CUDA allocator binding.  It calls no allocator at all.
 *
 * Its scratch is a fixed array of SPECV_NOALLOC_SCRATCH_BYTES bytes of device
 * memory built into the library; every GPU that loads the library holds one
 * copy until the process exits.  A call whose specv_verify_workspace_bytes()
 * exceeds it returns SPECV_ERR_UNSUPPORTED before any launch.  With the
 * default chunk sizes 8 MiB covers, e.g., B = 256, K = 8, V = 152064 fp32
 * (about 1.1 MB); the tuning variable SPECV_ITERS changes the chunk size,
 * hence the scratch a call needs, and a call it pushes past the limit is
 * refused the same way.
 *
 * The first call on a device looks up the scratch's device address
 * (cudaGetSymbolAddress, with that device current) and caches it per device
 * index for the life of the process; make that first call before any stream
 * capture.  The cache assumes one (primary) CUDA context per device that is
 * not reset: after cudaDeviceReset, or from a second context on the same
 * device, the cached address is stale -- do not call this entry point there.
 * All calls on a device share the one scratch array, which keeps the last
 * call's contents (nothing in it needs to start at zero): calls that can overlap on the GPU
 * -- other streams, other host threads -- race and corrupt each other's
 * results, so serialise them.
 */
#define SPECV_NOALLOC_SCRATCH_BYTES (8u << 20)
specv_status specv_verify_noalloc(const specv_verify_args* args, void* stream);

/*
 * One SSD round in a single pass over the logits ("Speculative Speculative
 * Decoding" §3.1 Algorithm 1, §4.1.1): verification exactly as specv_verify,
 * outcome keys exactly as specv_predict_outcomes (so draft_logits must hold
 * K+1 rows per batch row), and hit[b] as specv_check_hit on the realised
 * outcome.  Each draft row is read once and serves both q_i and the top-F
 * keys at lookahead i.  row_status (if given) also reports non-finite
 * logits in draft row K.
 */
typedef struct {
  specv_verify_args verify;  /* draft rows: K+1 per batch row */
  int32_t F;                 /* keys per lookahead, 1..32 (the width of keys) */
  int32_t* keys;             /* OUT [B, K+1, F] */
  float* key_logits;         /* OUT, optional [B, K+1, F] */
  uint8_t* hit;              /* OUT [B] */
  const int32_t* fanout;     /* optional HOST array [K+1]: keep only the first
                                fanout[k] keys at lookahead k (0..F; the rest
                                are -1), e.g. from specv_geometric_fanout.
                                NULL: F keys at every lookahead. */
  int32_t saguaro_F;         /* 0, or the drafts were sampled with Saguaro
                                sampling sigma_{saguaro_F, saguaro_C} (see
                                specv_saguaro_sample; 1 <= saguaro_F <= F): the
                                accept test and the residual then use
                                q_i = sigma(draft row i / T) instead of
                                softmax (greedy rows unaffected) */
  float saguaro_C;           /* in [0, 1] */
} specv_ssd_args;

size_t specv_ssd_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t F,
                                 int32_t dtype);
specv_status specv_ssd_round(const specv_ssd_args* args, void* workspace,
                             size_t workspace_bytes, void* stream);

/*
 * SSD outcome prediction ("Speculative Speculative Decoding" §4.1.1).
 * For every batch row b and lookahead k in [0, K]: keys[b, k, 0..F-1] are the
 * F largest logits of draft row k, ordered by (logit descending, index
 * ascending), with the draft token x_{k+1} = draft_tokens[b, k] removed for
 * k < K (it was sent for verification and cannot be the bonus); nothing is
 * removed at k = K.  Fewer than F candidates pad with -1.  The ranking is the
 * same for every temperature > 0 and for greedy, so no temperature is taken.
 */
typedef struct {
  int32_t B, K, V, F;
  int32_t dtype;
  const void* draft_logits;       /* K+1 rows per batch row */
  int64_t draft_batch_stride;
  int64_t draft_row_stride;
  const int32_t* draft_tokens;    /* [B, K] */
  int32_t* keys;                  /* OUT [B, K+1, F] */
  float* key_logits;              /* OUT, optional [B, K+1, F] (-inf pad) */
  int32_t* row_status;            /* OUT, optional [B] */
  const int32_t* fanout;          /* optional HOST [K+1], as in specv_ssd_args */
} specv_predict_args;

size_t specv_predict_workspace_bytes(int32_t B, int32_t K, int32_t V,
                                     int32_t F, int32_t dtype);
specv_status specv_predict_outcomes(const specv_predict_args* args,
                                    void* workspace, size_t workspace_bytes,
                                    void* stream);

/*
 * Draft-side Saguaro sampling ("Speculative Speculative Decoding" §4.2.1):
 * for each of B draft rows z (one lookahead of the drafter), with T =
 * temperature[b]:
 *   sigma_{F,C}(z/T)(t) is proportional to C * exp(z_t/T) for the F tokens of
 *   largest logit (ties to the lower index) and to exp(z_t/T) otherwise;
 *   tokens[b] = the smallest t whose running sum of sigma in index order
 *   exceeds uniforms[b] (T = 0: the first argmax, sigma not applied);
 *   q[b] = sigma(tokens[b]) (1 for greedy rows).
 * F = 0 samples softmax(z/T) itself.  A row with no mass left (C = 0 and every
 * finite logit in the top F) or a NaN / +inf logit gets token -1 and
 * SPECV_ROW_NONFINITE; a bad temperature SPECV_ROW_BAD_TEMP.  The drafts drawn
 * this way are verified with specv_ssd_args.saguaro_F / saguaro_C set to the
 * same F and C.
 */
typedef struct {
  int32_t B, V;
  int32_t dtype;             /* specv_dtype */
  const void* logits;        /* row b at logits + b * row_stride (elements) */
  int64_t row_stride;        /* >= V */
  const float* temperature;  /* [B] */
  int32_t F;                 /* 0..32 */
  float C;                   /* [0, 1] */
  const float* uniforms;     /* [B] in [0, 1) */
  int32_t* tokens;           /* OUT [B] */
  float* q;                  /* OUT, optional [B] */
  int32_t* row_status;       /* OUT, optional [B] */
} specv_saguaro_args;

size_t specv_saguaro_workspace_bytes(int32_t B, int32_t V, int32_t F, int32_t dtype);
specv_status specv_saguaro_sample(const specv_saguaro_args* args, void* workspace,
                                  size_t workspace_bytes, void* stream);

/*
 * Multi-step speculative sampling (MSS) at B token-tree nodes ("Lecture 5 -
 * Speculative Decoding and SpecInfer" §6.4; SpecInfer Theorems 4.2, 4.3).
 * Node b has a target row z_t and a draft row z_d (the draft model's logits
 * at that node), p = softmax(z_t/T), q = softmax(z_d/T), T = temperature[b],
 * and m_b candidate children x_0..x_{m_b-1} (candidates[b, 0..m_b-1]) that
 * the drafter drew independently from q.  The candidates are tested in
 * order: x_j is accepted iff q(x_j) > 0 and p_j(x_j)/q(x_j) >= u_j, where
 * p_0 = p and, after each rejection, p_{j+1} = norm(max(0, p_j - q)).  The
 * first accepted x_j is the node's token (accepted[b] = j); when all m_b are
 * rejected the token is the smallest v whose running sum of p_{m_b} exceeds
 * u_M (accepted[b] = -1).  u_j = uniforms[b, j], u_M = uniforms[b, M].  The
 * token's law is exactly p for any q; one candidate is plain speculative
 * sampling.  Greedy nodes (T = 0): the first candidate equal to argmax p is
 * accepted, else the token is argmax p (first maximum).
 * SPECV_MSS_NAIVE in flags: naive sampling, the correct rule when the
 * candidates were NOT drawn from q (e.g. the top-k of q): the token is drawn
 * from p by u_M and accepted[b] is the first j with x_j equal to it, or -1.
 * accept_prob[b, j] = min(1, p_j(x_j)/q(x_j)) for every tested candidate, 0
 * for the others (and under SPECV_MSS_NAIVE).
 * Row status: SPECV_ROW_BAD_TOKEN (a candidate outside [0, V)),
 * SPECV_ROW_BAD_COUNT (m_b outside [0, M]), SPECV_ROW_NONFINITE,
 * SPECV_ROW_BAD_TEMP, SPECV_ROW_DEVICE_TIMEOUT: the node gets token -1 and
 * accepted -1.  SPECV_ROW_FALLBACK (informational): a residual had no mass
 * (p_j <= q everywhere, reachable only by rounding), so the token was drawn
 * from p, or rounding left u_M past the end of the running sum.
 * All pointers are device pointers; target and draft rows 16-byte aligned
 * (base and strides) take the staged path, any other layout a slower one.
 * Each rejection costs one pass over the node's two rows.
 */
#define SPECV_MSS_NAIVE 1

typedef struct {
  int32_t B, M, V;             /* nodes; candidates per node (1..32); vocabulary */
  int32_t dtype;               /* specv_dtype */
  const void* target_logits;   /* node b's row at target_logits + b * target_row_stride */
  int64_t target_row_stride;   /* elements, >= V */
  const void* draft_logits;    /* node b's row at draft_logits + b * draft_row_stride */
  int64_t draft_row_stride;    /* elements, >= V */
  const int32_t* candidates;   /* [B, M] */
  const int32_t* num_candidates; /* optional [B]: m_b (NULL: every node has M) */
  const float* temperature;    /* [B] */
  const float* uniforms;       /* [B, M+1] in [0, 1) */
  int32_t flags;               /* 0 or SPECV_MSS_NAIVE */
  int32_t* accepted;           /* OUT [B] */
  int32_t* out_token;          /* OUT [B] */
  float* accept_prob;          /* OUT, optional [B, M] */
  int32_t* row_status;         /* OUT, optional [B] */
} specv_mss_args;

size_t specv_mss_workspace_bytes(int32_t B, int32_t M, int32_t V, int32_t dtype);
specv_status specv_mss_verify(const specv_mss_args* args, void* workspace,
                              size_t workspace_bytes, void* stream);

/*
 * Geometric fan-out ("Speculative Speculative Decoding" Theorem 12, proved in
 * Appendix A.2).  For a drafter with per-token acceptance rate a (0 < a < 1)
 * whose cache-miss probability at fan-out F is F^-r (r > 0), the fan-outs
 * maximising the hit rate under sum_k F_k <= budget are
 *   F_k = F_0 a^{k/(1+r)} for k < K,   F_K = F_0 a^{K/(1+r)} (1-a)^{-1/(1+r)},
 * with F_0 chosen so that they sum to budget.  The pages leave integer
 * rounding open: fanout[k] = floor(F_k), plus one for the lookaheads with the
 * largest fractional parts (lower k first on ties) until the budget is used,
 * then capped at max_f (so the sum is budget unless the cap binds).
 * Host-only: fanout (OUT [K+1]) and real (OUT, optional [K+1], the F_k before
 * rounding) are host arrays; no GPU work.  SPECV_ERR_INVALID_ARG on K outside
 * [1, 32], a outside (0, 1), r <= 0, budget < 0, max_f outside [0, 32] or a
 * NULL fanout.
 */
specv_status specv_geometric_fanout(int32_t K, double a, double r, int32_t budget,
                                    int32_t max_f, int32_t* fanout, double* real);

/*
 * Cache-hit check ("Speculative Speculative Decoding" §3.1: hit iff the
 * realised outcome (k, t*) is in the speculation cache).  hit[b] = 1 iff
 * 0 <= n <= K for n = accept_len[b] and out_tokens[b, n] is one of
 * keys[b, n, 0..F-1]; otherwise 0.  keys [B, K+1, F], accept_len [B],
 * out_tokens [B, K+1], hit [B] (uint8), all device pointers.
 */
specv_status specv_check_hit(int32_t B, int32_t K, int32_t F,
                             const int32_t* keys, const int32_t* accept_len,
                             const int32_t* out_tokens, uint8_t* hit,
                             void* stream);

/* Static description of a status code. */
const char* specv_status_string(specv_status s);

/* Message describing the most recent error on the calling host thread
 * ("" if none).  The string stays valid until that thread's next call. */
const char* specv_last_error(void);

/* Number of kernel launches the most recent successful call on this host
 * thread enqueued (for launch accounting in benchmarks). */
int32_t specv_last_launch_count(void);

/* Measurement hook.  While `event` (a cudaEvent_t created by the caller) is
 * set, every specv_verify / specv_ssd_round / specv_predict_outcomes /
 * specv_saguaro_sample / specv_mss_verify call made
 * by this host thread records it on its stream between the row-statistics
 * kernel and the decision kernel, so the two can be timed apart.  NULL clears
 * it.  The library does not create, own or destroy the event. */
void specv_set_split_event(void* event);

#ifdef __cplusplus
}
#endif

#endif /* SPECV_H */
