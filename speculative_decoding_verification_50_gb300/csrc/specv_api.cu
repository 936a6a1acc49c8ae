// C ABI of libspecv (declared in include/specv.h): argument checks, workspace
// sizing, cluster-size choice and kernel launches on the caller's stream.
#include <algorithm>
#include <cmath>
#include <atomic>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <mutex>
#include <string>

#include "specv.h"
#include "launch.cuh"

using namespace specv;

namespace {

thread_local std::string g_err;
thread_local int32_t g_launches = 0;
thread_local cudaEvent_t g_split_event = nullptr;  // measurement hook

// Records the caller's split event (if any) between the statistics kernel and
// the decision kernel.
cudaError_t record_split(cudaStream_t s) {
  return g_split_event ? cudaEventRecord(g_split_event, s) : cudaSuccess;
}

specv_status fail(specv_status s, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return s;
}

specv_status ok() {
  g_err.clear();
  return SPECV_OK;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int elem_bytes(int32_t dtype) { return dtype == SPECV_BF16 ? 2 : 4; }
int vec_width(int32_t dtype) { return dtype == SPECV_BF16 ? 8 : 4; }

// CTAs per batch row in the decision kernel (a cluster): enough CTAs in
// total to keep every SM streaming the re-read row, at most 16, and no more
// than there are 256-vector tiles in a row.  SPECV_CLUSTER (1..16) overrides
// it, for tuning runs.
int sm_count();

// A SPECV_* tuning variable as an integer (dflt when unset), read once per
// process: callers keep it in a function-local static, whose initialisation
// C++ makes thread-safe.
int env_int(const char* name, int dflt) {
  const char* e = getenv(name);
  return e ? atoi(e) : dflt;
}

int pick_cluster(int32_t B, int32_t V, int vw, int min_c = 1, int max_c = 16) {
  static const int env = env_int("SPECV_CLUSTER", -1);
  if (env >= 1 && env <= 16) return env;
  // About four CTAs per SM over the whole grid, rounded down to a power of
  // two: clusters of 2^k CTAs pack onto the GPCs without gaps.
  const int want = 4 * sm_count();
  int c = (want + B - 1) / (B > 0 ? B : 1);
  if (c < min_c) c = min_c;
  if (c > max_c) c = max_c;
  if (c > 16) c = 16;
  // Clusters of 16 need four free SMs of one GPC each: from eight batch rows
  // on, the last ones are left for a second wave (config 4, 32 clusters of
  // 16: 66.0 us per call, 58.1 with clusters of 8).
  if (B >= 8 && c > 8) c = 8;
  while (c & (c - 1)) c &= c - 1;
  const int tiles = static_cast<int>((static_cast<int64_t>(V) + kThreads * vw - 1) / (kThreads * vw));
  if (c > tiles) c = tiles;
  return c < 1 ? 1 : (c > 16 ? 16 : c);
}

// Slice length per CTA: ceil(V / C) rounded up to a whole 16-byte vector,
// and further to whole ring trips when no CTA is left empty (then only the
// row's last slice ends inside a trip, and the other CTAs run the check-free
// path of the residual pass alone).
int64_t slice_len(int32_t V, int C, int vw) {
  int64_t L = (static_cast<int64_t>(V) + C - 1) / C;
  L = (L + vw - 1) / vw * vw;
  const int64_t trip = static_cast<int64_t>(kVecs) * kThreads * vw;
  const int64_t Lt = (L + trip - 1) / trip * trip;
  if ((static_cast<int64_t>(V) + Lt - 1) / Lt == C) L = Lt;
  return L;
}

// Rows start 16-byte aligned: base and both strides (in bytes) multiples of 16.
bool vec_ok(const void* base, int64_t bs, int64_t rs, int es) {
  return aligned(base, 16) && ((bs * es) % 16 == 0) && ((rs * es) % 16 == 0);
}

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

// Sizes of one call: kernel A chunks, kernel B cluster and slices, workspace.
struct Plan {
  int iters;       // loop trips per kernel-A CTA
  int64_t chunk;   // logits per kernel-A CTA
  int64_t nchunk;  // chunks per row
  int CB;          // CTAs per batch row in kernel B
  int64_t L;       // kernel-B slice per CTA
  size_t smemB;    // kernel-B dynamic shared memory (segment sums)
  size_t recs_bytes, cand_bytes;
  size_t piece_bytes;  // the sampler's piece table (kMaxPieces entries per chunk), or 0
};

// Loop trips per chunk of rows that carry top-F candidates (outcome keys),
// on grids of at least four waves: the per-chunk selection and its ramp are
// paid fewer times than at 8 trips.
// cfg5-ssd (256 x 9 items of 152064 fp32) per call: 8 trips 0.4583 ms, 10
// 0.4531, 11 0.4551, 12 0.4528, 13 0.4543, 14 0.4622, 15 0.4654 (longer
// chunks leave more threads with two groups above the candidate bound, whose
// whole share is read again); the geometric fan-out and Saguaro rounds the
// same way (0.4729 -> 0.4642, 0.4640 -> 0.4584).  Verification alone stays
// at 8 (12: 0.4140 -> 0.4152 ms).
constexpr int kTopFIters = 12;

int sm_count() {
  static const int n = [] {
    int dev = 0, c = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || c <= 0)
      c = 152;
    return c;
  }();
  return n;
}

// min_cb: the smallest cluster; an MSS node may stream its rows once per
// rejection, and two CTAs per node halve each pass (measured best at 2048
// nodes of 152064 fp32 logits: 1 -> 0.69 ms, 2 -> 0.58, 4 -> 0.60, 8 -> 0.61).
// iters0: loop trips per chunk before halving.  The sampler's rows all carry
// top-F candidates, whose per-chunk selection is worth amortising over longer
// chunks (kernel A 258 -> 215 us on 2304 rows of 152064 fp32 at 16 trips; 32
// with its pieces); the decision kernel's chunk-local draw reads up to 16
// trips.  Other rows with top-F candidates take kTopFIters trips when their
// grid spans several waves (below).
Plan make_plan(int32_t B, int32_t K, int32_t V, int32_t F, int32_t dtype, int min_cb = 1,
               int iters0 = 8, int max_cb = 16, bool piece_table = false) {
  Plan pl;
  const int vw = vec_width(dtype);
  const int64_t units = static_cast<int64_t>(B > 0 ? B : 0) * (K + 1);
  // Loop trips per kernel-A CTA: long chunks amortise the per-CTA reductions;
  // halve them while there would be fewer than four chunks per SM.
  // SPECV_ITERS (1..64) fixes the trip count, for tuning runs.
  static const int env_iters = env_int("SPECV_ITERS", -1);
  pl.iters = (env_iters >= 1 && env_iters <= 64) ? env_iters : iters0;
  const int64_t slots = static_cast<int64_t>(sm_count()) * ((dtype == SPECV_BF16 && F > 0) ? 4 : 5);
  const int64_t want = 4LL * sm_count();
  for (;;) {
    pl.chunk = static_cast<int64_t>(pl.iters) * kVecs * kThreads * vw;
    pl.nchunk = (static_cast<int64_t>(V) + pl.chunk - 1) / pl.chunk;
    if (pl.iters == 1 || env_iters >= 1 || units * pl.nchunk >= want) break;
    pl.iters /= 2;
  }
  // A grid just over one wave of resident CTAs (5 per SM for fp32 rows, 4 for
  // bf16) leaves a few chunks to run after the rest: lengthen the chunks (up
  // to 16 trips) until they fit in one wave.  Config 4 (B=32, K=4, V=128256
  // bf16): 640 chunks of 8 trips -> 480 of 11, 0.0525 -> 0.0485 ms per call.
  if (env_iters < 1 && units * pl.nchunk > slots && 4 * units * pl.nchunk <= 5 * slots) {
    for (int it = pl.iters + 1; it <= 16; ++it) {
      const int64_t ch = static_cast<int64_t>(it) * kVecs * kThreads * vw;
      const int64_t nc = (static_cast<int64_t>(V) + ch - 1) / ch;
      if (units * nc <= slots) {
        pl.iters = it;
        pl.chunk = ch;
        pl.nchunk = nc;
        break;
      }
    }
  }
  // Rows with top-F candidates over a grid of several waves: longer chunks
  // (kTopFIters trips), so each chunk's selection is paid fewer times.
  if (env_iters < 1 && F > 0 && !piece_table && pl.iters < kTopFIters && units * pl.nchunk >= 4 * slots) {
    pl.iters = kTopFIters;
    pl.chunk = static_cast<int64_t>(pl.iters) * kVecs * kThreads * vw;
    pl.nchunk = (static_cast<int64_t>(V) + pl.chunk - 1) / pl.chunk;
  }
  // In a single wave the longest chunk sets the kernel's time: the same
  // number of chunks, each as short as that allows (config 4's rows of 31.3
  // trips: 12 + 12 + 7.3 -> 11 + 11 + 9.3).  Not for the sampler, whose
  // pieces are eighths of its chunks.
  if (env_iters < 1 && !piece_table && units * pl.nchunk <= slots && pl.nchunk > 1) {
    const int64_t trip = static_cast<int64_t>(kVecs) * kThreads * vw;
    const int64_t trips = (static_cast<int64_t>(V) + trip - 1) / trip;
    pl.iters = static_cast<int>((trips + pl.nchunk - 1) / pl.nchunk);
    pl.chunk = static_cast<int64_t>(pl.iters) * trip;
    pl.nchunk = (static_cast<int64_t>(V) + pl.chunk - 1) / pl.chunk;
  }
  pl.CB = pick_cluster(B, V, vw, min_cb, max_cb);
  pl.L = slice_len(V, pl.CB, vw);
  const int64_t ntiles = ((pl.L / vw) + kThreads - 1) / kThreads;
  pl.smemB = static_cast<size_t>(ntiles) * kWarps * sizeof(float);
  pl.recs_bytes = round_up(static_cast<size_t>(units * pl.nchunk) * sizeof(ChunkRec), 256);
  pl.cand_bytes = F > 0 ? round_up(static_cast<size_t>(units * pl.nchunk * F) * 4, 256) : 0;
  pl.piece_bytes =
      piece_table ? round_up(static_cast<size_t>(units * pl.nchunk) * kMaxPieces * sizeof(float2), 256) : 0;
  return pl;
}

size_t plan_workspace_split(const Plan& pl) { return pl.recs_bytes + 2 * pl.cand_bytes + pl.piece_bytes; }

size_t plan_workspace(const Plan& pl) { return plan_workspace_split(pl); }

constexpr size_t kMaxSegSmem = 200 * 1024;

// Loop trips per chunk of the Saguaro sampler's rows: long chunks amortise the
// per-chunk top-F epilogue (2304 rows of 152064 fp32: kernel A 0.2233 ms at
// 16 trips, 0.2114 at 32), and each chunk's eighths are recorded, so the draw
// reads 4 trips' worth (32 KB of fp32).
constexpr int kSampleIters = 32;

// Sampled rows per SM from which the sampler's decision runs one warp per row
// (fewer rows keep one CTA per row, whose eight warps read a row's piece of
// a chunk faster than one warp can).
constexpr int kWarpRowsPerSm = 8;

// Stages of the persistent path's ring (SPECV_STAGES = 2..8 fixes the count,
// for tuning runs).
int ring_stages() {
  static const int v = env_int("SPECV_STAGES", 0);
  return (v >= 2 && v <= kMaxStages) ? v : 2;
}

// Stages of the decision kernel's residual ring (SPECV_STAGES_B = 2..8 fixes
// the count, for tuning runs).  Its grid is small (B x cluster CTAs), so each
// CTA keeps more of its slice in flight than a row-statistics CTA does.
int ring_stages_b() {
  static const int v = env_int("SPECV_STAGES_B", 0);
  return (v >= 2 && v <= kMaxStages) ? v : 2;
}

// Kernel A for 16-byte aligned layouts: the staged path (one CTA per item) by
// default, the persistent path when SPECV_PERSIST=1 (for tuning runs); the
// register path for any other layout.
bool persistent_path() {
  static const int v = env_int("SPECV_PERSIST", 0);
  return v == 1;
}

// Test hook, off unless SPECV_TEST_STALL is set: "A:<i>" makes the first
// ring stage of row-statistics item i (staged path) wait for 16 bytes that no
// copy brings, "B:<b>" the first residual stage of batch row b in the decision
// kernel; the bounded wait then runs out (about a second) and the row comes
// back flagged SPECV_ROW_DEVICE_TIMEOUT.  Returns 1 + that index for kernel
// `which`, else 0.
int test_stall(char which) {
  struct Stall {
    char k;
    int v;
  };
  static const Stall st = [] {
    const char* e = getenv("SPECV_TEST_STALL");
    if (e && (e[0] == 'A' || e[0] == 'B') && e[1] == ':') return Stall{e[0], atoi(e + 2)};
    return Stall{0, -1};
  }();
  return (st.v >= 0 && st.k == which) ? st.v + 1 : 0;
}

// Checks shared by specv_verify and specv_ssd_round.
specv_status check_verify_args(const specv_verify_args* a, int draft_rows) {
  const int32_t B = a->B, K = a->K, V = a->V;
  if (B < 0) return fail(SPECV_ERR_INVALID_ARG, "B=%d < 0", B);
  if (K < 1 || K > 32) return fail(SPECV_ERR_INVALID_ARG, "K=%d outside [1, 32]", K);
  if (V < 1) return fail(SPECV_ERR_INVALID_ARG, "V=%d < 1", V);
  if (a->dtype != SPECV_BF16 && a->dtype != SPECV_FP32)
    return fail(SPECV_ERR_INVALID_ARG, "dtype=%d is not SPECV_BF16 or SPECV_FP32", a->dtype);
  if (a->flags & ~SPECV_NO_DRAFT_PROBS) return fail(SPECV_ERR_INVALID_ARG, "unknown flags 0x%x", a->flags);
  const bool nd = (a->flags & SPECV_NO_DRAFT_PROBS) != 0;
  if (a->cu_num_draft_tokens && a->num_draft_tokens < 0)
    return fail(SPECV_ERR_INVALID_ARG, "num_draft_tokens=%d < 0", a->num_draft_tokens);
  if (B == 0) return SPECV_OK;
  if (nd != (a->draft_logits == nullptr))
    return fail(SPECV_ERR_INVALID_ARG, "draft_logits must be NULL exactly when SPECV_NO_DRAFT_PROBS is set");
  if (!a->target_logits || !a->draft_tokens || !a->temperature || !a->uniforms ||
      !a->accept_len || !a->out_tokens)
    return fail(SPECV_ERR_INVALID_ARG, "a required pointer is NULL");
  const int es = elem_bytes(a->dtype);
  if (!aligned(a->cu_num_draft_tokens, 4))
    return fail(SPECV_ERR_INVALID_ARG, "a pointer is not aligned to its element size");
  if (!aligned(a->target_logits, es) || !aligned(a->draft_logits, es) ||
      !aligned(a->draft_tokens, 4) || !aligned(a->temperature, 4) || !aligned(a->uniforms, 4) ||
      !aligned(a->accept_len, 4) || !aligned(a->out_tokens, 4) || !aligned(a->p_draft, 4) ||
      !aligned(a->q_draft, 4) || !aligned(a->row_status, 4))
    return fail(SPECV_ERR_INVALID_ARG, "a pointer is not aligned to its element size");
  if (a->target_row_stride < V || (!nd && a->draft_row_stride < V))
    return fail(SPECV_ERR_INVALID_ARG, "row stride smaller than V");
  if (a->cu_num_draft_tokens) return SPECV_OK;  // packed rows: no batch strides
  if (B > 1 && (a->target_batch_stride < K * a->target_row_stride + V ||
                (!nd && a->draft_batch_stride < (draft_rows - 1) * a->draft_row_stride + V)))
    return fail(SPECV_ERR_INVALID_ARG, "batch stride too small for K+1 target / %d draft rows",
                draft_rows);
  return SPECV_OK;
}

}  // namespace

extern "C" {

const char* specv_status_string(specv_status s) {
  switch (s) {
    case SPECV_OK: return "ok";
    case SPECV_ERR_INVALID_ARG: return "invalid argument";
    case SPECV_ERR_UNSUPPORTED: return "unsupported size or layout";
    case SPECV_ERR_CUDA: return "CUDA error";
    case SPECV_ERR_WORKSPACE: return "workspace missing or too small";
  }
  return "unknown status";
}

const char* specv_last_error(void) { return g_err.c_str(); }

int32_t specv_last_launch_count(void) { return g_launches; }

void specv_set_split_event(void* event) { g_split_event = static_cast<cudaEvent_t>(event); }

size_t specv_verify_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t dtype) {
  if (B <= 0 || K < 1 || V < 1) return 0;
  return plan_workspace(make_plan(B, K, V, 0, dtype));
}

namespace {

// What an MSS call adds to the verification arguments.
struct MssExtra {
  const int32_t* ncand;
  int32_t naive;
  int32_t* acc;
  float* ap;
};

// Both kernels for one call: verification, an SSD round, (kModeSample, K =
// 0, the drafter's rows as draft rows) Saguaro sampling, or (kModeMss, K = M
// candidates, one target and one draft row per node) MSS.  sg_F/sg_C: the
// Saguaro sampling scheme of the drafts (sg_F = 0: none).
specv_status run_verify(const specv_verify_args* a, void* workspace, size_t workspace_bytes,
                        void* stream, int mode, int32_t F, int32_t* keys, float* key_logits,
                        uint8_t* hit, const int32_t* fanout, int32_t sg_F = 0, float sg_C = 1.f,
                        const MssExtra* mx = nullptr) {
  const int32_t B = a->B, K = a->K, V = a->V;
  const int32_t Ka = mode == kModeMss ? 0 : K;  // positions per row in the statistics kernel
  const bool cands = mode == kModeSsd || mode == kModeSample;
  const int es = elem_bytes(a->dtype);
  // Packed rows have no batch stride: row alignment follows from the row stride.
  const bool packed = a->cu_num_draft_tokens != nullptr;
  const bool nd = (a->flags & SPECV_NO_DRAFT_PROBS) != 0;
  const bool vec =
      vec_ok(a->target_logits, packed ? 0 : a->target_batch_stride, a->target_row_stride, es) &&
      (nd || vec_ok(a->draft_logits, packed ? 0 : a->draft_batch_stride, a->draft_row_stride, es));
  Plan pl = make_plan(B, Ka, V, cands ? F : 0, a->dtype, mode == kModeMss ? 2 : 1,
                      mode == kModeSample ? kSampleIters : 8, 16, mode == kModeSample);
  // The sampler's rows draw from one chunk each (the chunk-local draw) when a
  // chunk is shorter than the row: the other CTAs of a cluster would only
  // wait, so its rows take one CTA each.
  if (mode == kModeSample && pl.CB > 1 && pl.chunk < V) {
    const Plan one = make_plan(B, Ka, V, cands ? F : 0, a->dtype, 1, kSampleIters, 1, true);
    if (one.smemB <= kMaxSegSmem) pl = one;  // (a very long row keeps its cluster)
  }
  if (pl.smemB > kMaxSegSmem) return fail(SPECV_ERR_UNSUPPORTED, "V=%d too large", V);
  const size_t need = plan_workspace(pl);
  if (!workspace || workspace_bytes < need)
    return fail(SPECV_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, workspace_bytes);
  if (!aligned(workspace, 256)) return fail(SPECV_ERR_WORKSPACE, "workspace not 256-byte aligned");
  const int64_t units = static_cast<int64_t>(B) * (Ka + 1);
  if (units * pl.nchunk > 0x7fffffffLL || static_cast<int64_t>(B) * pl.CB > 0x7fffffffLL)
    return fail(SPECV_ERR_UNSUPPORTED, "B*(K+1) too large");
  char* ws = static_cast<char*>(workspace);
  ChunkRec* recs = reinterpret_cast<ChunkRec*>(ws);
  float* cand_v = pl.cand_bytes ? reinterpret_cast<float*>(ws + pl.recs_bytes) : nullptr;
  int32_t* cand_i = pl.cand_bytes ? reinterpret_cast<int32_t*>(ws + pl.recs_bytes + pl.cand_bytes) : nullptr;
  float2* piece_stats =
      pl.piece_bytes ? reinterpret_cast<float2*>(ws + pl.recs_bytes + 2 * pl.cand_bytes) : nullptr;

  StatsParams sp = {};
  sp.zt = a->target_logits;
  sp.t_bs = a->target_batch_stride;
  sp.t_rs = a->target_row_stride;
  sp.zd = a->draft_logits;
  sp.d_bs = a->draft_batch_stride;
  sp.d_rs = a->draft_row_stride;
  sp.tokens = a->draft_tokens;
  sp.temp = a->temperature;
  sp.recs = recs;
  sp.cand_v = cand_v;
  sp.cand_i = cand_i;
  sp.B = B;
  sp.K = Ka;
  sp.V = V;
  sp.F = F;
  sp.nchunk = static_cast<int32_t>(pl.nchunk);
  sp.chunk = static_cast<int32_t>(pl.chunk);
  sp.iters = pl.iters;
  // Candidates per chunk at each position: the fan-out (F when uniform), and
  // never fewer than the Saguaro F_s the draft rows' weights need.
  for (int k = 0; k <= Ka; ++k) sp.fk[k] = max(fanout ? fanout[k] : F, sg_F);
  sp.stages = ring_stages();
  // The sampler's staged chunks record their pieces apart (eighths when the
  // trip count divides by 8, else quarters or halves), so its draw reads one
  // piece.
  if (mode == kModeSample && vec && !persistent_path() && piece_stats) {
    sp.pieces = pl.iters % 8 == 0 ? 8 : pl.iters % 4 == 0 ? 4 : pl.iters % 2 == 0 ? 2 : 0;
    sp.piece = sp.pieces ? pl.iters / sp.pieces : 0;
    sp.piece_stats = piece_stats;
  }
  sp.cu = a->cu_num_draft_tokens;
  sp.ntok = a->num_draft_tokens;
  sp.stall = test_stall('A');
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t items = units * pl.nchunk;
  cudaError_t e =
      mode == kModeSsd      ? launch_stats<kModeSsd>(a->dtype, vec, persistent_path(), sm_count(), items, s, sp)
      : mode == kModeSample ? launch_stats<kModeSample>(a->dtype, vec, persistent_path(), sm_count(), items, s, sp)
      : mode == kModeMss    ? launch_stats<kModeMss>(a->dtype, vec, persistent_path(), sm_count(), items, s, sp)
                            : launch_stats<kModeVerify>(a->dtype, vec, persistent_path(), sm_count(), items, s, sp);
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "row-statistics launch: %s", cudaGetErrorString(e));
  e = record_split(s);
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "split event: %s", cudaGetErrorString(e));

  DecideParams dp = {};
  dp.zt = a->target_logits;
  dp.t_bs = a->target_batch_stride;
  dp.t_rs = a->target_row_stride;
  dp.zd = a->draft_logits;
  dp.d_bs = a->draft_batch_stride;
  dp.d_rs = a->draft_row_stride;
  dp.tokens = a->draft_tokens;
  dp.temp = a->temperature;
  dp.unif = a->uniforms;
  dp.recs = recs;
  dp.cand_v = cand_v;
  dp.cand_i = cand_i;
  dp.accept_len = a->accept_len;
  dp.out_tokens = a->out_tokens;
  dp.p_draft = a->p_draft;
  dp.q_draft = a->q_draft;
  dp.row_status = a->row_status;
  dp.keys = keys;
  dp.key_logits = key_logits;
  dp.hit = hit;
  dp.B = B;
  dp.K = K;
  dp.V = V;
  dp.F = F;
  dp.nchunk = static_cast<int32_t>(pl.nchunk);
  dp.CB = pl.CB;
  dp.L = static_cast<int32_t>(pl.L);
  dp.chunk = static_cast<int32_t>(pl.chunk);
  // A draw from a whole row reads one chunk on rank 0 instead of a slice on
  // every CTA of the cluster: worth it when the chunk is the shorter read.
  // SPECV_LOCAL_DRAW=0/1 overrides, for tuning runs.
  static const int env_local = env_int("SPECV_LOCAL_DRAW", -1);
  const int64_t span = sp.pieces ? pl.chunk / sp.pieces : pl.chunk;  // what the draw reads
  const bool fits = span <= static_cast<int64_t>(kDrawTiles) * kThreads * vec_width(a->dtype);
  dp.local_draw = fits && (env_local >= 0 ? env_local != 0 : pl.chunk < pl.L);
  dp.pieces = sp.pieces;
  dp.piece_stats = sp.piece_stats;
  dp.stall = test_stall('B');
  for (int k = 0; k <= K; ++k) dp.fk[k] = fanout ? fanout[k] : F;
  // Aligned rows stream the residual slice through a ring placed after the
  // segment sums in dynamic shared memory.
  // (Very long rows whose segment table leaves no room for it read directly.)
  dp.cu = a->cu_num_draft_tokens;
  dp.ntok = a->num_draft_tokens;
  dp.no_draft = (a->flags & SPECV_NO_DRAFT_PROBS) ? 1 : 0;
  dp.sg_F = sg_F;
  dp.sg_C = sg_C;
  dp.ring_off = static_cast<int32_t>(round_up(pl.smemB, 128));
  dp.stages = ring_stages_b();
  size_t smemB = dp.ring_off + static_cast<size_t>(dp.stages) * 2 * kTripBytes;
  if (!vec || smemB > kMaxSegSmem) {
    dp.stages = 0;
    smemB = pl.smemB;
  }
  if (mx) {
    dp.ncand = mx->ncand;
    dp.naive = mx->naive;
    dp.mss_acc = mx->acc;
    dp.mss_ap = mx->ap;
  }
  // The sampler's rows on one warp each, when they are many and their records
  // carry first halves (aligned rows, chunks of an even trip count).
  // SPECV_SAMPLE_WARP=0/1 overrides the row count, for tuning runs.
  static const int env_warp = env_int("SPECV_SAMPLE_WARP", -1);
  const int64_t nv_row = (static_cast<int64_t>(V) + vec_width(a->dtype) - 1) / vec_width(a->dtype);
  const size_t smem_row = static_cast<size_t>((nv_row + kThreads - 1) / kThreads) * kWarps * sizeof(float);
  const bool warp_rows = mode == kModeSample && vec && sp.pieces > 0 && smem_row <= kMaxSegSmem &&
                         (env_warp >= 0 ? env_warp != 0 : B >= kWarpRowsPerSm * sm_count());
  e = warp_rows             ? launch_sample_rows(a->dtype, B, smem_row, s, dp)
      : mode == kModeSsd    ? launch_decide<kModeSsd>(a->dtype, vec, pl.CB, B, smemB, s, dp)
      : mode == kModeSample ? launch_decide<kModeSample>(a->dtype, vec, pl.CB, B, smemB, s, dp)
      : mode == kModeMss    ? launch_decide<kModeMss>(a->dtype, vec, pl.CB, B, smemB, s, dp)
                            : launch_decide<kModeVerify>(a->dtype, vec, pl.CB, B, smemB, s, dp);
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "decision launch: %s", cudaGetErrorString(e));
  g_launches = 2;
  return ok();
}

}  // namespace

specv_status specv_verify(const specv_verify_args* a, void* workspace, size_t workspace_bytes,
                          void* stream) {
  g_launches = 0;
  if (!a) return fail(SPECV_ERR_INVALID_ARG, "args is NULL");
  specv_status st = check_verify_args(a, a->K);
  if (st != SPECV_OK) return st;
  if (a->B == 0) return ok();
  return run_verify(a, workspace, workspace_bytes, stream, kModeVerify, 0, nullptr, nullptr,
                    nullptr, nullptr);
}

size_t specv_ssd_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t F, int32_t dtype) {
  if (B <= 0 || K < 1 || V < 1 || F < 1) return 0;
  return plan_workspace(make_plan(B, K, V, F, dtype));
}

specv_status specv_ssd_round(const specv_ssd_args* a, void* workspace, size_t workspace_bytes,
                             void* stream) {
  g_launches = 0;
  if (!a) return fail(SPECV_ERR_INVALID_ARG, "args is NULL");
  specv_status st = check_verify_args(&a->verify, a->verify.K + 1);
  if (st != SPECV_OK) return st;
  if (a->F < 1 || a->F > 32) return fail(SPECV_ERR_INVALID_ARG, "F=%d outside [1, 32]", a->F);
  if (a->verify.flags & SPECV_NO_DRAFT_PROBS)
    return fail(SPECV_ERR_INVALID_ARG, "an SSD round ranks draft logits: SPECV_NO_DRAFT_PROBS does not apply");
  if (a->verify.cu_num_draft_tokens)
    return fail(SPECV_ERR_UNSUPPORTED, "per-row draft counts are supported by specv_verify only");
  if (a->verify.B == 0) return ok();
  if (!a->keys || !a->hit) return fail(SPECV_ERR_INVALID_ARG, "keys or hit is NULL");
  if (!aligned(a->keys, 4) || !aligned(a->key_logits, 4))
    return fail(SPECV_ERR_INVALID_ARG, "a pointer is not aligned to its element size");
  if (a->fanout)
    for (int k = 0; k <= a->verify.K; ++k)
      if (a->fanout[k] < 0 || a->fanout[k] > a->F)
        return fail(SPECV_ERR_INVALID_ARG, "fanout[%d]=%d outside [0, F=%d]", k, a->fanout[k], a->F);
  if (a->saguaro_F < 0 || a->saguaro_F > a->F)
    return fail(SPECV_ERR_INVALID_ARG, "saguaro_F=%d outside [0, F=%d]", a->saguaro_F, a->F);
  if (a->saguaro_F > 0 && !(a->saguaro_C >= 0.f && a->saguaro_C <= 1.f))
    return fail(SPECV_ERR_INVALID_ARG, "saguaro_C=%g outside [0, 1]", a->saguaro_C);
  return run_verify(&a->verify, workspace, workspace_bytes, stream, kModeSsd, a->F, a->keys,
                    a->key_logits, a->hit, a->fanout, a->saguaro_F,
                    a->saguaro_F > 0 ? a->saguaro_C : 1.f);
}

size_t specv_predict_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t F, int32_t dtype) {
  if (B <= 0 || K < 1 || V < 1 || F < 1) return 0;
  return plan_workspace_split(make_plan(B, K, V, F, dtype));
}

specv_status specv_predict_outcomes(const specv_predict_args* a, void* workspace,
                                    size_t workspace_bytes, void* stream) {
  g_launches = 0;
  if (!a) return fail(SPECV_ERR_INVALID_ARG, "args is NULL");
  const int32_t B = a->B, K = a->K, V = a->V, F = a->F;
  if (B < 0) return fail(SPECV_ERR_INVALID_ARG, "B=%d < 0", B);
  if (K < 1 || K > 32) return fail(SPECV_ERR_INVALID_ARG, "K=%d outside [1, 32]", K);
  if (V < 1) return fail(SPECV_ERR_INVALID_ARG, "V=%d < 1", V);
  if (F < 1 || F > 32) return fail(SPECV_ERR_INVALID_ARG, "F=%d outside [1, 32]", F);
  if (a->dtype != SPECV_BF16 && a->dtype != SPECV_FP32)
    return fail(SPECV_ERR_INVALID_ARG, "dtype=%d is not SPECV_BF16 or SPECV_FP32", a->dtype);
  if (a->fanout)
    for (int k = 0; k <= K; ++k)
      if (a->fanout[k] < 0 || a->fanout[k] > F)
        return fail(SPECV_ERR_INVALID_ARG, "fanout[%d]=%d outside [0, F=%d]", k, a->fanout[k], F);
  if (B == 0) return ok();
  if (!a->draft_logits || !a->draft_tokens || !a->keys)
    return fail(SPECV_ERR_INVALID_ARG, "a required pointer is NULL");
  const int es = elem_bytes(a->dtype);
  if (!aligned(a->draft_logits, es) || !aligned(a->draft_tokens, 4) || !aligned(a->keys, 4) ||
      !aligned(a->key_logits, 4) || !aligned(a->row_status, 4))
    return fail(SPECV_ERR_INVALID_ARG, "a pointer is not aligned to its element size");
  if (a->draft_row_stride < V) return fail(SPECV_ERR_INVALID_ARG, "row stride smaller than V");
  if (B > 1 && a->draft_batch_stride < K * a->draft_row_stride + V)
    return fail(SPECV_ERR_INVALID_ARG, "batch stride too small for K+1 draft rows");
  const Plan pl = make_plan(B, K, V, F, a->dtype);
  const size_t need = plan_workspace_split(pl);
  if (!workspace || workspace_bytes < need)
    return fail(SPECV_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, workspace_bytes);
  if (!aligned(workspace, 256)) return fail(SPECV_ERR_WORKSPACE, "workspace not 256-byte aligned");
  const int64_t units = static_cast<int64_t>(B) * (K + 1);
  if (units * pl.nchunk > 0x7fffffffLL) return fail(SPECV_ERR_UNSUPPORTED, "B*(K+1) too large");
  const bool vec = vec_ok(a->draft_logits, a->draft_batch_stride, a->draft_row_stride, es);
  char* ws = static_cast<char*>(workspace);
  StatsParams sp = {};
  sp.zd = a->draft_logits;
  sp.d_bs = a->draft_batch_stride;
  sp.d_rs = a->draft_row_stride;
  sp.tokens = a->draft_tokens;
  sp.recs = reinterpret_cast<ChunkRec*>(ws);
  sp.cand_v = reinterpret_cast<float*>(ws + pl.recs_bytes);
  sp.cand_i = reinterpret_cast<int32_t*>(ws + pl.recs_bytes + pl.cand_bytes);
  sp.B = B;
  sp.K = K;
  sp.V = V;
  sp.F = F;
  sp.nchunk = static_cast<int32_t>(pl.nchunk);
  sp.chunk = static_cast<int32_t>(pl.chunk);
  sp.iters = pl.iters;
  for (int k = 0; k <= K; ++k) sp.fk[k] = a->fanout ? a->fanout[k] : F;
  sp.stages = ring_stages();
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = launch_stats<kModePredict>(a->dtype, vec, persistent_path(), sm_count(), units * pl.nchunk, s, sp);
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "row-statistics launch: %s", cudaGetErrorString(e));
  e = record_split(s);
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "split event: %s", cudaGetErrorString(e));
  PredictKeysParams kp = {};
  kp.tokens = a->draft_tokens;
  kp.recs = sp.recs;
  kp.cand_v = sp.cand_v;
  kp.cand_i = sp.cand_i;
  kp.keys = a->keys;
  kp.key_logits = a->key_logits;
  kp.row_status = a->row_status;
  kp.B = B;
  kp.K = K;
  kp.V = V;
  kp.F = F;
  kp.nchunk = static_cast<int32_t>(pl.nchunk);
  for (int k = 0; k <= K; ++k) kp.fk[k] = a->fanout ? a->fanout[k] : F;
  e = launch_predict_keys(kp, B, s);
  if (e == cudaSuccess) e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "keys launch: %s", cudaGetErrorString(e));
  g_launches = 2;
  return ok();
}

size_t specv_saguaro_workspace_bytes(int32_t B, int32_t V, int32_t F, int32_t dtype) {
  if (B <= 0 || V < 1 || F < 0 || F > 32) return 0;
  return plan_workspace(make_plan(B, 0, V, F > 0 ? F : 1, dtype, 1, kSampleIters, 16, true));
}

// Saguaro sampling runs the verification pipeline with no drafts (K = 0):
// kernel A streams each row once (statistics and its top-F candidates), and
// kernel B draws the token from sigma_{F,C} by inverse CDF of the uniform.
specv_status specv_saguaro_sample(const specv_saguaro_args* a, void* workspace,
                                  size_t workspace_bytes, void* stream) {
  g_launches = 0;
  if (!a) return fail(SPECV_ERR_INVALID_ARG, "args is NULL");
  const int32_t B = a->B, V = a->V;
  if (B < 0) return fail(SPECV_ERR_INVALID_ARG, "B=%d < 0", B);
  if (V < 1) return fail(SPECV_ERR_INVALID_ARG, "V=%d < 1", V);
  if (a->dtype != SPECV_BF16 && a->dtype != SPECV_FP32)
    return fail(SPECV_ERR_INVALID_ARG, "dtype=%d is not SPECV_BF16 or SPECV_FP32", a->dtype);
  if (a->F < 0 || a->F > 32) return fail(SPECV_ERR_INVALID_ARG, "F=%d outside [0, 32]", a->F);
  if (!(a->C >= 0.f && a->C <= 1.f)) return fail(SPECV_ERR_INVALID_ARG, "C=%g outside [0, 1]", a->C);
  if (B == 0) return ok();
  if (!a->logits || !a->temperature || !a->uniforms || !a->tokens)
    return fail(SPECV_ERR_INVALID_ARG, "a required pointer is NULL");
  const int es = elem_bytes(a->dtype);
  if (!aligned(a->logits, es) || !aligned(a->temperature, 4) || !aligned(a->uniforms, 4) ||
      !aligned(a->tokens, 4) || !aligned(a->q, 4) || !aligned(a->row_status, 4))
    return fail(SPECV_ERR_INVALID_ARG, "a pointer is not aligned to its element size");
  if (a->row_stride < V) return fail(SPECV_ERR_INVALID_ARG, "row stride smaller than V");
  specv_verify_args v = {};
  v.B = B;
  v.K = 0;
  v.V = V;
  v.dtype = a->dtype;
  v.target_logits = a->logits;  // read through the draft slot; kept valid for the checks
  v.target_batch_stride = a->row_stride;
  v.target_row_stride = a->row_stride;
  v.draft_logits = a->logits;
  v.draft_batch_stride = a->row_stride;
  v.draft_row_stride = a->row_stride;
  v.temperature = a->temperature;
  v.uniforms = a->uniforms;
  v.out_tokens = a->tokens;
  v.q_draft = a->q;
  v.row_status = a->row_status;
  const int32_t F = a->F > 0 ? a->F : 1;
  return run_verify(&v, workspace, workspace_bytes, stream, kModeSample, F, nullptr, nullptr,
                    nullptr, nullptr, a->F, a->F > 0 ? a->C : 1.f);
}

size_t specv_mss_workspace_bytes(int32_t B, int32_t M, int32_t V, int32_t dtype) {
  if (B <= 0 || M < 1 || V < 1 || M > 32) return 0;
  return plan_workspace(make_plan(B, 0, V, 0, dtype, 2));
}

specv_status specv_mss_verify(const specv_mss_args* a, void* workspace, size_t workspace_bytes,
                              void* stream) {
  g_launches = 0;
  if (!a) return fail(SPECV_ERR_INVALID_ARG, "args is NULL");
  const int32_t B = a->B, M = a->M, V = a->V;
  if (B < 0) return fail(SPECV_ERR_INVALID_ARG, "B=%d < 0", B);
  if (M < 1 || M > 32) return fail(SPECV_ERR_INVALID_ARG, "M=%d outside [1, 32]", M);
  if (V < 1) return fail(SPECV_ERR_INVALID_ARG, "V=%d < 1", V);
  if (a->dtype != SPECV_BF16 && a->dtype != SPECV_FP32)
    return fail(SPECV_ERR_INVALID_ARG, "dtype=%d is not SPECV_BF16 or SPECV_FP32", a->dtype);
  if (a->flags & ~SPECV_MSS_NAIVE) return fail(SPECV_ERR_INVALID_ARG, "unknown flags 0x%x", a->flags);
  if (B == 0) return ok();
  if (!a->target_logits || !a->draft_logits || !a->candidates || !a->temperature ||
      !a->uniforms || !a->accepted || !a->out_token)
    return fail(SPECV_ERR_INVALID_ARG, "a required pointer is NULL");
  const int es = elem_bytes(a->dtype);
  if (!aligned(a->target_logits, es) || !aligned(a->draft_logits, es) || !aligned(a->candidates, 4) ||
      !aligned(a->num_candidates, 4) || !aligned(a->temperature, 4) || !aligned(a->uniforms, 4) ||
      !aligned(a->accepted, 4) || !aligned(a->out_token, 4) || !aligned(a->accept_prob, 4) ||
      !aligned(a->row_status, 4))
    return fail(SPECV_ERR_INVALID_ARG, "a pointer is not aligned to its element size");
  if (a->target_row_stride < V || a->draft_row_stride < V)
    return fail(SPECV_ERR_INVALID_ARG, "row stride smaller than V");
  specv_verify_args v = {};
  v.B = B;
  v.K = M;
  v.V = V;
  v.dtype = a->dtype;
  v.target_logits = a->target_logits;
  v.target_batch_stride = a->target_row_stride;  // one row per node
  v.target_row_stride = a->target_row_stride;
  v.draft_logits = a->draft_logits;
  v.draft_batch_stride = a->draft_row_stride;
  v.draft_row_stride = a->draft_row_stride;
  v.draft_tokens = a->candidates;
  v.temperature = a->temperature;
  v.uniforms = a->uniforms;
  v.out_tokens = a->out_token;
  v.row_status = a->row_status;
  const MssExtra mx{a->num_candidates, (a->flags & SPECV_MSS_NAIVE) ? 1 : 0, a->accepted, a->accept_prob};
  return run_verify(&v, workspace, workspace_bytes, stream, kModeMss, 0, nullptr, nullptr, nullptr,
                    nullptr, 0, 1.f, &mx);
}

// Theorem 12 of "Speculative Speculative Decoding": F_k = F_0 q^k (k < K) and
// F_K = F_0 q^K t with q = a^{1/(1+r)}, t = (1-a)^{-1/(1+r)}; the budget
// fixes F_0 = budget / (q^K t + sum_{k<K} q^k).  Rounded by largest remainder.
specv_status specv_geometric_fanout(int32_t K, double a, double r, int32_t budget, int32_t max_f,
                                    int32_t* fanout, double* real) {
  if (K < 1 || K > 32) return fail(SPECV_ERR_INVALID_ARG, "K=%d outside [1, 32]", K);
  if (!(a > 0.0 && a < 1.0)) return fail(SPECV_ERR_INVALID_ARG, "a=%g outside (0, 1)", a);
  if (!(r > 0.0) || !(r < 1e300)) return fail(SPECV_ERR_INVALID_ARG, "r=%g is not positive", r);
  if (budget < 0) return fail(SPECV_ERR_INVALID_ARG, "budget=%d < 0", budget);
  if (max_f < 0 || max_f > 32) return fail(SPECV_ERR_INVALID_ARG, "max_f=%d outside [0, 32]", max_f);
  if (!fanout) return fail(SPECV_ERR_INVALID_ARG, "fanout is NULL");
  const double q = std::pow(a, 1.0 / (1.0 + r));
  const double t = std::pow(1.0 - a, -1.0 / (1.0 + r));
  double head = 0.0, qk = 1.0;  // sum_{k<K} q^k
  for (int k = 0; k < K; ++k) {
    head += qk;
    qk *= q;
  }
  const double f0 = static_cast<double>(budget) / (qk * t + head);
  double x[33];
  int32_t whole[33];
  int64_t left = budget;
  double w = f0;
  for (int k = 0; k <= K; ++k) {
    x[k] = (k < K) ? w : w * t;
    w *= q;
    whole[k] = static_cast<int32_t>(std::floor(x[k]));
    left -= whole[k];
    fanout[k] = whole[k];
    if (real) real[k] = x[k];
  }
  // the leftover budget, one each, to the largest fractional parts
  while (left > 0) {
    int pick = -1;
    for (int k = 0; k <= K; ++k) {
      if (fanout[k] != whole[k]) continue;
      if (pick < 0 || x[k] - whole[k] > x[pick] - whole[pick]) pick = k;
    }
    if (pick < 0) break;
    ++fanout[pick];
    --left;
  }
  for (int k = 0; k <= K; ++k) fanout[k] = std::min(fanout[k], max_f);
  return ok();
}

specv_status specv_check_hit(int32_t B, int32_t K, int32_t F, const int32_t* keys,
                             const int32_t* accept_len, const int32_t* out_tokens, uint8_t* hit,
                             void* stream) {
  g_launches = 0;
  if (B < 0) return fail(SPECV_ERR_INVALID_ARG, "B=%d < 0", B);
  if (K < 1 || K > 32) return fail(SPECV_ERR_INVALID_ARG, "K=%d outside [1, 32]", K);
  if (F < 1 || F > 32) return fail(SPECV_ERR_INVALID_ARG, "F=%d outside [1, 32]", F);
  if (B == 0) return ok();
  if (!keys || !accept_len || !out_tokens || !hit)
    return fail(SPECV_ERR_INVALID_ARG, "a required pointer is NULL");
  if (!aligned(keys, 4) || !aligned(accept_len, 4) || !aligned(out_tokens, 4))
    return fail(SPECV_ERR_INVALID_ARG, "a pointer is not aligned to its element size");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const cudaError_t e = launch_check_hit(B, K, F, keys, accept_len, out_tokens, hit, s);
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "check_hit launch: %s", cudaGetErrorString(e));
  g_launches = 1;
  return ok();
}

}  // extern "C"

// ---- verification with the library's own scratch (no workspace argument) ----
//
// For callers that cannot allocate device memory where they call us: a server
// that reserved all free GPU memory for its KV cache at start-up, or a host
// language with no CUDA allocator binding.  The scratch (kernel A's per-chunk
// records) lives in a fixed array in device memory, one copy per GPU that
// loads this library, held until the process exits.

namespace {

constexpr size_t kNoAllocScratchBytes = SPECV_NOALLOC_SCRATCH_BYTES;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
std::mutex g_noalloc_mutex;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the scratch on the current device, looked up once per
// device (with that device current) and cached.
specv_status noalloc_scratch(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kNoAllocMaxDevices)
    return fail(SPECV_ERR_UNSUPPORTED, "device index %d beyond %d", dev, kNoAllocMaxDevices);
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (!g_noalloc_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return fail(SPECV_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
    g_noalloc_addr[dev] = p;
  }
  *out = g_noalloc_addr[dev];
  return SPECV_OK;
}

}  // namespace

extern "C" specv_status specv_verify_noalloc(const specv_verify_args* a, void* stream) {
  g_launches = 0;
  if (!a) return fail(SPECV_ERR_INVALID_ARG, "args is NULL");
  specv_status st = check_verify_args(a, a->K);
  if (st != SPECV_OK) return st;
  if (a->B == 0) return ok();
  const size_t need = specv_verify_workspace_bytes(a->B, a->K, a->V, a->dtype);
  if (need > kNoAllocScratchBytes)
    return fail(SPECV_ERR_UNSUPPORTED,
                "this call needs %zu bytes of scratch but the built-in scratch holds %zu "
                "(SPECV_NOALLOC_SCRATCH_BYTES); call specv_verify with a workspace instead",
                need, kNoAllocScratchBytes);
  void* ws = nullptr;
  st = noalloc_scratch(&ws);
  if (st != SPECV_OK) return st;
  // Every record kernel B reads is written by kernel A earlier in this same
  // call, so nothing in the scratch has to start at zero.
  return run_verify(a, ws, kNoAllocScratchBytes, stream, kModeVerify, 0, nullptr, nullptr,
                    nullptr, nullptr);
}
