// C ABI of libspecv (declared in include/specv.h): argument checks, workspace
// sizing, cluster-size choice and kernel launches on the caller's stream.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <string>

#include "specv.h"
#include "predict_kernels.cuh"
#include "verify_kernels.cuh"

using namespace specv;

namespace {

thread_local std::string g_err;
thread_local int32_t g_launches = 0;

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

// CTAs per cluster: one per ~8K logits of a row, at most 16.  SPECV_CLUSTER
// (1..16) overrides it, for tuning runs.
int pick_cluster(int32_t V) {
  static int env = -2;
  if (env == -2) {
    const char* s = getenv("SPECV_CLUSTER");
    env = s ? atoi(s) : -1;
  }
  if (env >= 1 && env <= 16) return env;
  int c = (V + 8191) / 8192;
  return c < 1 ? 1 : (c > 16 ? 16 : c);
}

// Slice length per CTA: ceil(V / C) rounded up to a whole 16-byte vector.
int64_t slice_len(int32_t V, int C, int vw) {
  int64_t L = (static_cast<int64_t>(V) + C - 1) / C;
  return (L + vw - 1) / vw * vw;
}

// Rows start 16-byte aligned: base and both strides (in bytes) multiples of 16.
bool vec_ok(const void* base, int64_t bs, int64_t rs, int es) {
  return aligned(base, 16) && ((bs * es) % 16 == 0) && ((rs * es) % 16 == 0);
}

template <typename Kern>
cudaError_t allow_cluster(Kern k, int C) {
  if (C <= 8) return cudaSuccess;
  return cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
}

template <typename Kern, typename Params>
cudaError_t launch_clustered(Kern k, int C, int64_t units, size_t smem, cudaStream_t stream,
                             const Params& p) {
  cudaError_t e = allow_cluster(k, C);
  if (e != cudaSuccess) return e;
  if (smem > 0) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

constexpr size_t kMaxSegSmem = 48 * 1024;

size_t round_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

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

size_t specv_verify_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t dtype) {
  (void)V;
  (void)dtype;
  if (B <= 0 || K < 1) return 0;
  return round_up(static_cast<size_t>(B) * (K + 1) * sizeof(UnitOut), 256);
}

specv_status specv_verify(const specv_verify_args* a, void* workspace, size_t workspace_bytes,
                          void* stream) {
  g_launches = 0;
  if (!a) return fail(SPECV_ERR_INVALID_ARG, "args is NULL");
  const int32_t B = a->B, K = a->K, V = a->V;
  if (B < 0) return fail(SPECV_ERR_INVALID_ARG, "B=%d < 0", B);
  if (K < 1 || K > 32) return fail(SPECV_ERR_INVALID_ARG, "K=%d outside [1, 32]", K);
  if (V < 1) return fail(SPECV_ERR_INVALID_ARG, "V=%d < 1", V);
  if (a->dtype != SPECV_BF16 && a->dtype != SPECV_FP32)
    return fail(SPECV_ERR_INVALID_ARG, "dtype=%d is not SPECV_BF16 or SPECV_FP32", a->dtype);
  if (B == 0) return ok();
  if (!a->target_logits || !a->draft_logits || !a->draft_tokens || !a->temperature ||
      !a->uniforms || !a->accept_len || !a->out_tokens)
    return fail(SPECV_ERR_INVALID_ARG, "a required pointer is NULL");
  const int es = elem_bytes(a->dtype);
  if (!aligned(a->target_logits, es) || !aligned(a->draft_logits, es) ||
      !aligned(a->draft_tokens, 4) || !aligned(a->temperature, 4) || !aligned(a->uniforms, 4) ||
      !aligned(a->accept_len, 4) || !aligned(a->out_tokens, 4) || !aligned(a->p_draft, 4) ||
      !aligned(a->q_draft, 4) || !aligned(a->row_status, 4))
    return fail(SPECV_ERR_INVALID_ARG, "a pointer is not aligned to its element size");
  if (a->target_row_stride < V || a->draft_row_stride < V)
    return fail(SPECV_ERR_INVALID_ARG, "row stride smaller than V");
  if (B > 1 && (a->target_batch_stride < K * a->target_row_stride + V ||
                a->draft_batch_stride < (K - 1) * a->draft_row_stride + V))
    return fail(SPECV_ERR_INVALID_ARG, "batch stride too small for K+1 target / K draft rows");
  const size_t need = specv_verify_workspace_bytes(B, K, V, a->dtype);
  if (!workspace || workspace_bytes < need)
    return fail(SPECV_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, workspace_bytes);
  if (!aligned(workspace, 256)) return fail(SPECV_ERR_WORKSPACE, "workspace not 256-byte aligned");

  const int C = pick_cluster(V);
  const int vw = vec_width(a->dtype);
  const int64_t L = slice_len(V, C, vw);
  const int64_t ntiles = ((L / vw) + kThreads - 1) / kThreads;
  const size_t smem = static_cast<size_t>(ntiles) * kWarps * sizeof(float);
  if (smem > kMaxSegSmem) return fail(SPECV_ERR_UNSUPPORTED, "V=%d too large for one cluster", V);
  const int64_t units = static_cast<int64_t>(B) * (K + 1);
  if (units * C > 0x7fffffffLL) return fail(SPECV_ERR_UNSUPPORTED, "B*(K+1) too large");

  VerifyParams p;
  p.zt = a->target_logits;
  p.t_bs = a->target_batch_stride;
  p.t_rs = a->target_row_stride;
  p.zd = a->draft_logits;
  p.d_bs = a->draft_batch_stride;
  p.d_rs = a->draft_row_stride;
  p.tokens = a->draft_tokens;
  p.temp = a->temperature;
  p.unif = a->uniforms;
  p.units = static_cast<UnitOut*>(workspace);
  p.B = B;
  p.K = K;
  p.V = V;
  p.C = C;
  p.L = static_cast<int32_t>(L);

  const bool vec = vec_ok(a->target_logits, a->target_batch_stride, a->target_row_stride, es) &&
                   vec_ok(a->draft_logits, a->draft_batch_stride, a->draft_row_stride, es);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (a->dtype == SPECV_BF16)
    e = vec ? launch_clustered(verify_units_kernel<0, true>, C, units, smem, s, p)
            : launch_clustered(verify_units_kernel<0, false>, C, units, smem, s, p);
  else
    e = vec ? launch_clustered(verify_units_kernel<1, true>, C, units, smem, s, p)
            : launch_clustered(verify_units_kernel<1, false>, C, units, smem, s, p);
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "verify launch: %s", cudaGetErrorString(e));
  verify_finalize_kernel<<<(B + 127) / 128, 128, 0, s>>>(
      p.units, a->draft_tokens, B, K, a->accept_len, a->out_tokens, a->p_draft, a->q_draft,
      a->row_status);
  e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "finalize launch: %s", cudaGetErrorString(e));
  g_launches = 2;
  return ok();
}

size_t specv_predict_workspace_bytes(int32_t B, int32_t K, int32_t V, int32_t F, int32_t dtype) {
  (void)V;
  (void)F;
  (void)dtype;
  if (B <= 0 || K < 1) return 0;
  return round_up(static_cast<size_t>(B) * (K + 1) * sizeof(int32_t), 256);
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
  const size_t need = a->row_status ? specv_predict_workspace_bytes(B, K, V, F, a->dtype) : 0;
  if (need && (!workspace || workspace_bytes < need))
    return fail(SPECV_ERR_WORKSPACE, "workspace needs %zu bytes, got %zu", need, workspace_bytes);
  if (need && !aligned(workspace, 256))
    return fail(SPECV_ERR_WORKSPACE, "workspace not 256-byte aligned");

  const int C = pick_cluster(V);
  const int vw = vec_width(a->dtype);
  const int64_t L = slice_len(V, C, vw);
  const int64_t units = static_cast<int64_t>(B) * (K + 1);
  if (units * C > 0x7fffffffLL) return fail(SPECV_ERR_UNSUPPORTED, "B*(K+1) too large");
  PredictParams p;
  p.zd = a->draft_logits;
  p.d_bs = a->draft_batch_stride;
  p.d_rs = a->draft_row_stride;
  p.tokens = a->draft_tokens;
  p.keys = a->keys;
  p.key_logits = a->key_logits;
  p.unit_status = a->row_status ? static_cast<int32_t*>(workspace) : nullptr;
  p.B = B;
  p.K = K;
  p.V = V;
  p.F = F;
  p.C = C;
  p.L = static_cast<int32_t>(L);
  const bool vec = vec_ok(a->draft_logits, a->draft_batch_stride, a->draft_row_stride, es);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e;
  if (a->dtype == SPECV_BF16)
    e = vec ? launch_clustered(predict_units_kernel<0, true>, C, units, 0, s, p)
            : launch_clustered(predict_units_kernel<0, false>, C, units, 0, s, p);
  else
    e = vec ? launch_clustered(predict_units_kernel<1, true>, C, units, 0, s, p)
            : launch_clustered(predict_units_kernel<1, false>, C, units, 0, s, p);
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "predict launch: %s", cudaGetErrorString(e));
  g_launches = 1;
  if (a->row_status) {
    predict_finalize_kernel<<<(B + 127) / 128, 128, 0, s>>>(p.unit_status, B, K, a->row_status);
    e = cudaGetLastError();
    if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "finalize launch: %s", cudaGetErrorString(e));
    g_launches = 2;
  }
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
  check_hit_kernel<<<(B + 127) / 128, 128, 0, s>>>(B, K, F, keys, accept_len, out_tokens, hit);
  const cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return fail(SPECV_ERR_CUDA, "check_hit launch: %s", cudaGetErrorString(e));
  g_launches = 1;
  return ok();
}

}  // extern "C"
