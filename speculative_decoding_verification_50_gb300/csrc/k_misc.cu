// The kernels without a mode: the outcome keys alone (specv_predict_outcomes)
// and the hit check (specv_check_hit).
#include "launch.cuh"

namespace specv {

__global__ void __launch_bounds__(kThreads) predict_keys_kernel(const PredictKeysParams P) {
  __shared__ int32_t status_all;
  __shared__ WarpKeys wkeys[kWarps];
  const int b = blockIdx.x;
  const int K = P.K, F = P.F;
  const int lane = threadIdx.x & 31;
  const int warp = threadIdx.x >> 5;
  const int64_t u0 = static_cast<int64_t>(b) * (K + 1);
  if (threadIdx.x == 0) status_all = 0;
  pdl_wait_primary();  // records and candidates come from the row-statistics kernel
  __syncthreads();
  for (int k = warp; k <= K; k += kWarps) {
    const int64_t u = u0 + k;
    int bad = 0;
    for (int q = lane; q < P.nchunk; q += 32) bad |= P.recs[u * P.nchunk + q].bad;
    bad = __reduce_or_sync(0xffffffffu, bad);
    const int x = (k < K) ? P.tokens[static_cast<int64_t>(b) * K + k] : 0;
    const int status = ((bad & 1) ? kNonFinite : 0) | ((bad & 2) ? kTimeout : 0) |
                       ((x < 0 || x >= P.V) ? kBadToken : 0);
    const WarpTopF L = warp_keys(P.cand_v + u * P.nchunk * F, P.cand_i + u * P.nchunk * F,
                                 P.nchunk * F, F, lane, wkeys[warp]);
    if (lane < F) {
      const bool good = status == 0 && lane < P.fk[k] && L.i != INT_MAX;
      P.keys[u * F + lane] = good ? L.i : -1;
      if (P.key_logits) P.key_logits[u * F + lane] = good ? L.v : neg_inf();
    }
    if (lane == 0 && status) atomicOr(&status_all, status);
  }
  __syncthreads();
  if (threadIdx.x == 0 && P.row_status) P.row_status[b] = status_all;
}

__global__ void check_hit_kernel(int B, int K, int F, const int32_t* __restrict__ keys,
                                 const int32_t* __restrict__ accept_len,
                                 const int32_t* __restrict__ out_tokens,
                                 uint8_t* __restrict__ hit) {
  const int b = blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= B) return;
  const int n = accept_len[b];
  uint8_t h = 0;
  if (n >= 0 && n <= K) {
    const int t = out_tokens[static_cast<int64_t>(b) * (K + 1) + n];
    if (t >= 0) {
      const int32_t* kk = keys + (static_cast<int64_t>(b) * (K + 1) + n) * F;
      for (int f = 0; f < F; ++f) h |= (kk[f] == t);
    }
  }
  hit[b] = h;
}


cudaError_t launch_predict_keys(const PredictKeysParams& kp, int B, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(B), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.stream = s;
  // scheduled while the row-statistics kernel drains; it waits for it
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, predict_keys_kernel, kp);
  return e == cudaSuccess ? cudaGetLastError() : e;
}

cudaError_t launch_check_hit(int B, int K, int F, const int32_t* keys, const int32_t* accept_len,
                             const int32_t* out_tokens, uint8_t* hit, cudaStream_t s) {
  check_hit_kernel<<<(B + 127) / 128, 128, 0, s>>>(B, K, F, keys, accept_len, out_tokens, hit);
  return cudaGetLastError();
}

}  // namespace specv
