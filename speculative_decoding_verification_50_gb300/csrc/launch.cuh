// Declarations of the kernel launchers (defined in launch_impl.cuh,
// instantiated per mode in k_verify.cu, k_ssd.cu, k_sample.cu, k_mss.cu,
// k_predict.cu; the kernels without a mode in k_misc.cu).
#pragma once

#include "specv.h"
#include "decide_kernel.cuh"

namespace specv {

// Row statistics (kernel A): register path (vec = false), staged path, or the
// persistent path (persistent, sms = the SM count).
template <int MODE>
cudaError_t launch_stats(int dtype, bool vec, bool persistent, int sms, int64_t items, cudaStream_t s,
                         const StatsParams& p);
// Decision kernel (kernel B): B clusters of CB CTAs.
template <int MODE>
cudaError_t launch_decide(int dtype, bool vec, int CB, int64_t B, size_t smem, cudaStream_t s,
                          const DecideParams& p);
// The sampler's decision with one warp per row (aligned rows whose records
// carry their first halves): ceil(rows / 8) CTAs, `smem` bytes of segment
// sums for the CTA-wide pass over a whole row.
cudaError_t launch_sample_rows(int dtype, int64_t rows, size_t smem, cudaStream_t s, const DecideParams& p);
cudaError_t launch_predict_keys(const PredictKeysParams& kp, int B, cudaStream_t s);
cudaError_t launch_check_hit(int B, int K, int F, const int32_t* keys, const int32_t* accept_len,
                             const int32_t* out_tokens, uint8_t* hit, cudaStream_t s);

#define SPECV_LAUNCHERS(MODE, EXT)                                                             \
  EXT template cudaError_t launch_stats<MODE>(int, bool, bool, int, int64_t, cudaStream_t,   \
                                              const StatsParams&);                            \
  EXT template cudaError_t launch_decide<MODE>(int, bool, int, int64_t, size_t, cudaStream_t, \
                                               const DecideParams&);

SPECV_LAUNCHERS(kModeVerify, extern)
SPECV_LAUNCHERS(kModeSsd, extern)
SPECV_LAUNCHERS(kModeSample, extern)
SPECV_LAUNCHERS(kModeMss, extern)
extern template cudaError_t launch_stats<kModePredict>(int, bool, bool, int, int64_t, cudaStream_t,
                                                       const StatsParams&);

}  // namespace specv
