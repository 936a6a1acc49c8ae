// Kernel instantiations of the sample mode (one translation unit per mode,
// compiled in parallel).
#include "launch_impl.cuh"
#include "sample_kernel.cuh"

namespace specv {
SPECV_LAUNCHERS(kModeSample, )

cudaError_t launch_sample_rows(int dtype, int64_t rows, size_t smem, cudaStream_t s, const DecideParams& p) {
  const int64_t blocks = (rows + kWarps - 1) / kWarps;
  return dtype == SPECV_BF16 ? launch_dependent(sample_rows_kernel<0>, blocks, smem, s, p)
                             : launch_dependent(sample_rows_kernel<1>, blocks, smem, s, p);
}
}  // namespace specv
