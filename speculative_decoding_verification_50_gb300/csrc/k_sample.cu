// Kernel instantiations of the sample mode (one translation unit per mode,
// compiled in parallel).
#include "launch_impl.cuh"

namespace specv {
SPECV_LAUNCHERS(kModeSample, )
}  // namespace specv
