// Kernel instantiations of the verify mode (one translation unit per mode,
// compiled in parallel).
#include "launch_impl.cuh"

namespace specv {
SPECV_LAUNCHERS(kModeVerify, )
}  // namespace specv
