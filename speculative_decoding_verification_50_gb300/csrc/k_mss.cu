// Kernel instantiations of the mss mode (one translation unit per mode,
// compiled in parallel).
#include "launch_impl.cuh"

namespace specv {
SPECV_LAUNCHERS(kModeMss, )
}  // namespace specv
