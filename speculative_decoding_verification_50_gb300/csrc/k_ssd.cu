// Kernel instantiations of the ssd mode (one translation unit per mode,
// compiled in parallel).
#include "launch_impl.cuh"

namespace specv {
SPECV_LAUNCHERS(kModeSsd, )
}  // namespace specv
