// Kernel instantiations of outcome prediction alone (row statistics).
#include "launch_impl.cuh"

namespace specv {
template cudaError_t launch_stats<kModePredict>(int, bool, bool, int, int64_t, cudaStream_t,
                                                const StatsParams&);
}  // namespace specv
