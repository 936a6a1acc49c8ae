// Kernel launchers, instantiated per mode in the k_*.cu translation units
// (compiled in parallel); specv_api.cu sees only their declarations.
#pragma once

#include <algorithm>
#include <atomic>

#include "launch.cuh"

namespace specv {

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
  if (smem > 0) {  // static + dynamic shared memory may pass the 48 KB default
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(units * C), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  // The kernel waits (griddepcontrol.wait) for the one before it on the
  // stream, so it may be scheduled while that one drains.
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(C);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k, p);
}

// One launch that may be scheduled while the kernel before it on the stream
// drains (it waits for that kernel with griddepcontrol.wait).
template <typename Kern, typename Params>
cudaError_t launch_dependent(Kern k, int64_t blocks, size_t smem, cudaStream_t stream, const Params& p) {
  if (smem > 0) {
    const cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k, p);
}

template <typename Kern, typename Params>
cudaError_t launch_plain(Kern k, int64_t blocks, size_t smem, cudaStream_t s, const Params& p) {
  if (smem > 0) {  // static + dynamic shared memory may pass the 48 KB default
    const cudaError_t e =
        cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
  }
  k<<<static_cast<unsigned>(blocks), kThreads, smem, s>>>(p);
  return cudaGetLastError();
}

// Persistent row-statistics kernel: as many CTAs as are resident at once on
// the GPU (at most one per work item), each with the ring in dynamic shared
// memory.  The occupancy query is made once per kernel and ring size.
template <int DT, int MODE>
cudaError_t launch_ring(int64_t items, int sms, cudaStream_t s, const StatsParams& p) {
  auto k = stats_ring_kernel<DT, MODE>;
  const size_t smem = static_cast<size_t>(p.stages) * 2 * kTripBytes;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  static std::atomic<int> occ_cache[kMaxStages + 1];
  int occ = occ_cache[p.stages].load(std::memory_order_relaxed);
  if (occ <= 0) {
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, k, kRingThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) occ = 1;
    occ_cache[p.stages].store(occ, std::memory_order_relaxed);
  }
  const int64_t grid = std::min<int64_t>(items, static_cast<int64_t>(occ) * sms);
  k<<<static_cast<unsigned>(grid), kRingThreads, smem, s>>>(p);
  return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_stats(int dtype, bool vec, bool persistent, int sms, int64_t items, cudaStream_t s,
                         const StatsParams& p) {
  const size_t ring_smem = static_cast<size_t>(p.stages) * 2 * kTripBytes;
  if (dtype == SPECV_BF16) {
    if (!vec) return launch_plain(stats_kernel<0, false, MODE>, items, 0, s, p);
    return persistent ? launch_ring<0, MODE>(items, sms, s, p)
                             : launch_plain(stats_kernel<0, true, MODE>, items, ring_smem, s, p);
  }
  if (!vec) return launch_plain(stats_kernel<1, false, MODE>, items, 0, s, p);
  return persistent ? launch_ring<1, MODE>(items, sms, s, p)
                           : launch_plain(stats_kernel<1, true, MODE>, items, ring_smem, s, p);
}

template <int MODE>
cudaError_t launch_decide(int dtype, bool vec, int CB, int64_t B, size_t smem, cudaStream_t s,
                          const DecideParams& p) {
  if (dtype == SPECV_BF16)
    return vec ? launch_clustered(decide_kernel<0, true, MODE>, CB, B, smem, s, p)
               : launch_clustered(decide_kernel<0, false, MODE>, CB, B, smem, s, p);
  return vec ? launch_clustered(decide_kernel<1, true, MODE>, CB, B, smem, s, p)
             : launch_clustered(decide_kernel<1, false, MODE>, CB, B, smem, s, p);
}

}  // namespace specv
