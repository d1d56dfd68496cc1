// Host-side kernel launch with an optional programmatic dependency on the
// kernel before it on the stream (see pdl_wait / pdl_trigger in common.cuh).
// The first kernel of a public call is launched without it, so it starts only
// after everything the caller queued earlier has completed; the kernels after
// it in the same call overlap their prologues (barrier setup, tensor-memory
// allocation, weight prefetch) with the tail of their predecessor.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <utility>

namespace llama {

// Kernels this process has launched through the library (every device);
// read by llama_launch_count().
extern std::atomic<unsigned long long> g_launch_count;

inline cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) g_launch_count.fetch_add(1, std::memory_order_relaxed);
  return e;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_kernel(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl,
                          Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return counted(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

// The same, for a kernel launched in thread-block clusters of cluster_x CTAs.
template <typename... KArgs, typename... Args>
cudaError_t launch_kernel_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                                  bool pdl, int cluster_x, Args&&... args) {
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = static_cast<unsigned>(cluster_x);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 2 : 1;
  return counted(cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...));
}

}  // namespace llama
