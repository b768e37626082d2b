// launch_util.cuh -- launching the persistent pipelines, with a cluster
// dimension for CTA-pair kernels, and the number of CTAs (pairs) that can be
// resident at once.
#pragma once

#include <cuda_runtime.h>

#include "vocab_pipeline.cuh"

namespace flp {

template <typename... KArgs, typename... Args>
cudaError_t launch_persistent(void (*kern)(KArgs...), int grid, int threads, int smem_bytes, int cg,
                              cudaStream_t stream, Args &&...args) {
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  if (cg > 1) {
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cg;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

// CTAs (cg = 1) or CTA pairs (cg = 2) of `kern` that fit on the device at once.
template <typename... KArgs>
int resident_units(void (*kern)(KArgs...), int threads, int smem_bytes, int cg, int num_sms) {
  if (cg == 1) return num_sms;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
      cudaSuccess)
    return num_sms / cg;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(num_sms));
  cfg.blockDim = dim3(static_cast<unsigned>(threads));
  cfg.dynamicSmemBytes = static_cast<size_t>(smem_bytes);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cg;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    return num_sms / cg;
  }
  return n < num_sms / cg ? n : num_sms / cg;
}

}  // namespace flp
