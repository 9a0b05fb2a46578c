// Shared body of the per-instantiation translation units.
#pragma once

#include <atomic>

#include "gge_kernel.cuh"
#include "gge_launch.h"

namespace gge {

template <int BN, bool GATHER>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const Params& p,
                        const LaunchShape& shape, cudaStream_t stream) {
  auto kern = gemm_kernel<BN, GATHER>;
  // the dynamic shared-memory limit is a per-device function attribute
  static std::atomic<size_t> smem_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || smem_set[dev].load() < shape.smem) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(shape.smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) smem_set[dev].store(shape.smem);
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(shape.grid, 1, 1);
  cfg.blockDim = dim3(shape.threads, 1, 1);
  cfg.dynamicSmemBytes = shape.smem;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
}

template <int BN, bool GATHER>
int kernel_threads() {
  return KernelCfg<BN, GATHER>::kThreads;
}

#define GGE_INSTANTIATE(BN, GATHER)                                                          \
  template cudaError_t launch_gemm<BN, GATHER>(const CUtensorMap&, const CUtensorMap&,     \
                                               const Params&, const LaunchShape&,          \
                                               cudaStream_t);                              \
  template int kernel_threads<BN, GATHER>();

}  // namespace gge
