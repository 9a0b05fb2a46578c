// Shared body of the per-instantiation translation units.
#pragma once

#include <atomic>

#include "gge_kernel.cuh"
#include "gge_launch.h"

namespace gge {

template <int BN, bool GATHER, int CG, bool TR = false>
cudaError_t set_smem_limit(size_t smem) {
  auto kern = gemm_kernel<BN, GATHER, CG, TR>;
  // the dynamic shared-memory limit is a per-device function attribute
  static std::atomic<size_t> smem_set[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64 || smem_set[dev].load() < smem) {
    RelaxedCaptureMode relaxed;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) smem_set[dev].store(smem);
  }
  return cudaSuccess;
}

template <int BN, bool GATHER, int CG, bool TR>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const Params& p,
                        const LaunchShape& shape, cudaStream_t stream) {
  auto kern = gemm_kernel<BN, GATHER, CG, TR>;
  cudaError_t e = set_smem_limit<BN, GATHER, CG, TR>(shape.smem);
  if (e != cudaSuccess) return e;
  cudaLaunchAttribute attr[2];
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(shape.grid, 1, 1);
  cfg.blockDim = dim3(shape.threads, 1, 1);
  cfg.dynamicSmemBytes = shape.smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  // programmatic dependent launch: this grid may start while the previous kernel
  // in the stream finishes (the kernel waits for it before reading global memory)
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.numAttrs = 1;
  if (shape.cluster > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = shape.cluster;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.numAttrs = 2;
  }
  return cudaLaunchKernelEx(&cfg, kern, tmA, tmB, p);
}

template <int BN, bool GATHER, int CG>
int kernel_threads() {
  return KernelCfg<BN, GATHER, CG>::kThreads;
}

template <int BN, bool GATHER, int CG>
int max_active_units(size_t smem, int cluster) {
  auto kern = gemm_kernel<BN, GATHER, CG>;
  if (set_smem_limit<BN, GATHER, CG>(smem) != cudaSuccess) return -1;
  if (cluster <= 1) {
    int per_sm = 0, dev = 0, sms = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, KernelCfg<BN, GATHER, CG>::kThreads,
                                                      smem) != cudaSuccess)
      return -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return -1;
    if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    return per_sm * sms;
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(cluster * 64, 1, 1);
  cfg.blockDim = dim3(KernelCfg<BN, GATHER, CG>::kThreads, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return -1;
  return n;
}

#define GGE_INSTANTIATE(BN, GATHER, CG)                                                      \
  template cudaError_t launch_gemm<BN, GATHER, CG, false>(const CUtensorMap&,              \
                                                          const CUtensorMap&, const Params&, \
                                                          const LaunchShape&, cudaStream_t); \
  template int kernel_threads<BN, GATHER, CG>();                                           \
  template int max_active_units<BN, GATHER, CG>(size_t, int);

// The transposed-output (swap_ab) instance of a one-CTA TMA tile.
#define GGE_INSTANTIATE_TRANS(BN)                                                             \
  template cudaError_t launch_gemm<BN, false, 1, true>(const CUtensorMap&, const CUtensorMap&, \
                                                       const Params&, const LaunchShape&,      \
                                                       cudaStream_t);

}  // namespace gge
