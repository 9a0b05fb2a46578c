// Launch entry points of the kernel instantiations (one translation unit each).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "gge_params.h"

namespace gge {

struct LaunchShape {
  int grid;
  int threads;
  size_t smem;
};

template <int BN, bool GATHER, int CG>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const Params& p,
                        const LaunchShape& shape, cudaStream_t stream);

template <int BN, bool GATHER, int CG>
int kernel_threads();

// Clusters of CG CTAs (with `smem` bytes each) that can be resident at once.
template <int BN, bool GATHER, int CG>
int max_active_units(size_t smem);

}  // namespace gge
