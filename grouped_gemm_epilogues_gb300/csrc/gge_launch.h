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

template <int BN, bool GATHER>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const Params& p,
                        const LaunchShape& shape, cudaStream_t stream);

template <int BN, bool GATHER>
int kernel_threads();

}  // namespace gge
