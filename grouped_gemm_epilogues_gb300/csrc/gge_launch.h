// Launch entry points of the kernel instantiations (one translation unit each).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gge.h"
#include "gge_params.h"

namespace gge {

// Device queries that are not stream work (a function's shared-memory limit,
// occupancy) are refused while the calling thread captures a stream in the
// default (global) mode.  For the lifetime of this object the thread is in
// relaxed mode, which allows them, so a launch shape's first call on a device
// may itself be captured into a CUDA graph.
struct RelaxedCaptureMode {
  cudaStreamCaptureMode saved = cudaStreamCaptureModeRelaxed;
  RelaxedCaptureMode() { cudaThreadExchangeStreamCaptureMode(&saved); }
  ~RelaxedCaptureMode() { cudaThreadExchangeStreamCaptureMode(&saved); }
  RelaxedCaptureMode(const RelaxedCaptureMode&) = delete;
  RelaxedCaptureMode& operator=(const RelaxedCaptureMode&) = delete;
};

struct LaunchShape {
  int grid;
  int threads;
  size_t smem;
  int cluster;  // CTAs per cluster: 1, or 2 (a CTA pair)
};

// TR: the swap_ab instance, whose epilogue stores C / D / PostAct transposed.
template <int BN, bool GATHER, int CG, bool TR = false>
cudaError_t launch_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const Params& p,
                        const LaunchShape& shape, cudaStream_t stream);

template <int BN, bool GATHER, int CG>
int kernel_threads();

// Clusters of `cluster` CTAs (with `smem` bytes each) that can be resident at once.
template <int BN, bool GATHER, int CG>
int max_active_units(size_t smem, int cluster);

// Host-only validation of one call of entry point `op` (GGE_OP_*) as it would
// be planned, without launching or touching the GPU (gge_api.cu).
int32_t validate_op(const ::gge_gemm_args* args, int32_t op, int32_t num_groups);

}  // namespace gge
