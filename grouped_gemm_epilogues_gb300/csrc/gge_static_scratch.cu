// gge_gemm_act_static_scratch: the fused GEMM + activation call for callers
// that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at the point where they run the GEMM:
// for example, a host framework that owns all device memory through its own
// arena or caching allocator and forbids outside allocations, or a
// latency-critical path that must not touch the allocator (an allocation can
// synchronise the device).  The regular entry points take a caller-owned
// workspace; this one uses a fixed scratch area that lives in the library
// itself instead, so the caller passes only its inputs and outputs.
//
// The scratch is a file-scope __device__ array (kStaticScratchBytes): every
// GPU that loads the library keeps it until the process exits.  In host code
// the array's name is only a stand-in for the device symbol, never a device
// address, so its address is looked up once per device with
// cudaGetSymbolAddress (on that device, during the first call there) and that
// address is what the kernel receives.
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/gge.h"

namespace {

constexpr size_t kStaticScratchBytes = 1024;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

struct DeviceScratch {
  std::once_flag once;
  void* ptr = nullptr;
  cudaError_t err = cudaSuccess;
};

DeviceScratch g_device_scratch[64];

// Device address of the scratch array on the current device (set up once).
void* scratch_address(gge_status* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    *status = GGE_ERR_CUDA;
    return nullptr;
  }
  DeviceScratch& d = g_device_scratch[dev];
  std::call_once(d.once, [&d] {
    void* p = nullptr;
    d.err = cudaGetSymbolAddress(&p, g_static_scratch);
    d.ptr = p;
  });
  if (d.err != cudaSuccess || d.ptr == nullptr) {
    *status = GGE_ERR_CUDA;
    return nullptr;
  }
  return d.ptr;
}

}  // namespace

extern "C" gge_status gge_gemm_act_static_scratch(const gge_gemm_args* args,
                                                  gge_stream_t stream) {
  if (args == nullptr) return GGE_ERR_INVALID_ARG;
  // the status words only: with no room for partial sums the last wave is not
  // split (the fixed area is small)
  const size_t need = 256;
  if (need > kStaticScratchBytes) return GGE_ERR_WORKSPACE;
  gge_status status = GGE_OK;
  void* scratch = scratch_address(&status);
  if (scratch == nullptr) return status;
  // the area keeps the previous call's contents: the status words must start at zero
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(scratch, 0, need, st) != cudaSuccess) return GGE_ERR_CUDA;
  return gge_gemm_act(args, scratch, need, stream);
}
