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

// The array's device address per device, filled in by the first successful
// lookup on that device.  A failed lookup is not cached: the next call tries
// again (a call made during stream capture, or after a sticky error, fails
// without spoiling later calls).
std::mutex g_scratch_mu;
void* g_scratch_ptr[64] = {};

// Device address of the scratch array on the current device.
void* scratch_address(gge_status* status) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    *status = GGE_ERR_CUDA;
    return nullptr;
  }
  std::lock_guard<std::mutex> g(g_scratch_mu);
  if (g_scratch_ptr[dev] == nullptr) {
    void* p = nullptr;
    const cudaError_t e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess || p == nullptr) {
      cudaGetLastError();  // clear the error so that the caller's next CUDA call is not blamed
      *status = GGE_ERR_CUDA;
      return nullptr;
    }
    g_scratch_ptr[dev] = p;
  }
  return g_scratch_ptr[dev];
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
  // The area keeps the previous call's contents.  The scheduler counters after
  // the first 16 bytes must start at zero; the error record in those 16 bytes
  // is kept until gge_read_static_scratch_status reads and clears it, so that an
  // error is not lost to the next call.  (A __device__ array starts zeroed.)
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemsetAsync(static_cast<unsigned char*>(scratch) + 16, 0, need - 16, st) != cudaSuccess)
    return GGE_ERR_CUDA;
  return gge_gemm_act(args, scratch, need, stream);
}

// The device status that calls of gge_gemm_act_static_scratch on the current
// device recorded in the library's scratch area (the same words
// gge_read_device_status reads from a caller's workspace).
extern "C" gge_status gge_read_static_scratch_status(gge_stream_t stream, int32_t* detail) {
  gge_status status = GGE_OK;
  void* scratch = scratch_address(&status);
  if (scratch == nullptr) return status;
  return gge_read_device_status(scratch, stream, detail);
}
