// The library's fixed device scratch, for dit_attn_chunk_fwd_splitkv_noalloc: split-KV
// attention whose partials live here instead of in a caller-provided workspace, so that
// call allocates nothing.  The array is part of the library's device code: the CUDA runtime
// reserves it on a device when it loads that code there, which under the default lazy
// module loading is the first call that uses the device (under CUDA_MODULE_LOADING=EAGER,
// as soon as the library is loaded), so every process that uses the library holds it.  On a
// device too full to take it, that first call fails with DIT_ERR_CUDA.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ditattn::kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

}  // namespace

namespace ditattn {

// Device address of the scratch array on the current device: looked up once per device
// number with that device current (cudaGetSymbolAddress); null if the lookup fails.  The
// cache assumes the runtime's primary context on each device (no cudaDeviceReset between
// calls, no other context current).
void* noalloc_scratch() {
  static std::mutex mu;
  static void* cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    cached[dev] = p;
  }
  return cached[dev];
}

}  // namespace ditattn
