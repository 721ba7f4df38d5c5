// The library's fixed device scratch, for dit_attn_chunk_fwd_splitkv_noalloc: split-KV
// attention whose partials live here instead of in a caller-provided workspace, so that
// call allocates nothing.  In its own translation unit so that the array's device module
// is loaded only by processes that use it.
#include <cuda_runtime.h>

#include <mutex>

#include "launch.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ditattn::kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;

}  // namespace

namespace ditattn {

// Device address of the scratch array on the current device: looked up once per device
// with that device current (cudaGetSymbolAddress); null if the lookup fails.
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
