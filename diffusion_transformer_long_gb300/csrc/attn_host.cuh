// Host-side launch of the attention kernel's instantiations, shared by the translation
// units that instantiate them (attn_fwd.cu: the forms whose epilogue warpgroup drains O;
// attn_fwd_short.cu: the forms for short work items, whose softmax warpgroups drain O).
#pragma once

#include <cuda_runtime.h>

#include <mutex>

#include "attn_kernel.cuh"

namespace ditattn {
namespace host {

// Streaming multiprocessors of the current device, cached per device.
inline int sm_count() {
  static int cached[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 1;
  if (cached[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1)
      n = 1;
    cached[dev] = n;
  }
  return cached[dev];
}

// Launches one instantiation on `st` with a persistent grid: one CTA per SM (shared memory
// and TMEM allow no more), capped by `grid_limit` (0: none) and by the work items.
template <int D, bool kF32, bool kAccum = false, bool kLse = true, bool kSoftDrain = false>
cudaError_t launch_typed(const AttnParams& prm, cudaStream_t st, int grid_limit) {
  constexpr int kSmem = AttnSmem<D>::kBytes;
  auto kern = attn_fwd_kernel<D, kF32, kAccum, kLse, kSoftDrain>;
  // The shared-memory opt-in is set once per device and instantiation, so that later
  // launches are only the launch itself.
  static std::mutex mu;
  static bool done[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!done[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
      if (e != cudaSuccess) return e;
      done[dev] = true;
    }
  }
  int ctas = sm_count();
  if (grid_limit > 0 && grid_limit < ctas) ctas = grid_limit;
  if (prm.num_items < ctas) ctas = prm.num_items;
  const dim3 grid(static_cast<unsigned>(ctas));
  kern<<<grid, kThreads, kSmem, st>>>(prm);
  return cudaGetLastError();
}

// Work items of at most this many KV tiles take the soft-drain form (attn_fwd_short.cu).
constexpr int kShortItemTiles = 16;
// The soft-drain instantiations (attn_fwd_short.cu): fused/chunk/split passes, with or
// without the LSE; bf16 output needs prm.tm_o (the output's TMA map).
cudaError_t launch_short(const AttnParams& prm, int d, bool out_f32, bool lse, cudaStream_t st,
                         int grid_limit);

}  // namespace host
}  // namespace ditattn
