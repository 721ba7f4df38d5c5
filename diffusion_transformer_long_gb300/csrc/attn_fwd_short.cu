// The attention kernel's soft-drain instantiations (the softmax warpgroups drain O; used
// when every work item has few KV tiles, e.g. video queries against a few hundred
// replicated text keys), in a translation unit of their own so that they compile in
// parallel with the others.
#include <cuda_runtime.h>

#include "attn_host.cuh"

namespace ditattn {
namespace host {

cudaError_t launch_short(const AttnParams& prm, int d, bool out_f32, cudaStream_t st,
                         int grid_limit) {
  if (d == 64)
    return out_f32 ? launch_typed<64, true, false, true, true>(prm, st, grid_limit)
                   : launch_typed<64, false, false, true, true>(prm, st, grid_limit);
  return out_f32 ? launch_typed<128, true, false, true, true>(prm, st, grid_limit)
                 : launch_typed<128, false, false, true, true>(prm, st, grid_limit);
}

}  // namespace host
}  // namespace ditattn
