// The attention kernel's soft-drain instantiations (the softmax warpgroups drain O; used
// when every work item has few KV tiles, e.g. video queries against a few hundred
// replicated text keys), in a translation unit of their own so that they compile in
// parallel with the others.
#include <cuda_runtime.h>

#include "attn_host.cuh"

namespace ditattn {
namespace host {

template <int D, bool kLse>
cudaError_t launch_short_d(const AttnParams& prm, bool out_f32, cudaStream_t st, int grid_limit) {
  return out_f32 ? launch_typed<D, true, false, kLse, true>(prm, st, grid_limit)
                 : launch_typed<D, false, false, kLse, true>(prm, st, grid_limit);
}

cudaError_t launch_short(const AttnParams& prm, int d, bool out_f32, bool lse, cudaStream_t st,
                         int grid_limit) {
  if (d == 64)
    return lse ? launch_short_d<64, true>(prm, out_f32, st, grid_limit)
               : launch_short_d<64, false>(prm, out_f32, st, grid_limit);
  return lse ? launch_short_d<128, true>(prm, out_f32, st, grid_limit)
             : launch_short_d<128, false>(prm, out_f32, st, grid_limit);
}

}  // namespace host
}  // namespace ditattn
