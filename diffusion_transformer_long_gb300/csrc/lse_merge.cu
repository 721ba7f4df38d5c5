// Exact log-sum-exp merge of p KV-chunk partials (one Ring-attention hop's
// combination, applied to all p virtual ranks at once):
//   M = max_c lse_c,  lse = M + ln sum_c exp(lse_c - M),  O = sum_c exp(lse_c - lse) O_c
// (arganzheng.life multi-GPU diffusion parallelism, section 4.2 Ring: the
// per-round blocks are combined by online softmax accumulation).
//
// HBM-bound: it reads p*(D*sizeof(partial) + 4) bytes and writes
// D*sizeof(out) + 4 bytes per query row.  Each thread owns one 16-byte vector
// of one row (4 fp32 or 8 bf16 partial elements); the threads of a row are
// consecutive, so every partial row is read by fully coalesced 16-byte
// streaming loads.  The per-row arithmetic is in merge_math.cuh.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "merge_math.cuh"

namespace ditattn {
namespace {

constexpr int kMergeThreads = 256;

template <typename PT, typename OT, int D>
__global__ void __launch_bounds__(kMergeThreads, 4) lse_merge_kernel(
    const PT* __restrict__ partials, const float* __restrict__ lses, int p, long long rows,
    OT* __restrict__ out, float* __restrict__ lse_out) {
  constexpr int kV = merge::Vec<PT>::kN;
  constexpr int kTpr = D / kV;  // threads per row
  const long long gt = static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x;
  const long long row = gt / kTpr;
  if (row >= rows) return;
  const int col = static_cast<int>(gt % kTpr) * kV;
  merge::merge_row<PT, OT, D>(partials, lses, p, rows, row, col, out, lse_out);
}

template <typename PT, typename OT, int D>
cudaError_t launch_typed(const MergeLaunch& a, cudaStream_t st) {
  constexpr int kTpr = D / merge::Vec<PT>::kN;
  const long long threads = a.rows * kTpr;
  const long long blocks = (threads + kMergeThreads - 1) / kMergeThreads;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  lse_merge_kernel<PT, OT, D><<<static_cast<unsigned>(blocks), kMergeThreads, 0, st>>>(
      static_cast<const PT*>(a.partials), a.lses, a.p, a.rows, static_cast<OT*>(a.out), a.lse);
  return cudaGetLastError();
}

template <typename PT, typename OT>
cudaError_t launch_d(const MergeLaunch& a, cudaStream_t st) {
  return a.d == 64 ? launch_typed<PT, OT, 64>(a, st) : launch_typed<PT, OT, 128>(a, st);
}

}  // namespace

cudaError_t launch_merge(const MergeLaunch& a, cudaStream_t st) {
  if (a.part_f32)
    return a.out_f32 ? launch_d<float, float>(a, st) : launch_d<float, __nv_bfloat16>(a, st);
  return a.out_f32 ? launch_d<__nv_bfloat16, float>(a, st)
                   : launch_d<__nv_bfloat16, __nv_bfloat16>(a, st);
}

}  // namespace ditattn
