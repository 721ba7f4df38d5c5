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
// streaming loads, and a batch of up to 8 chunks' loads is issued before any
// of them is used.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"
#include "sm103_ptx.cuh"

namespace ditattn {
namespace {

constexpr int kMergeThreads = 256;
constexpr int kBatch = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int kN = 4;
  __device__ static void load(const float* p, float (&x)[4]) {
    const float4 v = __ldcs(reinterpret_cast<const float4*>(p));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  __device__ static void load(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 v = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

template <int N>
__device__ __forceinline__ void store_out(float* dst, const float (&a)[N]) {
#pragma unroll
  for (int i = 0; i < N; i += 4)
    *reinterpret_cast<float4*>(dst + i) = make_float4(a[i], a[i + 1], a[i + 2], a[i + 3]);
}
template <int N>
__device__ __forceinline__ void store_out(__nv_bfloat16* dst, const float (&a)[N]) {
  static_assert(N % 8 == 0 || N == 4, "vector width");
  if constexpr (N == 4) {
    uint2 w;
    w.x = ptx::pack_bf16x2(a[0], a[1]);
    w.y = ptx::pack_bf16x2(a[2], a[3]);
    *reinterpret_cast<uint2*>(dst) = w;
  } else {
#pragma unroll
    for (int i = 0; i < N; i += 8) {
      uint4 w;
      w.x = ptx::pack_bf16x2(a[i + 0], a[i + 1]);
      w.y = ptx::pack_bf16x2(a[i + 2], a[i + 3]);
      w.z = ptx::pack_bf16x2(a[i + 4], a[i + 5]);
      w.w = ptx::pack_bf16x2(a[i + 6], a[i + 7]);
      *reinterpret_cast<uint4*>(dst + i) = w;
    }
  }
}

template <typename PT, typename OT, int D>
__global__ void __launch_bounds__(kMergeThreads) lse_merge_kernel(
    const PT* __restrict__ partials, const float* __restrict__ lses, int p, long long rows,
    OT* __restrict__ out, float* __restrict__ lse_out) {
  constexpr int kV = Vec<PT>::kN;
  constexpr int kTpr = D / kV;  // threads per row
  const long long gt = static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x;
  const long long row = gt / kTpr;
  if (row >= rows) return;
  const int col = static_cast<int>(gt % kTpr) * kV;

  float M = -INFINITY;
  for (int c = 0; c < p; ++c) M = fmaxf(M, __ldg(lses + c * rows + row));
  float acc[kV];
#pragma unroll
  for (int i = 0; i < kV; ++i) acc[i] = 0.f;
  float L = -INFINITY;
  if (M != -INFINITY) {
    float sum = 0.f;
    for (int c = 0; c < p; ++c) sum += ptx::ex2_approx((__ldg(lses + c * rows + row) - M) * kLog2e);
    float lg;
    asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(sum));
    L = M + lg * kLn2;
    const PT* base = partials + row * D + col;
    const long long cstride = rows * D;
    for (int c0 = 0; c0 < p; c0 += kBatch) {
      float x[kBatch][kV];
      float w[kBatch];
#pragma unroll
      for (int b = 0; b < kBatch; ++b) {
        if (c0 + b < p) {
          Vec<PT>::load(base + (c0 + b) * cstride, x[b]);
          w[b] = ptx::ex2_approx((__ldg(lses + (c0 + b) * rows + row) - L) * kLog2e);
        }
      }
#pragma unroll
      for (int b = 0; b < kBatch; ++b)
        if (c0 + b < p) {
#pragma unroll
          for (int i = 0; i < kV; ++i) acc[i] = fmaf(w[b], x[b][i], acc[i]);
        }
    }
  }
  store_out(out + row * D + col, acc);
  if (col == 0) lse_out[row] = L;
}

template <typename PT, typename OT, int D>
cudaError_t launch_typed(const MergeLaunch& a, cudaStream_t st) {
  constexpr int kTpr = D / Vec<PT>::kN;
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
