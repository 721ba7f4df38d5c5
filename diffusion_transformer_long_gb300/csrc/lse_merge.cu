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
// streaming loads.  Chunks are taken in batches of up to 8: all loads of a
// batch (LSEs and partial vectors) are issued before any arithmetic, and the
// batches are combined online (running max M, running sum S of exp(lse_c - M),
// running weighted sum A), then O = A / S and lse = M + ln S.
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
  using Raw = float4;
  __device__ static Raw load(const float* p) { return __ldcs(reinterpret_cast<const float4*>(p)); }
  __device__ static void widen(const Raw& v, float (&x)[4]) {
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  using Raw = uint4;
  __device__ static Raw load(const __nv_bfloat16* p) {
    return __ldcs(reinterpret_cast<const uint4*>(p));
  }
  __device__ static void widen(const Raw& v, float (&x)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = ptx::bf16lo(w[i]);
      x[2 * i + 1] = ptx::bf16hi(w[i]);
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
__global__ void __launch_bounds__(kMergeThreads, 4) lse_merge_kernel(
    const PT* __restrict__ partials, const float* __restrict__ lses, int p, long long rows,
    OT* __restrict__ out, float* __restrict__ lse_out) {
  constexpr int kV = Vec<PT>::kN;
  constexpr int kTpr = D / kV;  // threads per row
  const long long gt = static_cast<long long>(blockIdx.x) * kMergeThreads + threadIdx.x;
  const long long row = gt / kTpr;
  if (row >= rows) return;
  const int col = static_cast<int>(gt % kTpr) * kV;
  const PT* base = partials + row * D + col;
  const long long cstride = rows * D;

  float M = -INFINITY;  // running max of the LSEs seen so far
  float S = 0.f;        // running sum of exp(lse_c - M)
  float acc[kV];        // running sum of exp(lse_c - M) * O_c
#pragma unroll
  for (int i = 0; i < kV; ++i) acc[i] = 0.f;

  for (int c0 = 0; c0 < p; c0 += kBatch) {
    typename Vec<PT>::Raw raw[kBatch];
    float lv[kBatch];
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (c0 + b < p) {
        lv[b] = __ldg(lses + (c0 + b) * rows + row);
        raw[b] = Vec<PT>::load(base + (c0 + b) * cstride);
      } else {
        lv[b] = -INFINITY;
      }
    }
    float mb = lv[0];
#pragma unroll
    for (int b = 1; b < kBatch; ++b) mb = fmaxf(mb, lv[b]);
    const float Mn = fmaxf(M, mb);
    if (Mn == -INFINITY) continue;  // nothing but empty chunks so far
    const float r = ptx::ex2_approx((M - Mn) * kLog2e);  // 0 while M = -inf
    S *= r;
#pragma unroll
    for (int i = 0; i < kV; ++i) acc[i] *= r;
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (c0 + b < p) {
        const float w = ptx::ex2_approx((lv[b] - Mn) * kLog2e);  // 0 for an empty chunk
        float x[kV];
        Vec<PT>::widen(raw[b], x);
        S += w;
#pragma unroll
        for (int i = 0; i < kV; ++i) acc[i] = fmaf(w, x[i], acc[i]);
      }
    }
    M = Mn;
  }
  float L = -INFINITY;
  if (M != -INFINITY) {
    const float inv = 1.f / S;
#pragma unroll
    for (int i = 0; i < kV; ++i) acc[i] *= inv;
    float lg;
    asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(S));
    L = M + lg * kLn2;
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
