// Per-row arithmetic of the exact log-sum-exp merge of p KV-chunk partials,
//   M = max_c lse_c,  lse = M + ln sum_c exp(lse_c - M),  O = sum_c exp(lse_c - lse) O_c
// (arganzheng.life multi-GPU diffusion parallelism, section 4.2 Ring: the per-round
// blocks are combined by online softmax accumulation), for the merge kernel (lse_merge.cu).
//
// A thread owns one 16-byte vector of one row (4 fp32 or 8 bf16 partial elements).
// Chunks are absorbed in batches of up to 8: the caller issues all loads of a batch
// (LSEs and partial vectors) before any arithmetic; the batches are combined online
// (running max M, running sum S of exp(lse_c - M), running weighted sum acc).
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace ditattn {
namespace merge {

constexpr int kBatch = 8;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

template <typename T> struct Vec;
template <> struct Vec<float> {
  static constexpr int kN = 4;
  using Raw = uint4;
  // Streaming load: a merge reads each partial once.
  __device__ static Raw load(const float* p) { return __ldcs(reinterpret_cast<const uint4*>(p)); }
  __device__ static void widen(const Raw& v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x);
    x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z);
    x[3] = __uint_as_float(v.w);
  }
};
template <> struct Vec<__nv_bfloat16> {
  static constexpr int kN = 8;
  using Raw = uint4;
  __device__ static Raw load(const __nv_bfloat16* p) {
    return Vec<float>::load(reinterpret_cast<const float*>(p));
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

__device__ __forceinline__ float load_lse(const float* p) { return __ldg(p); }

// Running state of one thread's vector of one row.
template <typename PT>
struct RowMerge {
  static constexpr int kV = Vec<PT>::kN;
  float M = -INFINITY;  // running max of the LSEs seen so far
  float S = 0.f;        // running sum of exp(lse_c - M)
  float acc[kV];        // running sum of exp(lse_c - M) * O_c

  __device__ __forceinline__ RowMerge() {
#pragma unroll
    for (int i = 0; i < kV; ++i) acc[i] = 0.f;
  }

  // Absorbs the chunks c0 .. c0 + kBatch - 1 (those below p) of one row: chunk c's vector
  // sits at part_row + c * cstride and its LSE at lse_row + c * lstride.  The two addresses
  // advance chunk by chunk, so few registers are live while the batch's loads are in flight.
  __device__ __forceinline__ void absorb(const PT* part_row, long long cstride,
                                         const float* lse_row, long long lstride, int c0, int p) {
    typename Vec<PT>::Raw raw[kBatch];
    float lv[kBatch];
    const PT* pp = part_row + c0 * cstride;
    const float* pl = lse_row + c0 * lstride;
#pragma unroll
    for (int b = 0; b < kBatch; ++b) {
      if (c0 + b < p) {
        lv[b] = load_lse(pl);
        raw[b] = Vec<PT>::load(pp);
      } else {
        lv[b] = -INFINITY;
      }
      pp += cstride;
      pl += lstride;
    }
    float mb = lv[0];
#pragma unroll
    for (int b = 1; b < kBatch; ++b) mb = fmaxf(mb, lv[b]);
    const float Mn = fmaxf(M, mb);
    if (Mn == -INFINITY) return;  // nothing but empty chunks so far
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

  // Normalises acc in place into the merged output vector and returns the merged LSE
  // (-inf, with acc = 0, when every chunk was empty).
  __device__ __forceinline__ float finish() {
    float L = -INFINITY;
    if (M != -INFINITY) {
      const float inv = 1.f / S;
#pragma unroll
      for (int i = 0; i < kV; ++i) acc[i] *= inv;
      float lg;
      asm("lg2.approx.f32 %0, %1;" : "=f"(lg) : "f"(S));
      L = M + lg * kLn2;
    }
    return L;
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

// Merges row `row` (of `rows`) for the thread's vector at column `col`: out[row][col..],
// and lse_out[row] from the thread at column 0.  Partial block c starts c * rows * D
// elements after `part`, its LSEs c * rows after `lses`.
template <typename PT, typename OT, int D>
__device__ __forceinline__ void merge_row(const PT* part, const float* lses, int p, long long rows,
                                          long long row, int col, OT* out, float* lse_out) {
  RowMerge<PT> m;
  const PT* part_row = part + row * D + col;
  const float* lse_row = lses + row;
  for (int c0 = 0; c0 < p; c0 += kBatch)
    m.absorb(part_row, rows * D, lse_row, rows, c0, p);
  const float L = m.finish();
  store_out(out + row * D + col, m.acc);
  if (col == 0) lse_out[row] = L;
}

}  // namespace merge
}  // namespace ditattn
