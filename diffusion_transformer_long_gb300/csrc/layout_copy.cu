// Strided copy of a logical [B, H, N, D] tensor between two views whose last
// dimension is contiguous.  This is the local, on-GPU half of the sequence <->
// head re-shard that Ulysses sequence parallelism wraps around attention
// (arganzheng.life multi-GPU diffusion parallelism, section 4.1 Ulysses: an
// all-to-all turns a token shard of all heads into all tokens of a head shard;
// valdrada.cn Wan2.2, CP section): the token-major (BSND) <-> head-major (BHND)
// transpose and the packing of per-rank send buffers are all such copies.  The
// same copy writes fresh K/V rows into a KV buffer in place.
//
// HBM-bound: every row is D*esize contiguous bytes (128-512 B) on both sides,
// moved as 16-byte vectors by consecutive threads, so each warp access covers
// whole 128-byte lines whatever the strides between rows.  A block owns one
// (b, h) head and a run of rows; all eight loads of a thread are issued before
// its stores (streaming cache hints: the data is touched once).  One launch may move two
// tensors of the same shape and strides (K and V of a KV-buffer update).
#include <cuda_runtime.h>

#include <cstdint>

#include "launch.h"

namespace ditattn {
namespace {

constexpr int kCopyThreads = 256;
constexpr int kCopyUnroll = 8;  // 16-byte vectors in flight per thread (4: 5.6 TB/s, 8: 6.2 TB/s)

struct CopyParams {
  const char* src[2];  // blockIdx.z picks the pair (one or two tensors per launch)
  char* dst[2];
  long long ss_b, ss_h, ss_n;  // source strides (bytes)
  long long ds_b, ds_h, ds_n;  // destination strides (bytes)
  int heads;
  int n;
};

// kVpr: 16-byte vectors per row (D * element size / 16).
template <int kVpr>
__global__ void __launch_bounds__(kCopyThreads) layout_copy_kernel(const CopyParams p) {
  constexpr int kRowsPerPass = kCopyThreads / kVpr;
  const int bh = blockIdx.x;
  const int b = bh / p.heads, h = bh - b * p.heads;
  const char* src = p.src[blockIdx.z] + b * p.ss_b + h * p.ss_h;
  char* dst = p.dst[blockIdx.z] + b * p.ds_b + h * p.ds_h;
  const int sub = threadIdx.x / kVpr;
  const int vec = threadIdx.x % kVpr;
  const int n0 = blockIdx.y * (kRowsPerPass * kCopyUnroll) + sub;
  uint4 v[kCopyUnroll];
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int row = n0 + u * kRowsPerPass;
    if (row < p.n)
      v[u] = __ldcs(reinterpret_cast<const uint4*>(src + row * p.ss_n) + vec);
  }
#pragma unroll
  for (int u = 0; u < kCopyUnroll; ++u) {
    const int row = n0 + u * kRowsPerPass;
    if (row < p.n) __stcs(reinterpret_cast<uint4*>(dst + row * p.ds_n) + vec, v[u]);
  }
}

template <int kVpr>
cudaError_t launch_copy(const CopyParams& p, int bh, int pairs, cudaStream_t st) {
  constexpr int kRowsPerBlock = (kCopyThreads / kVpr) * kCopyUnroll;
  const dim3 grid(static_cast<unsigned>(bh), static_cast<unsigned>((p.n + kRowsPerBlock - 1) / kRowsPerBlock),
                  static_cast<unsigned>(pairs));
  layout_copy_kernel<kVpr><<<grid, kCopyThreads, 0, st>>>(p);
  return cudaGetLastError();
}

}  // namespace

long long layout_copy_max_rows(int d, int elem_bytes) {
  const int vpr = d * elem_bytes / 16;
  if (vpr < 1 || kCopyThreads % vpr) return 0;
  return 65535LL * (kCopyThreads / vpr) * kCopyUnroll;  // grid y limit x rows per block
}

cudaError_t launch_layout_copy(const CopyLaunch& a, cudaStream_t st) {
  CopyParams p;
  const int pairs = a.src2 ? 2 : 1;
  p.src[0] = static_cast<const char*>(a.src);
  p.dst[0] = static_cast<char*>(a.dst);
  p.src[1] = static_cast<const char*>(a.src2 ? a.src2 : a.src);
  p.dst[1] = static_cast<char*>(a.src2 ? a.dst2 : a.dst);
  const long long e = a.elem_bytes;
  p.ss_b = a.ss.b_ * e;
  p.ss_h = a.ss.h_ * e;
  p.ss_n = a.ss.n_ * e;
  p.ds_b = a.ds.b_ * e;
  p.ds_h = a.ds.h_ * e;
  p.ds_n = a.ds.n_ * e;
  p.heads = a.heads;
  p.n = a.n;
  const int bh = a.batch * a.heads;
  switch (a.d * a.elem_bytes / 16) {
    case 8: return launch_copy<8>(p, bh, pairs, st);
    case 16: return launch_copy<16>(p, bh, pairs, st);
    case 32: return launch_copy<32>(p, bh, pairs, st);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace ditattn
