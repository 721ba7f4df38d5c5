// Internal launch interface between the C ABI (ditattn_api.cu) and the
// kernel translation units.  Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>

namespace ditattn {

// Element strides of a logical [B, H, N, D] view: x[b][h][n][d] sits at
// b * b_ + h * h_ + n * n_ + d elements from the base.
struct Strides {
  long long b_, h_, n_;
};

struct AttnLaunch {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;                // contiguous [B, H, N_q]; null: no LSE output (one key range)
  int* status;               // device status word
  int batch;                 // B
  int heads;                 // H
  int n_q;
  int n_kv;
  int d;                     // 64 or 128
  Strides qs, ks, vs, os;    // views of q, k, v (bf16) and out
  float scale;
  bool out_f32;
  // Ring-hop accumulate: out (fp32) and lse hold a running (O, lse) that this pass
  // merges into in place.
  bool accumulate = false;
  // Split-KV: each (head, Q pair) is split over `splits` key ranges whose fp32 partials
  // go to ws_o [splits, B, H, N_q, D] and ws_lse [splits, B, H, N_q]; a merge launch
  // then writes out (contiguous BHND) and lse.  splits == 1: no workspace.
  int splits = 1;
  float* ws_o = nullptr;
  float* ws_lse = nullptr;
  // Batched chunks (virtual ranks): chunk_starts (host, chunks + 1 increasing row offsets
  // into k/v) defines `chunks` key ranges; one launch writes each chunk's partial O to
  // out + c * B*H*N_q*D (contiguous BHND, fp32 or bf16) and its LSE to lse + c * B*H*N_q.
  // No merge.  0 = off.
  int chunks = 0;
  const int* chunk_starts = nullptr;
};

// Encodes the TMA descriptors and launches the attention kernel on `st`.
// Returns cudaErrorInvalidValue if a descriptor cannot be encoded.
cudaError_t launch_attention(const AttnLaunch& a, cudaStream_t st);

struct MergeLaunch {
  const void* partials;  // [p, rows, d]
  const float* lses;     // [p, rows]
  int p;
  long long rows;        // B * H * N
  int d;
  void* out;             // [rows, d]
  float* lse;            // [rows]
  bool part_f32;
  bool out_f32;
};

cudaError_t launch_merge(const MergeLaunch& a, cudaStream_t st);

struct CopyLaunch {
  const void* src;
  void* dst;
  const void* src2 = nullptr;  // optional second pair with the same shape and strides
  void* dst2 = nullptr;
  Strides ss, ds;   // element strides of the two [B, H, N, D] views
  int batch, heads, n, d;
  int elem_bytes;   // 2 (bf16) or 4 (fp32); d * elem_bytes / 16 in {8, 16, 32}
};

// Row-vectorised strided copy between two views (the layout-copy kernel).
cudaError_t launch_layout_copy(const CopyLaunch& a, cudaStream_t st);
// Most rows per (b, h) head one layout-copy launch handles (its grid height limit).
long long layout_copy_max_rows(int d, int elem_bytes);

// Size of the library's fixed device scratch (noalloc.cu) and its address on the current
// device (null on failure).
constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(128) << 20;
void* noalloc_scratch();

// Test-only failure injection behind dit_test_inject_stall.
void set_stall_injection(int enable, long long wait_limit_cycles);

// Test-only cap on the attention kernel's persistent grid (0 = one CTA per SM).
void set_grid_limit(int max_ctas);

}  // namespace ditattn
