// Internal launch interface between the C ABI (ditattn_api.cu) and the
// kernel translation units.  Arguments arrive here already validated.
#pragma once

#include <cuda_runtime.h>

namespace ditattn {

struct AttnLaunch {
  const void* q;
  const void* k;
  const void* v;
  void* out;
  float* lse;
  int* status;               // device status word
  int bh;                    // B * H
  int n_q;
  int n_kv;
  int d;                     // 64 or 128
  long long q_head_stride;   // elements
  long long kv_head_stride;  // elements
  float scale;
  bool out_f32;
  // Ring-hop accumulate: out (fp32) and lse hold a running (O, lse) that this pass
  // merges into in place.
  bool accumulate = false;
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

// Test-only failure injection behind dit_test_inject_stall.
void set_stall_injection(int enable, long long wait_limit_cycles);

// Test-only cap on the attention kernel's persistent grid (0 = one CTA per SM).
void set_grid_limit(int max_ctas);

}  // namespace ditattn
