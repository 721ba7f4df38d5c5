// C ABI of the library (declared in include/ditattn.h): argument validation,
// the device status word, and dispatch to the kernel launchers.  Validation
// runs before any CUDA call, so a rejected call touches no device.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/ditattn.h"
#include "launch.h"

namespace {

// Set by kernels whose bounded waits expired; read and cleared by dit_attn_check.
__device__ int g_status_word;

constexpr int kMaxDevices = 64;

int* status_ptr() {
  static std::mutex mu;
  static int* cached[kMaxDevices] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(mu);
  if (!cached[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_status_word) != cudaSuccess) return nullptr;
    cached[dev] = static_cast<int*>(p);
  }
  return cached[dev];
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
  uintptr_t lo, hi;  // [lo, hi)
};
Range span(const void* p, long long bytes) {
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + static_cast<uintptr_t>(bytes)};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

bool valid_dtype(dit_dtype t) { return t == DIT_F32 || t == DIT_BF16; }
int dtype_bytes(dit_dtype t) { return t == DIT_F32 ? 4 : 2; }

dit_status check_dims(long long B, long long H, long long N, int D) {
  if (B < 1 || H < 1 || N < 1 || D < 1) return DIT_ERR_INVALID_ARG;
  if (B * H > INT_MAX || N > INT_MAX) return DIT_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return DIT_ERR_UNSUPPORTED;
  return DIT_OK;
}

dit_status validate_attention(const void* q, const void* k, const void* v, const void* out,
                              const float* lse, int B, int H, int N_q, int n_kv, int D,
                              long long kv_head_stride, float scale, dit_dtype out_dtype) {
  dit_status s = check_dims(B, H, N_q, D);
  if (s != DIT_OK) return s;
  if (n_kv < 1) return DIT_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || !lse) return DIT_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) ||
      !aligned(lse, 4))
    return DIT_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return DIT_ERR_INVALID_ARG;
  if (!valid_dtype(out_dtype)) return DIT_ERR_INVALID_ARG;
  if (kv_head_stride < static_cast<long long>(n_kv) * D || kv_head_stride % 8 != 0 ||
      kv_head_stride >= (1LL << 39))
    return DIT_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  const long long q_pairs = (static_cast<long long>(N_q) + 255) / 256;
  if (q_pairs * bh > INT_MAX) return DIT_ERR_INVALID_ARG;
  const long long qkv_rows = bh * N_q;
  const Range rq = span(q, qkv_rows * D * 2);
  const long long kv_bytes = ((bh - 1) * kv_head_stride + static_cast<long long>(n_kv) * D) * 2;
  const Range rk = span(k, kv_bytes), rv = span(v, kv_bytes);
  const Range ro = span(out, qkv_rows * D * dtype_bytes(out_dtype));
  const Range rl = span(lse, qkv_rows * 4);
  for (Range in : {rq, rk, rv})
    if (overlap(ro, in) || overlap(rl, in)) return DIT_ERR_INVALID_ARG;
  if (overlap(ro, rl)) return DIT_ERR_INVALID_ARG;
  return DIT_OK;
}

dit_status run_attention(const void* q, const void* k, const void* v, void* out, float* lse,
                         int B, int H, int N_q, int n_kv, int D, long long kv_head_stride,
                         float scale, dit_dtype out_dtype, dit_stream stream,
                         bool accumulate = false) {
  int* status = status_ptr();
  if (!status) return DIT_ERR_CUDA;
  ditattn::AttnLaunch a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.status = status;
  a.bh = B * H;
  a.n_q = N_q;
  a.n_kv = n_kv;
  a.d = D;
  a.q_head_stride = static_cast<long long>(N_q) * D;
  a.kv_head_stride = kv_head_stride;
  a.scale = scale;
  a.out_f32 = out_dtype == DIT_F32;
  a.accumulate = accumulate;
  return ditattn::launch_attention(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DIT_OK
             : DIT_ERR_CUDA;
}

}  // namespace

extern "C" {

dit_status dit_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                        int H, int N, int D, float scale, dit_dtype out_dtype, dit_stream stream) {
  const long long hs = static_cast<long long>(N) * D;
  dit_status s = validate_attention(q, k, v, out, lse, B, H, N, N, D, hs, scale, out_dtype);
  if (s != DIT_OK) return s;
  return run_attention(q, k, v, out, lse, B, H, N, N, D, hs, scale, out_dtype, stream);
}

dit_status dit_attn_chunk_fwd(const void* q, const void* k, const void* v, void* out_partial,
                              float* lse_partial, int B, int H, int N_q, int n_kv, int D,
                              long long kv_head_stride, float scale, dit_dtype partial_dtype,
                              dit_stream stream) {
  dit_status s = validate_attention(q, k, v, out_partial, lse_partial, B, H, N_q, n_kv, D,
                                    kv_head_stride, scale, partial_dtype);
  if (s != DIT_OK) return s;
  return run_attention(q, k, v, out_partial, lse_partial, B, H, N_q, n_kv, D, kv_head_stride,
                       scale, partial_dtype, stream);
}

dit_status dit_attn_chunk_fwd_accumulate(const void* q, const void* k, const void* v, float* o_run,
                                         float* lse_run, int B, int H, int N_q, int n_kv, int D,
                                         long long kv_head_stride, float scale, dit_stream stream) {
  dit_status s = validate_attention(q, k, v, o_run, lse_run, B, H, N_q, n_kv, D, kv_head_stride,
                                    scale, DIT_F32);
  if (s != DIT_OK) return s;
  return run_attention(q, k, v, o_run, lse_run, B, H, N_q, n_kv, D, kv_head_stride, scale, DIT_F32,
                       stream, /*accumulate=*/true);
}

dit_status dit_attn_lse_merge(const void* partials, const float* lses, int p, void* out,
                              float* lse, int B, int H, int N, int D, dit_dtype partial_dtype,
                              dit_dtype out_dtype, dit_stream stream) {
  dit_status s = check_dims(B, H, N, D);
  if (s != DIT_OK) return s;
  if (p < 1) return DIT_ERR_INVALID_ARG;
  if (!partials || !lses || !out || !lse) return DIT_ERR_INVALID_ARG;
  if (!valid_dtype(partial_dtype) || !valid_dtype(out_dtype)) return DIT_ERR_INVALID_ARG;
  if (!aligned(partials, 16) || !aligned(out, 16) || !aligned(lses, 4) || !aligned(lse, 4))
    return DIT_ERR_INVALID_ARG;
  const long long rows = static_cast<long long>(B) * H * N;
  const Range rp = span(partials, p * rows * D * dtype_bytes(partial_dtype));
  const Range rl = span(lses, p * rows * 4);
  const Range ro = span(out, rows * D * dtype_bytes(out_dtype));
  const Range rs = span(lse, rows * 4);
  if (overlap(ro, rp) || overlap(ro, rl) || overlap(rs, rp) || overlap(rs, rl) || overlap(ro, rs))
    return DIT_ERR_INVALID_ARG;
  ditattn::MergeLaunch a;
  a.partials = partials;
  a.lses = lses;
  a.p = p;
  a.rows = rows;
  a.d = D;
  a.out = out;
  a.lse = lse;
  a.part_f32 = partial_dtype == DIT_F32;
  a.out_f32 = out_dtype == DIT_F32;
  return ditattn::launch_merge(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DIT_OK
             : DIT_ERR_CUDA;
}

dit_status dit_attn_check(dit_stream stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) return DIT_ERR_CUDA;
  int v = 0;
  if (cudaMemcpyFromSymbol(&v, g_status_word, sizeof v) != cudaSuccess) return DIT_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpyToSymbol(g_status_word, &zero, sizeof zero) != cudaSuccess) return DIT_ERR_CUDA;
    return DIT_ERR_TIMEOUT;
  }
  return DIT_OK;
}

void dit_test_inject_stall(int enable, long long wait_limit_cycles) {
  ditattn::set_stall_injection(enable, wait_limit_cycles);
}

void dit_test_set_grid_limit(int max_ctas) { ditattn::set_grid_limit(max_ctas); }

const char* dit_status_string(dit_status s) {
  switch (s) {
    case DIT_OK: return "ok";
    case DIT_ERR_INVALID_ARG: return "invalid argument";
    case DIT_ERR_UNSUPPORTED: return "unsupported configuration";
    case DIT_ERR_CUDA: return "CUDA error";
    case DIT_ERR_TIMEOUT: return "device wait timed out";
  }
  return "unknown status";
}

int dit_version(void) { return 100; }

}  // extern "C"
