// C ABI of the library (declared in include/ditattn.h): argument validation,
// the device status word, and dispatch to the kernel launchers.  Validation
// runs before any CUDA call, so a rejected call touches no device.
#include <cuda_runtime.h>

#include <climits>
#include <cmath>
#include <algorithm>
#include <cstdint>
#include <mutex>
#include <initializer_list>
#include <utility>

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
                              long long kv_head_stride, float scale, dit_dtype out_dtype,
                              bool lse_optional = false) {
  dit_status s = check_dims(B, H, N_q, D);
  if (s != DIT_OK) return s;
  if (n_kv < 1) return DIT_ERR_INVALID_ARG;
  if (!q || !k || !v || !out || (!lse && !lse_optional)) return DIT_ERR_INVALID_ARG;
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
  const Range rl = span(lse, lse ? qkv_rows * 4 : 0);
  for (Range in : {rq, rk, rv})
    if (overlap(ro, in) || overlap(rl, in)) return DIT_ERR_INVALID_ARG;
  if (overlap(ro, rl)) return DIT_ERR_INVALID_ARG;
  return DIT_OK;
}

// Bytes spanned by a strided [B, H, N, D] view (from its base to one past its last element).
long long view_span(const dit_strides& s, long long B, long long H, long long N, long long D,
                    int esize) {
  return ((B - 1) * s.b + (H - 1) * s.h + (N - 1) * s.n + D) * esize;
}

dit_strides contiguous(long long H, long long N, long long D) { return {H * N * D, N * D, D}; }

// Split-KV workspace: fp32 partial O [splits, rows, D], then (256-byte aligned) fp32 partial
// LSEs [splits, rows].
long long splitkv_lse_offset(long long rows, long long D, long long splits) {
  return (splits * rows * D * 4 + 255) / 256 * 256;
}
long long splitkv_bytes(long long rows, long long D, long long splits) {
  return splitkv_lse_offset(rows, D, splits) + splits * rows * 4;
}

// A strided view usable by the kernels: strides positive multiples of 8 elements (16-byte
// TMA strides) below 2^39, and the view must fit 64-bit byte offsets comfortably.
bool valid_strides(const dit_strides& s) {
  for (long long x : {s.b, s.h, s.n})
    if (x < 8 || x % 8 != 0 || x >= (1LL << 39)) return false;
  return true;
}

// True if no two elements of the view share an address: sorted by stride, every stride
// must clear the span of the dimensions below it.
bool no_self_overlap(const dit_strides& s, long long B, long long H, long long N, long long D) {
  struct Dim {
    long long stride, extent;
  } d[3] = {{s.n, N}, {s.h, H}, {s.b, B}};
  for (int i = 0; i < 3; ++i)  // sort by stride
    for (int j = i + 1; j < 3; ++j)
      if (d[j].stride < d[i].stride) std::swap(d[i], d[j]);
  long long span = D;
  for (const Dim& x : d) {
    if (x.extent <= 1) continue;
    if (x.stride < span) return false;
    span = x.stride * (x.extent - 1) + span;
  }
  return true;
}

dit_status run_attention(const void* q, const dit_strides& qs, const void* k, const dit_strides& ks,
                         const void* v, const dit_strides& vs, void* out, const dit_strides& os,
                         float* lse, int B, int H, int N_q, int n_kv, int D, float scale,
                         dit_dtype out_dtype, dit_stream stream, bool accumulate = false,
                         int splits = 1, void* workspace = nullptr, int chunks = 0,
                         const int* chunk_starts = nullptr) {
  int* status = status_ptr();
  if (!status) return DIT_ERR_CUDA;
  ditattn::AttnLaunch a;
  a.q = q;
  a.k = k;
  a.v = v;
  a.out = out;
  a.lse = lse;
  a.status = status;
  a.batch = B;
  a.heads = H;
  a.n_q = N_q;
  a.n_kv = n_kv;
  a.d = D;
  a.qs = {qs.b, qs.h, qs.n};
  a.ks = {ks.b, ks.h, ks.n};
  a.vs = {vs.b, vs.h, vs.n};
  a.os = {os.b, os.h, os.n};
  a.scale = scale;
  a.out_f32 = out_dtype == DIT_F32;
  a.accumulate = accumulate;
  a.splits = splits;
  a.chunks = chunks;
  a.chunk_starts = chunk_starts;
  if (splits > 1) {
    const long long rows = static_cast<long long>(B) * H * N_q;
    a.ws_o = static_cast<float*>(workspace);
    a.ws_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) + splitkv_lse_offset(rows, D, splits));
  }
  return ditattn::launch_attention(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DIT_OK
             : DIT_ERR_CUDA;
}

// Contiguous q/out, K/V heads kv_head_stride elements apart (the chunk form).
dit_status run_contiguous(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                          int H, int N_q, int n_kv, int D, long long kv_head_stride, float scale,
                          dit_dtype out_dtype, dit_stream stream, bool accumulate = false,
                          int splits = 1, void* workspace = nullptr, int chunks = 0,
                          const int* chunk_starts = nullptr) {
  const dit_strides qs = contiguous(H, N_q, D);
  const dit_strides kvs = {H * kv_head_stride, kv_head_stride, D};
  return run_attention(q, qs, k, kvs, v, kvs, out, qs, lse, B, H, N_q, n_kv, D, scale, out_dtype,
                       stream, accumulate, splits, workspace, chunks, chunk_starts);
}

// Split-KV arguments: 1 <= splits <= min(64, KV tiles); with splits > 1 a 256-byte-aligned
// workspace of at least dit_attn_splitkv_workspace_bytes that overlaps none of `others`.
dit_status validate_splits(int splits, int n_kv, const void* workspace, size_t workspace_bytes,
                           int B, int H, int N_q, int D, std::initializer_list<Range> others) {
  const int tiles = (n_kv + 127) / 128;
  if (splits < 1 || splits > 64 || splits > tiles) return DIT_ERR_INVALID_ARG;
  if (splits == 1) return DIT_OK;
  const long long rows = static_cast<long long>(B) * H * N_q;
  const long long need = splitkv_bytes(rows, D, splits);
  if (!workspace || !aligned(workspace, 256) || static_cast<long long>(workspace_bytes) < need)
    return DIT_ERR_INVALID_ARG;
  const Range rw = span(workspace, need);
  for (Range o : others)
    if (overlap(rw, o)) return DIT_ERR_INVALID_ARG;
  return DIT_OK;
}

// Chunk arguments (all virtual ranks in one launch): the attention arguments for the
// partial blocks, 1 <= p <= 64 increasing chunk starts within [0, n_kv], and p partial blocks
// and LSE rows clear of the inputs and of each other.
dit_status validate_chunks(const void* q, const void* k, const void* v, void* partials,
                           float* lses, int B, int H, int N_q, int n_kv, int D,
                           long long kv_head_stride, int p, const int* chunk_starts, float scale,
                           dit_dtype partial_dtype) {
  dit_status s = validate_attention(q, k, v, partials, lses, B, H, N_q, n_kv, D, kv_head_stride,
                                    scale, partial_dtype);
  if (s != DIT_OK) return s;
  if (p < 1 || p > 64 || !chunk_starts) return DIT_ERR_INVALID_ARG;
  if (chunk_starts[0] < 0 || chunk_starts[p] > n_kv) return DIT_ERR_INVALID_ARG;
  for (int c = 0; c < p; ++c)
    if (chunk_starts[c + 1] <= chunk_starts[c]) return DIT_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (((static_cast<long long>(N_q) + 255) / 256) * bh * p > INT_MAX) return DIT_ERR_INVALID_ARG;
  const long long rows = bh * N_q;
  const Range rp = span(partials, p * rows * D * dtype_bytes(partial_dtype));
  const Range rl = span(lses, p * rows * 4);
  const long long kv_bytes = ((bh - 1) * kv_head_stride + static_cast<long long>(n_kv) * D) * 2;
  for (Range in : {span(q, rows * D * 2), span(k, kv_bytes), span(v, kv_bytes)})
    if (overlap(rp, in) || overlap(rl, in)) return DIT_ERR_INVALID_ARG;
  if (overlap(rp, rl)) return DIT_ERR_INVALID_ARG;
  return DIT_OK;
}

}  // namespace

extern "C" {

dit_status dit_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse, int B,
                        int H, int N, int D, float scale, dit_dtype out_dtype, dit_stream stream) {
  const long long hs = static_cast<long long>(N) * D;
  dit_status s = validate_attention(q, k, v, out, lse, B, H, N, N, D, hs, scale, out_dtype,
                                    /*lse_optional=*/true);
  if (s != DIT_OK) return s;
  return run_contiguous(q, k, v, out, lse, B, H, N, N, D, hs, scale, out_dtype, stream);
}

dit_status dit_attn_chunk_fwd(const void* q, const void* k, const void* v, void* out_partial,
                              float* lse_partial, int B, int H, int N_q, int n_kv, int D,
                              long long kv_head_stride, float scale, dit_dtype partial_dtype,
                              dit_stream stream) {
  dit_status s = validate_attention(q, k, v, out_partial, lse_partial, B, H, N_q, n_kv, D,
                                    kv_head_stride, scale, partial_dtype);
  if (s != DIT_OK) return s;
  return run_contiguous(q, k, v, out_partial, lse_partial, B, H, N_q, n_kv, D, kv_head_stride,
                        scale, partial_dtype, stream);
}

dit_status dit_attn_chunks_fwd(const void* q, const void* k, const void* v, void* partials,
                               float* lses, int B, int H, int N_q, int n_kv, int D,
                               long long kv_head_stride, int p, const int* chunk_starts,
                               float scale, dit_dtype partial_dtype, dit_stream stream) {
  dit_status s = validate_chunks(q, k, v, partials, lses, B, H, N_q, n_kv, D, kv_head_stride, p,
                                 chunk_starts, scale, partial_dtype);
  if (s != DIT_OK) return s;
  return run_contiguous(q, k, v, partials, lses, B, H, N_q, n_kv, D, kv_head_stride, scale,
                        partial_dtype, stream, false, 1, nullptr, p, chunk_starts);
}

dit_status dit_attn_chunk_fwd_accumulate(const void* q, const void* k, const void* v, float* o_run,
                                         float* lse_run, int B, int H, int N_q, int n_kv, int D,
                                         long long kv_head_stride, float scale, dit_stream stream) {
  dit_status s = validate_attention(q, k, v, o_run, lse_run, B, H, N_q, n_kv, D, kv_head_stride,
                                    scale, DIT_F32);
  if (s != DIT_OK) return s;
  return run_contiguous(q, k, v, o_run, lse_run, B, H, N_q, n_kv, D, kv_head_stride, scale, DIT_F32,
                        stream, /*accumulate=*/true);
}

dit_status dit_attn_fwd_strided(const void* q, const dit_strides* q_strides, const void* k,
                                const dit_strides* k_strides, const void* v,
                                const dit_strides* v_strides, void* out,
                                const dit_strides* out_strides, float* lse, int B, int H, int N_q,
                                int n_kv, int D, float scale, dit_dtype out_dtype,
                                dit_stream stream) {
  dit_status s = check_dims(B, H, N_q, D);
  if (s != DIT_OK) return s;
  if (n_kv < 1 || n_kv > INT_MAX) return DIT_ERR_INVALID_ARG;
  if (!q || !k || !v || !out) return DIT_ERR_INVALID_ARG;  // lse may be NULL
  if (!valid_dtype(out_dtype)) return DIT_ERR_INVALID_ARG;
  if (!(scale > 0.f) || !std::isfinite(scale)) return DIT_ERR_INVALID_ARG;
  // The stride of a size-1 dimension addresses nothing: any valid value will do.
  auto norm = [&](const dit_strides* p, long long n_rows) {
    dit_strides x = p ? *p : contiguous(H, n_rows, D);
    if (B == 1) x.b = D;
    if (H == 1) x.h = D;
    if (n_rows == 1) x.n = D;
    return x;
  };
  const dit_strides qs = norm(q_strides, N_q), ks = norm(k_strides, n_kv),
                    vs = norm(v_strides, n_kv), os = norm(out_strides, N_q);
  for (const dit_strides* x : {&qs, &ks, &vs, &os})
    if (!valid_strides(*x)) return DIT_ERR_INVALID_ARG;
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(out, 16) || !aligned(lse, 4))
    return DIT_ERR_INVALID_ARG;
  const long long bh = static_cast<long long>(B) * H;
  if (((static_cast<long long>(N_q) + 255) / 256) * bh > INT_MAX) return DIT_ERR_INVALID_ARG;
  const int oes = dtype_bytes(out_dtype);
  if (!no_self_overlap(os, B, H, N_q, D)) return DIT_ERR_INVALID_ARG;
  const Range rq = span(q, view_span(qs, B, H, N_q, D, 2));
  const Range rk = span(k, view_span(ks, B, H, n_kv, D, 2));
  const Range rv = span(v, view_span(vs, B, H, n_kv, D, 2));
  const Range ro = span(out, view_span(os, B, H, N_q, D, oes));
  const Range rl = span(lse, lse ? bh * N_q * 4 : 0);
  for (Range in : {rq, rk, rv})
    if (overlap(ro, in) || overlap(rl, in)) return DIT_ERR_INVALID_ARG;
  if (overlap(ro, rl)) return DIT_ERR_INVALID_ARG;
  return run_attention(q, qs, k, ks, v, vs, out, os, lse, B, H, N_q, n_kv, D, scale, out_dtype,
                       stream);
}

dit_status dit_layout_copy(const void* src, const dit_strides* src_strides, void* dst,
                           const dit_strides* dst_strides, int B, int H, int N, int D,
                           dit_dtype dtype, dit_stream stream) {
  dit_status s = check_dims(B, H, N, D);
  if (s != DIT_OK) return s;
  if (!src || !dst || !valid_dtype(dtype)) return DIT_ERR_INVALID_ARG;
  if (!aligned(src, 16) || !aligned(dst, 16)) return DIT_ERR_INVALID_ARG;
  const int es = dtype_bytes(dtype);
  auto norm = [&](const dit_strides* p) {
    dit_strides x = p ? *p : contiguous(H, N, D);
    if (B == 1) x.b = D;
    if (H == 1) x.h = D;
    if (N == 1) x.n = D;
    return x;
  };
  const dit_strides ss = norm(src_strides), ds = norm(dst_strides);
  if (!valid_strides(ss) || !valid_strides(ds)) return DIT_ERR_INVALID_ARG;
  if (!no_self_overlap(ds, B, H, N, D)) return DIT_ERR_INVALID_ARG;
  if (overlap(span(src, view_span(ss, B, H, N, D, es)), span(dst, view_span(ds, B, H, N, D, es))))
    return DIT_ERR_INVALID_ARG;
  if (N > ditattn::layout_copy_max_rows(D, es)) return DIT_ERR_UNSUPPORTED;
  ditattn::CopyLaunch a;
  a.src = src;
  a.dst = dst;
  a.ss = {ss.b, ss.h, ss.n};
  a.ds = {ds.b, ds.h, ds.n};
  a.batch = B;
  a.heads = H;
  a.n = N;
  a.d = D;
  a.elem_bytes = es;
  return ditattn::launch_layout_copy(a, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? DIT_OK
             : DIT_ERR_CUDA;
}

dit_status dit_attn_stale_kv_fwd(const void* q, const void* k_new, const void* v_new, void* k_buf,
                                 void* v_buf, void* out, float* lse, int B, int H, int m, int N,
                                 int D, int row0, float scale, dit_dtype out_dtype, int splits,
                                 void* workspace, size_t workspace_bytes, dit_stream stream) {
  dit_status s = check_dims(B, H, N, D);
  if (s != DIT_OK) return s;
  if (m < 1 || row0 < 0 || row0 > N - m) return DIT_ERR_INVALID_ARG;
  if (!k_new || !v_new || !k_buf || !v_buf) return DIT_ERR_INVALID_ARG;
  if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_buf, 16) || !aligned(v_buf, 16))
    return DIT_ERR_INVALID_ARG;
  // Attention arguments: m patch queries against the N rows of the (updated) buffer.
  const long long hs = static_cast<long long>(N) * D;
  s = validate_attention(q, k_buf, v_buf, out, lse, B, H, m, N, D, hs, scale, out_dtype);
  if (s != DIT_OK) return s;
  const long long bh = static_cast<long long>(B) * H;
  const Range rkb = span(k_buf, bh * hs * 2), rvb = span(v_buf, bh * hs * 2);
  const Range rkn = span(k_new, bh * m * D * 2), rvn = span(v_new, bh * m * D * 2);
  const Range rq = span(q, bh * m * D * 2);
  if (overlap(rkb, rvb)) return DIT_ERR_INVALID_ARG;
  const Range ro = span(out, bh * m * D * dtype_bytes(out_dtype)), rl = span(lse, bh * m * 4);
  for (Range buf : {rkb, rvb})
    for (Range other : {rkn, rvn, rq})
      if (overlap(buf, other)) return DIT_ERR_INVALID_ARG;
  for (Range fresh : {rkn, rvn})
    if (overlap(fresh, ro) || overlap(fresh, rl)) return DIT_ERR_INVALID_ARG;
  s = validate_splits(splits, N, workspace, workspace_bytes, B, H, m, D,
                      {rq, rkn, rvn, rkb, rvb, ro, rl});
  if (s != DIT_OK) return s;
  if (m > ditattn::layout_copy_max_rows(D, 2)) return DIT_ERR_UNSUPPORTED;  // copy grid
  // 1) fresh patch rows overwrite their stale rows, K and V in one launch
  ditattn::CopyLaunch c;
  c.src = k_new;
  c.dst = static_cast<char*>(k_buf) + static_cast<long long>(row0) * D * 2;
  c.src2 = v_new;
  c.dst2 = static_cast<char*>(v_buf) + static_cast<long long>(row0) * D * 2;
  c.ss = {static_cast<long long>(H) * m * D, static_cast<long long>(m) * D, D};
  c.ds = {H * hs, hs, D};
  c.batch = B;
  c.heads = H;
  c.n = m;
  c.d = D;
  c.elem_bytes = 2;
  if (ditattn::launch_layout_copy(c, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return DIT_ERR_CUDA;
  // 2) the patch's queries against the whole buffer (fresh own rows, stale others)
  return run_contiguous(q, k_buf, v_buf, out, lse, B, H, m, N, D, hs, scale, out_dtype, stream,
                        false, splits, workspace);
}

size_t dit_attn_splitkv_workspace_bytes(int B, int H, int N_q, int D, int splits) {
  if (B < 1 || H < 1 || N_q < 1 || D < 1 || splits < 1) return 0;
  if (splits == 1) return 0;
  return static_cast<size_t>(splitkv_bytes(static_cast<long long>(B) * H * N_q, D, splits));
}

int dit_attn_splitkv_suggest(int B, int H, int N_q, int n_kv) {
  if (B < 1 || H < 1 || N_q < 1 || n_kv < 1) return 1;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms < 1)
    return 1;
  // Estimated time of each split count S on the persistent grid (one CTA per SM walking the
  // (head, Q pair, key range) items): ceil(items * S / SMs) waves, each as long as one item's
  // ceil(T / S) KV tiles plus a fixed per-item cost (Q load, first and last tiles, the O drain:
  // about four tile periods, measured), plus for S > 1 the merge launch, which reads the S fp32
  // partials and writes the output at HBM speed.  A tile period is about 1.5 us (both Q tiles of
  // a CTA against one 128-key tile).  The cheapest S wins (ties: fewer splits).
  constexpr double kTileUs = 1.5, kItemTiles = 4.0, kMergeLaunchUs = 5.0, kHbmBytesPerUs = 6.5e6;
  const long long items = static_cast<long long>(B) * H * ((N_q + 255) / 256);
  const long long tiles = (n_kv + 127) / 128;
  const double rows = static_cast<double>(B) * H * N_q;
  auto cost = [&](long long S) {
    const long long waves = (items * S + sms - 1) / sms;
    const long long item_tiles = (tiles + S - 1) / S;
    double us = static_cast<double>(waves) * (static_cast<double>(item_tiles) + kItemTiles) * kTileUs;
    if (S > 1) us += kMergeLaunchUs + rows * (S + 1) * (128 * 4 + 4) / kHbmBytesPerUs;
    return us;
  };
  long long best = 1;
  double best_us = cost(1);
  const long long s_max = std::min<long long>(16, tiles / 2);
  for (long long S = 2; S <= s_max; ++S) {
    const double us = cost(S);
    if (us < best_us) {
      best_us = us;
      best = S;
    }
  }
  return static_cast<int>(best);
}

dit_status dit_attn_chunk_fwd_splitkv(const void* q, const void* k, const void* v, void* out,
                                      float* lse, int B, int H, int N_q, int n_kv, int D,
                                      long long kv_head_stride, float scale, dit_dtype out_dtype,
                                      int splits, void* workspace, size_t workspace_bytes,
                                      dit_stream stream) {
  dit_status s = validate_attention(q, k, v, out, lse, B, H, N_q, n_kv, D, kv_head_stride, scale,
                                    out_dtype);
  if (s != DIT_OK) return s;
  const long long bh = static_cast<long long>(B) * H;
  if (((N_q + 255) / 256) * bh * splits > INT_MAX) return DIT_ERR_INVALID_ARG;
  const long long kv_bytes = ((bh - 1) * kv_head_stride + static_cast<long long>(n_kv) * D) * 2;
  s = validate_splits(splits, n_kv, workspace, workspace_bytes, B, H, N_q, D,
                      {span(q, bh * N_q * D * 2), span(k, kv_bytes), span(v, kv_bytes),
                       span(out, bh * N_q * D * dtype_bytes(out_dtype)), span(lse, bh * N_q * 4)});
  if (s != DIT_OK) return s;
  return run_contiguous(q, k, v, out, lse, B, H, N_q, n_kv, D, kv_head_stride, scale, out_dtype,
                        stream, false, splits, workspace);
}

dit_status dit_attn_chunk_fwd_splitkv_noalloc(const void* q, const void* k, const void* v,
                                              void* out, float* lse, int B, int H, int N_q,
                                              int n_kv, int D, long long kv_head_stride,
                                              float scale, dit_dtype out_dtype, int splits,
                                              dit_stream stream) {
  dit_status s = validate_attention(q, k, v, out, lse, B, H, N_q, n_kv, D, kv_head_stride, scale,
                                    out_dtype);
  if (s != DIT_OK) return s;
  const long long bh = static_cast<long long>(B) * H;
  const int tiles = (n_kv + 127) / 128;
  if (splits < 1 || splits > 64 || splits > tiles) return DIT_ERR_INVALID_ARG;
  if (((N_q + 255) / 256) * bh * splits > INT_MAX) return DIT_ERR_INVALID_ARG;
  // The partials must fit the fixed scratch; nothing in it needs to start at zero (the pass
  // writes every partial element the merge reads).
  if (splits > 1 && splitkv_bytes(bh * N_q, D, splits) >
                        static_cast<long long>(ditattn::kNoAllocScratchBytes))
    return DIT_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  if (splits > 1 && !(scratch = ditattn::noalloc_scratch())) return DIT_ERR_CUDA;
  return run_contiguous(q, k, v, out, lse, B, H, N_q, n_kv, D, kv_head_stride, scale, out_dtype,
                        stream, false, splits, scratch);
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
