// Host side of the attention kernel: TMA descriptor encoding and launch.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <mutex>

#include "attn_host.cuh"
#include "launch.h"

namespace ditattn {
namespace {

// Test-only failure injection (dit_test_inject_stall).
int g_stall_kv = 0;
long long g_wait_limit = kDefaultWaitLimit;
// Test-only cap on the persistent grid (0: one CTA per SM).
int g_grid_limit = 0;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encoder() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q{};
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(f);
  });
  return fn;
}

// 4-D bf16 map (d, rows, heads, batch) of a strided [B, H, rows, d] view, with
// 128-row x 64-column boxes and 128-byte swizzle; rows past `rows` read as zero.
bool encode_view(CUtensorMap* m, const void* base, int d, int rows, int heads, int batch,
                 const Strides& st) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  const cuuint64_t dims[4] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch)};
  const cuuint64_t strides[3] = {static_cast<cuuint64_t>(st.n_) * 2,
                                 static_cast<cuuint64_t>(st.h_) * 2,
                                 static_cast<cuuint64_t>(st.b_) * 2};
  const cuuint32_t box[4] = {64, static_cast<cuuint32_t>(kBlockM), 1, 1};
  const cuuint32_t elem_strides[4] = {1, 1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides, box,
            elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 5-D map (d, rows, heads, batch, key range) of the output (bf16 or fp32) of a short-item
// pass, for its TMA stores: boxes of 128 rows x 128 bytes (64 bf16 or 32 fp32 columns),
// 128-byte swizzle (the P tile's layout); rows past `rows` are not written.  Range r's
// output starts range_stride elements after range r-1's (one range: the stride only has to
// be valid).
bool encode_out_view(CUtensorMap* m, void* base, bool f32, int d, int rows, int heads, int batch,
                     int ranges, const Strides& st, long long range_stride) {
  EncodeTiledFn fn = encoder();
  if (!fn) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  const cuuint64_t dims[5] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(rows),
                              static_cast<cuuint64_t>(heads), static_cast<cuuint64_t>(batch),
                              static_cast<cuuint64_t>(ranges)};
  const cuuint64_t strides[4] = {static_cast<cuuint64_t>(st.n_) * es,
                                 static_cast<cuuint64_t>(st.h_) * es,
                                 static_cast<cuuint64_t>(st.b_) * es,
                                 static_cast<cuuint64_t>(range_stride) * es};
  const cuuint32_t box[5] = {static_cast<cuuint32_t>(128 / es), static_cast<cuuint32_t>(kBlockM),
                             1, 1, 1};
  const cuuint32_t elem_strides[5] = {1, 1, 1, 1, 1};
  return fn(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 5, base,
            dims, strides, box, elem_strides, CU_TENSOR_MAP_INTERLEAVE_NONE,
            CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

cudaError_t launch_attention(const AttnLaunch& a, cudaStream_t st) {
  AttnParams prm;
  if (!encode_view(&prm.tm_q, a.q, a.d, a.n_q, a.heads, a.batch, a.qs) ||
      !encode_view(&prm.tm_k, a.k, a.d, a.n_kv, a.heads, a.batch, a.ks) ||
      !encode_view(&prm.tm_v, a.v, a.d, a.n_kv, a.heads, a.batch, a.vs))
    return cudaErrorInvalidValue;
  const bool split = a.splits > 1;
  const bool batched = a.chunks > 0;
  if (split && (a.accumulate || batched || !a.ws_o || !a.ws_lse)) return cudaErrorInvalidValue;
  if (batched && (a.accumulate || a.chunks > kMaxRanges || !a.chunk_starts))
    return cudaErrorInvalidValue;
  if (!a.lse && (a.accumulate || split || batched)) return cudaErrorInvalidValue;
  // Split-KV passes write fp32 partials, contiguous, into the workspace.
  const bool f32 = split || a.out_f32;
  void* const obase = split ? static_cast<void*>(a.ws_o) : a.out;
  const Strides os = split ? Strides{static_cast<long long>(a.heads) * a.n_q * a.d,
                                     static_cast<long long>(a.n_q) * a.d, a.d}
                           : a.os;
  prm.out_f32 = f32 ? static_cast<float*>(obase) : nullptr;
  prm.out_bf16 = f32 ? nullptr : static_cast<__nv_bfloat16*>(obase);
  prm.o_sb = os.b_;
  prm.o_sh = os.h_;
  prm.o_sn = os.n_;
  // 32-byte row segments need the base and every stride (in bytes) 32-byte aligned.
  const long long esize = f32 ? 4 : 2;
  prm.out_align32 = (reinterpret_cast<uintptr_t>(obase) % 32 == 0 && (os.b_ * esize) % 32 == 0 &&
                     (os.h_ * esize) % 32 == 0 && (os.n_ * esize) % 32 == 0)
                        ? 1
                        : 0;
  prm.lse = split ? a.ws_lse : a.lse;
  prm.status = a.status;
  prm.n_q = a.n_q;
  prm.n_kv = a.n_kv;
  prm.bh_count = a.batch * a.heads;
  prm.heads = a.heads;
  prm.q_pairs = (a.n_q + 2 * kBlockM - 1) / (2 * kBlockM);
  prm.splits = split ? a.splits : batched ? a.chunks : 1;
  prm.tiles_total = (a.n_kv + kBlockN - 1) / kBlockN;
  const long long rows = static_cast<long long>(prm.bh_count) * a.n_q;
  prm.ws_o_stride = (split || batched) ? rows * a.d : 0;
  prm.ws_l_stride = (split || batched) ? rows : 0;
  prm.explicit_ranges = batched ? 1 : 0;
  for (int c = 0; c <= kMaxRanges; ++c)
    prm.kv_starts[c] = (batched && c <= a.chunks) ? a.chunk_starts[c] : 0;
  prm.num_items = prm.q_pairs * prm.bh_count * prm.splits;
  prm.scale_log2 = a.scale * 1.4426950408889634f;
  prm.wait_limit = g_wait_limit;
  prm.stall_kv = g_stall_kv;
  // KV tiles of the longest work item: short items take the soft-drain form.
  int item_tiles = prm.tiles_total;
  if (batched) {
    item_tiles = 0;
    for (int c = 0; c < a.chunks; ++c)
      item_tiles = std::max(item_tiles, (a.chunk_starts[c + 1] - a.chunk_starts[c] + kBlockN - 1) /
                                            kBlockN);
  } else if (split) {
    item_tiles = (prm.tiles_total + a.splits - 1) / a.splits;
  }
  // Short items store O (or part of it) through a TMA map of the output; where the output
  // view cannot be mapped (alignment), they take the epilogue-drain form instead.
  bool short_items = item_tiles <= host::kShortItemTiles && !a.accumulate;
  if (short_items)
    short_items = encode_out_view(&prm.tm_o, obase, f32, a.d, a.n_q, a.heads, a.batch, prm.splits,
                                  os, (split || batched) ? prm.ws_o_stride : os.b_ * a.batch);
  if (a.accumulate) {
    if (!a.out_f32) return cudaErrorInvalidValue;
    return a.d == 64 ? host::launch_typed<64, true, true>(prm, st, g_grid_limit)
                     : host::launch_typed<128, true, true>(prm, st, g_grid_limit);
  }
  if (split) {
    const cudaError_t e = short_items ? host::launch_short(prm, a.d, true, true, st, g_grid_limit)
                          : a.d == 64 ? host::launch_typed<64, true>(prm, st, g_grid_limit)
                                      : host::launch_typed<128, true>(prm, st, g_grid_limit);
    if (e != cudaSuccess) return e;
    MergeLaunch m;
    m.partials = a.ws_o;
    m.lses = a.ws_lse;
    m.p = a.splits;
    m.rows = rows;
    m.d = a.d;
    m.out = a.out;
    m.lse = a.lse;
    m.part_f32 = true;
    m.out_f32 = a.out_f32;
    return launch_merge(m, st);
  }
  if (!a.lse) {  // no LSE output (one key range; checked above)
    if (short_items) return host::launch_short(prm, a.d, a.out_f32, false, st, g_grid_limit);
    if (a.d == 64)
      return a.out_f32 ? host::launch_typed<64, true, false, false>(prm, st, g_grid_limit)
                       : host::launch_typed<64, false, false, false>(prm, st, g_grid_limit);
    return a.out_f32 ? host::launch_typed<128, true, false, false>(prm, st, g_grid_limit)
                     : host::launch_typed<128, false, false, false>(prm, st, g_grid_limit);
  }
  if (short_items) return host::launch_short(prm, a.d, a.out_f32, true, st, g_grid_limit);
  if (a.d == 64)
    return a.out_f32 ? host::launch_typed<64, true>(prm, st, g_grid_limit)
                     : host::launch_typed<64, false>(prm, st, g_grid_limit);
  return a.out_f32 ? host::launch_typed<128, true>(prm, st, g_grid_limit)
                   : host::launch_typed<128, false>(prm, st, g_grid_limit);
}

void set_grid_limit(int max_ctas) { g_grid_limit = max_ctas > 0 ? max_ctas : 0; }

void set_stall_injection(int enable, long long wait_limit_cycles) {
  g_stall_kv = enable ? 1 : 0;
  g_wait_limit = wait_limit_cycles > 0 ? wait_limit_cycles : kDefaultWaitLimit;
}

}  // namespace ditattn
