// Fused non-causal attention forward for sm_103a: tcgen05 MMA with TMEM
// accumulators, TMA-staged bf16 tiles, fp32 online softmax.
//
// Computes, per head bh and query row i of the CTA's two 128-row Q tiles,
//   o_i = sum_j softmax_j(scale * q_i . k_j) v_j   over key rows j in [0, n_kv)
//   lse_i = ln sum_j exp(scale * q_i . k_j)
// (MindIE-SD parallelism docs, "Ring Sequence Parallel" usage example: local
// attention; arganzheng.life multi-GPU diffusion parallelism, section 4.2 Ring:
// one KV block per round, combined by online softmax).  The same kernel serves
// the fused pass (n_kv = N) and one KV chunk of the ring decomposition (K/V
// pointers offset to the chunk, n_kv = chunk length, explicit head stride).
//
// CTA organisation (320 threads, one CTA per SM):
//   warps 0-3  softmax for Q tile 0   (thread = query row = TMEM lane)
//   warps 4-7  softmax for Q tile 1
//   warp  8    TMA producer (Q once, then K_j / V_j through a 3-slot ring)
//   warp  9    TMEM allocator + single-thread tcgen05.mma issuer
// Tensor memory (512 columns): S0 | S1 | O0 | O1, fp32, lane = query row.
// Shared memory: Q0, Q1, P0, P1 (bf16 probabilities, written by the softmax
// warps in the 128-byte-swizzled K-major layout the MMA reads) and the K/V ring.
//
// Per KV tile j the MMA warp issues, in order,
//   O0 += P0_j V_j ; S0 = Q0 K_{j+1}^T ; O1 += P1_j V_j ; S1 = Q1 K_{j+1}^T
// so the tensor core works on one Q tile while the other tile's softmax runs.
// A commit after S_t(j+1) also covers PV_t(j), so when softmax t sees S_t(j+1)
// ready, O_t and P_t are free: one S, O and P buffer per Q tile suffice.
//
// Online softmax (base 2, scale folded into log2e): the running max m is only
// raised when a tile's max exceeds it by more than kRescaleLog2 (then O and l
// are rescaled by 2^(m_old - m_new)); otherwise exponentials are taken against
// the stale m, which bounds P by 2^kRescaleLog2.  The result is exact either
// way: O / l and m + log2 l do not depend on which m was used.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

namespace ditattn {

constexpr int kBlockM = 128;              // query rows per Q tile (two per CTA)
constexpr int kBlockN = 128;              // keys per KV tile
constexpr int kStages = 3;                // K/V ring slots
constexpr int kThreads = 320;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleLog2 = 8.0f;      // lazy-rescale threshold (log2 units)
constexpr long long kDefaultWaitLimit = 4000000000LL;  // ~2 s of SM clocks per wait
constexpr int kStatusTimeout = 1;

struct AttnParams {
  CUtensorMap tm_q;   // (D, n_q, bh) bf16, box (64, 128, 1), 128B swizzle
  CUtensorMap tm_k;   // (D, n_kv, bh), head stride = kv_head_stride
  CUtensorMap tm_v;
  void* out;          // [bh, n_q, D] fp32 or bf16
  float* lse;         // [bh, n_q]
  int* status;        // device status word (timeouts)
  int n_q;
  int n_kv;
  int bh_count;
  int q_pairs;        // ceil(n_q / 256)
  float scale_log2;   // scale * log2(e)
  long long wait_limit;  // SM clocks a bounded wait may spin before giving up
  int stall_kv;          // test-only failure injection: never issue K/V copies
};

template <int D>
struct AttnSmem {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr uint32_t kRegion = kBlockM * 128;        // one 128-byte-wide swizzle column
  static constexpr uint32_t kTile = kBlockM * D * 2;        // Q / K / V tile
  static constexpr uint32_t kPTile = kBlockM * kBlockN * 2; // P tile
  static constexpr uint32_t kQ0 = 0;
  static constexpr uint32_t kQ1 = kQ0 + kTile;
  static constexpr uint32_t kP0 = kQ1 + kTile;
  static constexpr uint32_t kP1 = kP0 + kPTile;
  static constexpr uint32_t kKV = kP1 + kPTile;
  static constexpr uint32_t kBars = kKV + kStages * kTile;
  // barrier indices
  static constexpr int bQFull = 0;
  static constexpr int bKVFull = 1;                  // + slot
  static constexpr int bKVEmpty = bKVFull + kStages; // + slot
  static constexpr int bSFull = bKVEmpty + kStages;  // + tile
  static constexpr int bPFull = bSFull + 2;          // + tile
  static constexpr int bODone = bPFull + 2;
  static constexpr int bDrain = bODone + 1;
  static constexpr int kNumBars = bDrain + 1;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kUsed = kAbort + 4;
  static constexpr uint32_t kBytes = kUsed + 1024;   // slack for 1024-byte alignment
  static_assert(kBytes <= 232448, "shared memory budget");
};

namespace detail {

// Bounded wait that also gives up when another role has aborted.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              const volatile int* abort_flag, long long limit) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  while (!ptx::mbar_try_wait(bar, parity)) {
    if (*abort_flag) return false;
    if (clock64() - t0 > limit) return false;
  }
  return true;
}

__device__ __forceinline__ void raise_abort(const AttnParams& p, volatile int* abort_flag) {
  *abort_flag = 1;
  atomicOr(p.status, kStatusTimeout);
}

template <int D>
__device__ __forceinline__ void producer(const AttnParams& p, uint32_t sbase, int bh, int q_row0,
                                         int n_tiles, volatile int* abort_flag) {
  using L = AttnSmem<D>;
  constexpr int kRegions = D / 64;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };

  ptx::mbar_arrive_expect_tx(bar(L::bQFull), 2 * L::kTile);
#pragma unroll
  for (int t = 0; t < 2; ++t)
#pragma unroll
    for (int r = 0; r < kRegions; ++r)
      ptx::tma_load_3d(sbase + (t ? L::kQ1 : L::kQ0) + r * L::kRegion, &p.tm_q, bar(L::bQFull),
                       r * 64, q_row0 + t * kBlockM, bh);

  if (p.stall_kv) return;  // test-only: the consumers' first K wait will expire

  int last_it[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) last_it[s] = -1;
  bool ok = true;
  for (int it = 0; it < 2 * n_tiles; ++it) {
    const int s = it % kStages;
    const uint32_t ph = (it / kStages) & 1;
    if (!wait_or_abort(bar(L::bKVEmpty + s), ph ^ 1, abort_flag, p.wait_limit)) {
      ok = false;
      break;
    }
    const CUtensorMap* tm = (it & 1) ? &p.tm_v : &p.tm_k;
    const int j = it >> 1;
    ptx::mbar_arrive_expect_tx(bar(L::bKVFull + s), L::kTile);
#pragma unroll
    for (int r = 0; r < kRegions; ++r)
      ptx::tma_load_3d(sbase + L::kKV + s * L::kTile + r * L::kRegion, tm, bar(L::bKVFull + s),
                       r * 64, j * kBlockN, bh);
#pragma unroll
    for (int q = 0; q < kStages; ++q)
      if (q == s) last_it[q] = it;
  }
  if (!ok) {
    raise_abort(p, abort_flag);
    // Let every copy this thread started land before the CTA can exit.
    ptx::mbar_wait(bar(L::bQFull), 0, p.wait_limit);
#pragma unroll
    for (int s = 0; s < kStages; ++s)
      if (last_it[s] >= 0)
        ptx::mbar_wait(bar(L::bKVFull + s), (last_it[s] / kStages) & 1, p.wait_limit);
  }
}

template <int D>
__device__ __forceinline__ void mma_issuer(const AttnParams& p, uint32_t sbase, uint32_t tmem,
                                           int n_tiles, volatile int* abort_flag) {
  using L = AttnSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  constexpr uint32_t kIdescQK = ptx::idesc_bf16_f32(kBlockM, kBlockN, false, false);
  constexpr uint32_t kIdescPV = ptx::idesc_bf16_f32(kBlockM, D, false, true);
  const uint32_t qs[2] = {sbase + L::kQ0, sbase + L::kQ1};
  const uint32_t ps[2] = {sbase + L::kP0, sbase + L::kP1};

  // S_t = Q_t K^T: K-major A and B, 16 keys' worth of D per instruction.
  auto issue_s = [&](int t, int slot) {
    const uint32_t kb = sbase + L::kKV + slot * L::kTile;
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = (k / 4) * L::kRegion + (k % 4) * 32;
      ptx::mma_bf16_ss(tmem + t * kBlockN, ptx::sdesc_sw128(qs[t] + off, 16, 1024),
                       ptx::sdesc_sw128(kb + off, 16, 1024), kIdescQK, k > 0 ? 1u : 0u);
    }
  };
  // O_t += P_t V: P K-major, V MN-major (D contiguous); 16 keys per instruction.
  auto issue_pv = [&](int t, int slot, bool acc) {
    const uint32_t vb = sbase + L::kKV + slot * L::kTile;
#pragma unroll
    for (int k = 0; k < kBlockN / 16; ++k) {
      const uint32_t aoff = (k / 4) * L::kRegion + (k % 4) * 32;
      ptx::mma_bf16_ss(tmem + 2 * kBlockN + t * D, ptx::sdesc_sw128(ps[t] + aoff, 16, 1024),
                       ptx::sdesc_sw128(vb + k * 16 * 128, L::kRegion, 1024), kIdescPV,
                       (acc || k > 0) ? 1u : 0u);
    }
  };
  auto kv_wait = [&](int it) {
    return wait_or_abort(bar(L::bKVFull + it % kStages), (it / kStages) & 1, abort_flag,
                         p.wait_limit);
  };

  bool ok = wait_or_abort(bar(L::bQFull), 0, abort_flag, p.wait_limit) && kv_wait(0);
  if (ok) {
    ptx::tc_fence_after();
    issue_s(0, 0);
    ptx::mma_commit(bar(L::bSFull + 0));
    issue_s(1, 0);
    ptx::mma_commit(bar(L::bSFull + 1));
    ptx::mma_commit(bar(L::bKVEmpty + 0));
  }
  for (int j = 0; ok && j < n_tiles; ++j) {
    const int itV = 2 * j + 1, sV = itV % kStages;
    const int itK = 2 * j + 2, sK = itK % kStages;
    const bool more = j + 1 < n_tiles;
    if (!(ok = kv_wait(itV))) break;
    if (!(ok = wait_or_abort(bar(L::bPFull + 0), j & 1, abort_flag, p.wait_limit))) break;
    ptx::tc_fence_after();
    issue_pv(0, sV, j > 0);
    if (more) {
      if (!(ok = kv_wait(itK))) break;
      ptx::tc_fence_after();
      issue_s(0, sK);
      ptx::mma_commit(bar(L::bSFull + 0));
    }
    if (!(ok = wait_or_abort(bar(L::bPFull + 1), j & 1, abort_flag, p.wait_limit))) break;
    ptx::tc_fence_after();
    issue_pv(1, sV, j > 0);
    ptx::mma_commit(bar(L::bKVEmpty + sV));
    if (more) {
      issue_s(1, sK);
      ptx::mma_commit(bar(L::bSFull + 1));
      ptx::mma_commit(bar(L::bKVEmpty + sK));
    }
  }
  if (ok) {
    ptx::mma_commit(bar(L::bODone));
  } else {
    raise_abort(p, abort_flag);
    // No MMA may still be writing tensor memory when it is released.
    ptx::mma_commit(bar(L::bDrain));
    ptx::mbar_wait(bar(L::bDrain), 0, p.wait_limit);
  }
}

template <int D, bool kOutF32>
__device__ __forceinline__ void softmax_epilogue(const AttnParams& p, uint32_t sbase,
                                                 uint32_t tmem, int t, int warp, int lane, int bh,
                                                 int q_row0, int n_tiles,
                                                 volatile int* abort_flag) {
  using L = AttnSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;  // row in the Q tile == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + t * kBlockN + lane_off;
  const uint32_t tO = tmem + 2 * kBlockN + t * D + lane_off;
  const uint32_t sP = sbase + (t ? L::kP1 : L::kP0);
  const float c = p.scale_log2;

  float m = -INFINITY;  // running max of scale*log2e*s (possibly stale by < 2^8)
  float l = 0.f;        // running sum of 2^(c*s - m), for the LSE
  float lp = 0.f;       // running sum of the bf16-rounded P the PV GEMM sees, for O
  bool ok = true;
  for (int j = 0; j < n_tiles; ++j) {
    ok = wait_or_abort(bar(L::bSFull + t), j & 1, abort_flag, p.wait_limit);
    if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
    ptx::tc_fence_after();

    float s[kBlockN];
#pragma unroll
    for (int cc = 0; cc < kBlockN / 32; ++cc) {
      uint32_t u[32];
      ptx::tmem_ld32(tS + cc * 32, u);
#pragma unroll
      for (int i = 0; i < 32; ++i) s[cc * 32 + i] = __uint_as_float(u[i]);
    }
    ptx::tmem_wait_ld();

    const int valid = p.n_kv - j * kBlockN;
    if (valid < kBlockN) {
#pragma unroll
      for (int i = 0; i < kBlockN; ++i)
        if (i >= valid) s[i] = -INFINITY;
    }
    // Tile row max: 8 independent 3-input max chains, then a short tree.
    float mx;
    {
      float a[8];
#pragma unroll
      for (int g = 0; g < 8; ++g) {
        a[g] = ptx::fmax3(s[16 * g], s[16 * g + 1], s[16 * g + 2]);
#pragma unroll
        for (int i = 3; i < 15; i += 2) a[g] = ptx::fmax3(a[g], s[16 * g + i], s[16 * g + i + 1]);
        a[g] = fmaxf(a[g], s[16 * g + 15]);
      }
      mx = ptx::fmax3(ptx::fmax3(a[0], a[1], a[2]), ptx::fmax3(a[3], a[4], a[5]), fmaxf(a[6], a[7]));
    }
    const float m_tile = mx * c;
    const bool raise = m_tile > m + kRescaleLog2;  // always true on the first tile
    float alpha = 1.f;
    if (raise) {
      alpha = ptx::ex2_approx(m - m_tile);  // 0 on the first tile (m = -inf)
      m = m_tile;
    }
    l *= alpha;
    lp *= alpha;
    if (j > 0 && __any_sync(0xffffffffu, raise)) {
      // PV_t(j-1) has completed (covered by the commit after S_t(j)); rescale O_t.
#pragma unroll
      for (int cc = 0; cc < D / 16; ++cc) {
        uint32_t u[16];
        ptx::tmem_ld16(tO + cc * 16, u);
        ptx::tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 16; ++i) u[i] = __float_as_uint(__uint_as_float(u[i]) * alpha);
        ptx::tmem_st16(tO + cc * 16, u);
      }
      ptx::tmem_wait_st();
    }

    // P = 2^(c*s - m), two elements per packed FMA.
    const uint64_t c2 = ptx::f2pack(c, c);
    const uint64_t nm2 = ptx::f2pack(-m, -m);
#pragma unroll
    for (int i = 0; i < kBlockN; i += 2) {
      float x0, x1;
      ptx::f2unpack(ptx::ffma2(ptx::f2pack(s[i], s[i + 1]), c2, nm2), x0, x1);
      s[i] = ptx::ex2_approx(x0);
      s[i + 1] = ptx::ex2_approx(x1);
    }

    // Pack P to bf16, store it (row r -> two 128-byte-swizzled K-major regions: keys 0-63,
    // 64-127), and accumulate both row sums in 4 independent packed chains each.
    uint64_t acc_l[4], acc_lp[4];
#pragma unroll
    for (int g = 0; g < 4; ++g) acc_l[g] = acc_lp[g] = 0;
#pragma unroll
    for (int ch = 0; ch < kBlockN / 8; ++ch) {
      uint32_t w[4];
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const float p0 = s[8 * ch + 2 * g], p1 = s[8 * ch + 2 * g + 1];
        w[g] = ptx::pack_bf16x2(p0, p1);
        acc_l[g] = ptx::fadd2(acc_l[g], ptx::f2pack(p0, p1));
        acc_lp[g] = ptx::fadd2(acc_lp[g], ptx::f2pack(ptx::bf16lo(w[g]), ptx::bf16hi(w[g])));
      }
      const uint32_t addr =
          sP + (ch / 8) * L::kRegion + r * 128 + ((((ch % 8) ^ (r & 7))) << 4);
      asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]),
                   "r"(w[2]), "r"(w[3])
                   : "memory");
    }
    {
      const uint64_t sl = ptx::fadd2(ptx::fadd2(acc_l[0], acc_l[1]), ptx::fadd2(acc_l[2], acc_l[3]));
      const uint64_t sp = ptx::fadd2(ptx::fadd2(acc_lp[0], acc_lp[1]),
                                     ptx::fadd2(acc_lp[2], acc_lp[3]));
      float a0, a1, b0, b1;
      ptx::f2unpack(sl, a0, a1);
      ptx::f2unpack(sp, b0, b1);
      l += a0 + a1;
      lp += b0 + b1;
    }
    ptx::fence_proxy_async_smem();
    ptx::tc_fence_before();
    ptx::mbar_arrive(bar(L::bPFull + t));
  }
  if (ok) {
    ok = wait_or_abort(bar(L::bODone), 0, abort_flag, p.wait_limit);
    ok = __all_sync(0xffffffffu, ok);
  }
  if (!ok) {
    raise_abort(p, abort_flag);
    return;
  }
  ptx::tc_fence_after();

  const int row = q_row0 + t * kBlockM + r;
  const bool store = row < p.n_q;
  // O is normalised by the sum of the rounded weights it was built from, so the weights
  // sum to one; the LSE uses the unrounded sum.
  const float inv_l = 1.f / lp;
  const size_t out_row = (static_cast<size_t>(bh) * p.n_q + row) * D;
#pragma unroll
  for (int cc = 0; cc < D / 32; ++cc) {
    uint32_t u[32];
    ptx::tmem_ld32(tO + cc * 32, u);
    ptx::tmem_wait_ld();
    if (store) {
      if constexpr (kOutF32) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) + out_row + cc * 32);
#pragma unroll
        for (int i = 0; i < 8; ++i)
          dst[i] = make_float4(__uint_as_float(u[4 * i + 0]) * inv_l,
                               __uint_as_float(u[4 * i + 1]) * inv_l,
                               __uint_as_float(u[4 * i + 2]) * inv_l,
                               __uint_as_float(u[4 * i + 3]) * inv_l);
      } else {
        uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) + out_row + cc * 32);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          uint4 w;
          w.x = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 0]) * inv_l, __uint_as_float(u[8 * i + 1]) * inv_l);
          w.y = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 2]) * inv_l, __uint_as_float(u[8 * i + 3]) * inv_l);
          w.z = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 4]) * inv_l, __uint_as_float(u[8 * i + 5]) * inv_l);
          w.w = ptx::pack_bf16x2(__uint_as_float(u[8 * i + 6]) * inv_l, __uint_as_float(u[8 * i + 7]) * inv_l);
          dst[i] = w;
        }
      }
    }
  }
  if (store) p.lse[static_cast<size_t>(bh) * p.n_q + row] = (m + log2f(l)) * 0.69314718055994530942f;
}

}  // namespace detail

template <int D, bool kOutF32>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  using L = AttnSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const int bh = blockIdx.x / p.q_pairs;
  const int q_row0 = (blockIdx.x % p.q_pairs) * 2 * kBlockM;
  const int n_tiles = (p.n_kv + kBlockN - 1) / kBlockN;

  if (threadIdx.x == 0) {
    auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
    ptx::mbar_init(bar(L::bQFull), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(L::bKVFull + s), 1);
      ptx::mbar_init(bar(L::bKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar(L::bSFull + t), 1);
      ptx::mbar_init(bar(L::bPFull + t), kBlockM);
    }
    ptx::mbar_init(bar(L::bODone), 1);
    ptx::mbar_init(bar(L::bDrain), 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
  }
  if (warp == kLoadWarp && lane == 0) {
    ptx::tma_prefetch_desc(&p.tm_q);
    ptx::tma_prefetch_desc(&p.tm_k);
    ptx::tma_prefetch_desc(&p.tm_v);
  }
  if (warp == kMmaWarp) {
    ptx::tmem_alloc(sbase + L::kTmemSlot, 512);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kTmemSlot);

  if (warp == kLoadWarp) {
    if (lane == 0) detail::producer<D>(p, sbase, bh, q_row0, n_tiles, abort_flag);
  } else if (warp == kMmaWarp) {
    if (lane == 0) detail::mma_issuer<D>(p, sbase, tmem, n_tiles, abort_flag);
    __syncwarp();
  } else {
    detail::softmax_epilogue<D, kOutF32>(p, sbase, tmem, warp >> 2, warp, lane, bh, q_row0,
                                         n_tiles, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
}

}  // namespace ditattn
