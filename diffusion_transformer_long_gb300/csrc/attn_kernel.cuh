// Fused non-causal attention forward for sm_103a: tcgen05 MMA with TMEM
// accumulators, TMA-staged bf16 tiles, fp32 online softmax.
//
// Computes, per head bh and query row i,
//   o_i = sum_j softmax_j(scale * q_i . k_j) v_j   over key rows j in [0, n_kv)
//   lse_i = ln sum_j exp(scale * q_i . k_j)
// (MindIE-SD parallelism docs, "Ring Sequence Parallel" usage example: local
// attention; arganzheng.life multi-GPU diffusion parallelism, section 4.2 Ring:
// one KV block per round, combined by online softmax).  The same kernel serves
// the fused pass (n_kv = N), one KV chunk of the ring decomposition, all p chunks
// (virtual ranks) in one launch, the ring hop merged into a running (O, lse)
// (kAccum), and split-KV partials.  Q/K/V are read
// through 4-D tensor maps (d, rows, heads, batch) with any strides, O is written
// through per-head offsets and a row stride, so token-major (BSND) views work too.
//
// Persistent: one CTA per SM walks work items (head bh, pair of 128-row Q tiles,
// key range) w = blockIdx.x, blockIdx.x + gridDim.x, ...  (head-major, so the CTAs
// resident at any moment share a head's K/V in L2; the key range is the whole key
// set, a tile-aligned split, or one chunk at any row offset).  Every barrier's phase
// count runs on across items, so the next item's Q load and first S MMAs overlap this
// item's epilogue.
//
// CTA organisation (512 threads, four warpgroups):
//   warps 0-3   softmax for Q tile 0   (thread = query row = TMEM lane)
//   warps 4-7   softmax for Q tile 1
//   warp  8     TMA producer (Q per item, then K/V tiles through a 3-slot ring)
//   warp  9     TMEM allocator + single-thread issuer of S = Q K^T
//   warp 10     single-thread issuer of O += P V       (warp 11 idle)
//   warps 12-15 epilogue: O_t out of TMEM, normalised, stored; both Q tiles
//               (kSoftDrain, for work items of few KV tiles: each softmax warpgroup drains
//               its own O_t once the item's last PV has landed, staging it through its
//               P_t buffer for TMA stores, and warps 12-15 idle)
// Two issuers keep the tensor pipe fed: its queue is about one instruction deep,
// and a barrier wait stalls the waiting thread for longer than one MMA, so while
// one issuer waits the other issues.
// Tensor memory (512 columns): S0 | S1 | O0 | O1, fp32, lane = query row.
// Shared memory: Q0, Q1, P0, P1 (bf16 probabilities, written by the softmax
// warps in the 128-byte-swizzled K-major layout the MMA reads), the K/V ring and
// the per-row scale factors handed from the softmax to the epilogue.
//
// Pipeline.  A softmax warpgroup releases its S buffer (S_EMPTY) as soon as
// the scores are in registers, so the S issuer computes S_t(g+1) = Q_t K^T while
// softmax t is still turning S_t(g) into probabilities; softmax t starts the next
// tile the moment it has published P_t(g) (P_FULL).  O_t += P_t V is committed to
// its own barrier (PV_DONE), which softmax t waits on only before it rescales O_t
// or overwrites the P_t buffer.  P_t is published in two halves (keys 0-63 on P_LO,
// 64-127 on P_FULL), so the PV issuer starts on the first half while the softmax still
// computes the second.  Q_EMPTY (last S MMA of an item done) lets the
// producer refill Q; at an item's end softmax t publishes 1/rowsum (EPI_READY) and
// moves on; the epilogue warpgroup takes it (EPI_TAKEN), waits for the last PV,
// reads O_t and releases it (O_EMPTY) to the next item's first PV.  The K/V ring is
// filled in consumption order: K0, K1, V0, K2, V1, ... per item.
//
// Online softmax (base 2, scale folded into log2e): the running max m is only
// raised when a tile's max exceeds it by more than kRescaleLog2 (then O and the
// row sums are rescaled by 2^(m_old - m_new)); otherwise exponentials are taken
// against the stale m, which bounds P by 2^kRescaleLog2.  The result is exact
// either way: O / l and m + log2 l do not depend on which m was used.
#pragma once

#include <type_traits>

#include <cuda_bf16.h>
#include <cstdint>

#include "sm103_ptx.cuh"

// Optional phase tracing (compile with -DDITATTN_TRACE): one CTA records SM-clock
// timestamps of pipeline events for its first 64 KV tiles into
// ditattn_trace_buf[event][tile].  Compiled out by default.
#ifdef DITATTN_TRACE
#ifndef DITATTN_TRACE_CTA
#define DITATTN_TRACE_CTA 0
#endif
__device__ long long ditattn_trace_buf[32 * 64];
#define DIT_TRACE(ev, j)                                                   \
  do {                                                                      \
    if (blockIdx.x == DITATTN_TRACE_CTA && (j) >= 0 && (j) < 64)            \
      ditattn_trace_buf[(ev) * 64 + (j)] = clock64();                       \
  } while (0)
#else
#define DIT_TRACE(ev, j) \
  do {                   \
  } while (0)
#endif

namespace ditattn {

enum TraceEvent {
  kTrProdEmpty = 0, kTrProdIssue, kTrMmaK, kTrMmaS0, kTrMmaS1, kTrMmaV, kTrMmaP0, kTrMmaPv0,
  kTrMmaP1, kTrMmaPv1, kTrSmFull0, kTrSmLd0, kTrSmMax0, kTrSmExp0, kTrSmArrive0,
  kTrSmFull1, kTrSmLd1, kTrSmMax1, kTrSmExp1, kTrSmArrive1, kTrCta, kTrQIssue, kTrQFull
};
// Per-tile events are indexed by the CTA-global tile count; kTrCta slots: 0 start,
// 1 first S seen, then per item i: 2 + 2i epilogue start, 3 + 2i epilogue end
// (tile-0 warpgroup); 63 CTA exit.

constexpr int kBlockM = 128;              // query rows per Q tile (two per work item)
constexpr int kBlockN = 128;              // keys per KV tile
constexpr int kStages = 3;                // K/V ring slots
constexpr int kThreads = 512;
constexpr int kLoadWarp = 8;
constexpr int kMmaWarp = 9;     // S = Q K^T issuer, owns the TMEM allocation
constexpr int kPvWarp = 10;     // O += P V issuer
constexpr int kEpiWarp0 = 12;   // warps 12-15: epilogue warpgroup
// Register split (setmaxnreg): 512 threads launch with 128 registers each (65536); the
// producer/issuer warpgroup shrinks to 72 and the softmax warpgroups take what the
// epilogue warpgroup leaves: per SM sub-partition (one warp of each warpgroup) the four
// shares add up to 512, i.e. 65536 registers over the block.
//   epilogue drains O:        softmax 176, issuers 72, epilogue 88
//   softmax drains O (short
//   items, kSoftDrain):       softmax 208, issuers 72, the idle epilogue warpgroup 24
template <bool kSoftDrain>
struct RegSplit {
  static constexpr uint32_t kIssue = 72;
  static constexpr uint32_t kEpilogue = kSoftDrain ? 24 : 88;
  static constexpr uint32_t kSoftmax = (512 - kIssue - kEpilogue) / 2;
  static_assert(kSoftmax % 8 == 0 && 2 * kSoftmax + kIssue + kEpilogue == 512, "register split");
};
constexpr float kRescaleLog2 = 8.0f;      // lazy-rescale threshold (log2 units)
constexpr long long kDefaultWaitLimit = 4000000000LL;  // ~2 s of SM clocks per wait
constexpr int kStatusTimeout = 1;
constexpr int kMaxRanges = 64;            // key ranges (splits or explicit chunks) per launch

struct AttnParams {
  CUtensorMap tm_q;   // (D, n_q, bh) bf16, box (64, 128, 1), 128B swizzle
  CUtensorMap tm_k;   // (D, n_kv, bh), head stride = kv_head_stride
  CUtensorMap tm_v;
  CUtensorMap tm_o;   // output of the short-item form: (D, n_q, H, B, key range), boxes of
                      // 128 rows x 128 bytes, 128B swizzle (the P tile's layout)
  float* out_f32;     // (fp32 output) or null; O[b][h][n][d] at b*o_sb + h*o_sh + n*o_sn + d
  __nv_bfloat16* out_bf16;  // (bf16 output) or null; same addressing
  long long o_sb, o_sh, o_sn;  // output strides in elements
  int out_align32;    // base and strides keep every row segment 32-byte aligned
  float* lse;         // [bh, n_q] contiguous
  int* status;        // device status word (timeouts)
  int n_q;
  int n_kv;
  int bh_count;
  int heads;          // H: head bh is (b, h) = (bh / H, bh % H)
  int q_pairs;        // ceil(n_q / 256)
  int splits;         // key ranges per (head, Q pair): 1, or S for split-KV / chunk partials
  int tiles_total;    // ceil(n_kv / 128)
  long long ws_o_stride;  // elements between consecutive ranges' partial O (0 for one range)
  long long ws_l_stride;  // elements between consecutive ranges' partial LSEs (0 for one range)
  int explicit_ranges;    // 1: range s is keys [kv_starts[s], kv_starts[s+1]); 0: equal tile
                          // splits [s*T/S, (s+1)*T/S) of the T tiles
  int kv_starts[kMaxRanges + 1];
  int num_items;      // bh_count * q_pairs * splits
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
  static constexpr int bQFull = 0;                   // Q tiles of an item landed
  static constexpr int bQEmpty = 1;                  // last S MMA of an item done (MMA commit)
  static constexpr int bKFull = 2;                   // + slot: a K tile landed in the slot
  static constexpr int bVFull = bKFull + kStages;    // + slot: a V tile landed in the slot
  static constexpr int bKVEmpty = bVFull + kStages;  // + slot: the slot's tile was consumed
  static constexpr int bSFull = bKVEmpty + kStages;  // + tile: S_t computed (MMA commit)
  static constexpr int bSEmpty = bSFull + 2;         // + tile: S_t read into registers (128 arrivals)
  static constexpr int bPLo = bSEmpty + 2;           // + tile: keys 0-63 of P_t written (128)
  static constexpr int bPFull = bPLo + 2;            // + tile: keys 64-127 of P_t written (128)
  static constexpr int bPVDone = bPFull + 2;         // + tile: O_t += P_t V done (MMA commit)
  static constexpr int bOEmpty = bPVDone + 2;        // + tile: O_t read by the epilogue (128 arrivals)
  static constexpr int bEpiReady = bOEmpty + 2;      // + tile: normaliser of an item written (128)
  static constexpr int bEpiTaken = bEpiReady + 2;    // + tile: normaliser read by the epilogue (128)
  static constexpr int bStaged = bEpiTaken + 2;      // + tile: O_t staged in P_t (128 arrivals)
  static constexpr int bStageFree = bStaged + 2;     // + tile: P_t's staged O read by the TMA
  static constexpr int bDrainS = bStageFree + 2;     // abort drain, S issuer
  static constexpr int bDrainPV = bDrainS + 1;       // abort drain, PV issuer
  static constexpr int kNumBars = bDrainPV + 1;
  static constexpr uint32_t kTmemSlot = kBars + kNumBars * 8;
  static constexpr uint32_t kAbort = kTmemSlot + 4;
  static constexpr uint32_t kInvLp = (kAbort + 4 + 15) & ~15u;  // [2][128] fp32: 1 / row sum
  static constexpr uint32_t kUsed = kInvLp + 2 * kBlockM * 4;
  static constexpr uint32_t kBytes = kUsed + 1024;   // slack for 1024-byte alignment
  static_assert(kBytes <= 232448, "shared memory budget");
};

namespace detail {

// Bounded wait that also gives up when another role has aborted.  A phase that has already
// completed is seen by the non-blocking test first; otherwise try_wait suspends the thread.
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity,
                                              const volatile int* abort_flag, long long limit) {
  if (ptx::mbar_test_wait(bar, parity)) return true;
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

struct Item {
  int bh;      // b * H + h
  int b, h;
  int q_row0;  // first query row of the pair of Q tiles
  int split;   // key range of the item (0 unless split-KV or batched chunks)
  int kv0;     // first key row of the range
  int kv_len;  // keys in the range (>= 1)
  int ntiles;  // KV tiles in the range: ceil(kv_len / 128)
  __device__ __forceinline__ size_t out_off(const AttnParams& p) const {
    return static_cast<size_t>(b) * p.o_sb + static_cast<size_t>(h) * p.o_sh +
           static_cast<size_t>(split) * p.ws_o_stride;
  }
  __device__ __forceinline__ size_t lse_off(const AttnParams& p) const {
    return static_cast<size_t>(bh) * p.n_q + static_cast<size_t>(split) * p.ws_l_stride;
  }
};
// Work item w: (head, Q pair, key range), key range fastest.  Range s is either the tile
// split [s*T/S, (s+1)*T/S) of the T tiles (ending at n_kv), or keys [kv_starts[s],
// kv_starts[s+1]) (one virtual rank's chunk of the ring decomposition).
__device__ __forceinline__ Item item_of(const AttnParams& p, int w) {
  const int qi = w / p.splits;
  const int split = w - qi * p.splits;
  const int bh = qi / p.q_pairs;
  const int b = bh / p.heads;
  int kv0, kv1;
  if (p.explicit_ranges) {
    kv0 = p.kv_starts[split];
    kv1 = p.kv_starts[split + 1];
  } else {
    kv0 = static_cast<int>(static_cast<long long>(split) * p.tiles_total / p.splits) * kBlockN;
    kv1 = min(p.n_kv,
              static_cast<int>(static_cast<long long>(split + 1) * p.tiles_total / p.splits) *
                  kBlockN);
  }
  return {bh, b, bh - b * p.heads, (qi % p.q_pairs) * 2 * kBlockM, split, kv0, kv1 - kv0,
          (kv1 - kv0 + kBlockN - 1) / kBlockN};
}

// K/V ring items of one work item, in consumption order: K_0, then per KV tile j:
// K_{j+1} (if any), V_j.  Ring index i goes to slot i % kStages; the ring index runs on
// across work items (2 * n_tiles per item).  K and V tiles landing in a slot complete
// different barriers (K_FULL / V_FULL), so each MMA issuer observes the phases of only
// the barriers it consumes, in order, and can never mistake an older fill for a newer one.
__device__ __forceinline__ int k_item(int j) { return j == 0 ? 0 : 2 * j - 1; }
__device__ __forceinline__ int v_item(int j, int n_tiles) {
  return (j + 1 < n_tiles) ? 2 * j + 2 : 2 * j + 1;
}

template <int D>
__device__ __forceinline__ void producer(const AttnParams& p, uint32_t sbase,
                                         volatile int* abort_flag) {
  using L = AttnSmem<D>;
  constexpr int kRegions = D / 64;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  auto wait = [&](int b, uint32_t parity) {
    return wait_or_abort(bar(b), parity, abort_flag, p.wait_limit);
  };

  uint32_t kpar = 0, vpar = 0;  // bit s: parity of the next K_FULL[s] / V_FULL[s] phase
  int last_bar[kStages];        // barrier and parity of the newest copy into each slot
  uint32_t last_par[kStages];
#pragma unroll
  for (int s = 0; s < kStages; ++s) {
    last_bar[s] = -1;
    last_par[s] = 0;
  }
  int q_loads = 0;  // Q loads issued (QFULL phases armed)
  int it = 0;       // ring index
  bool ok = true;
  auto load = [&](bool is_v, int row, const Item& item) {
    const int s = it % kStages;
    const uint32_t ph = (it / kStages) & 1;
    if (!wait(L::bKVEmpty + s, ph ^ 1)) return false;
    DIT_TRACE(kTrProdEmpty, it);
    const int fb = (is_v ? L::bVFull : L::bKFull) + s;
    const uint32_t par = ((is_v ? vpar : kpar) >> s) & 1;
    if (is_v) vpar ^= 1u << s; else kpar ^= 1u << s;
    ptx::mbar_arrive_expect_tx(bar(fb), L::kTile);
    const CUtensorMap* tm = is_v ? &p.tm_v : &p.tm_k;
#pragma unroll
    for (int r = 0; r < kRegions; ++r)
      ptx::tma_load_4d(sbase + L::kKV + s * L::kTile + r * L::kRegion, tm, bar(fb), r * 64,
                       row, item.h, item.b);
    DIT_TRACE(kTrProdIssue, it);
#pragma unroll
    for (int q = 0; q < kStages; ++q)
      if (q == s) {
        last_bar[q] = fb;
        last_par[q] = par;
      }
    ++it;
    return true;
  };

  for (int w = blockIdx.x; ok && w < p.num_items; w += gridDim.x) {
    const Item item = item_of(p, w);
    // Q_t is free once the previous item's last S MMAs have completed.
    if (!(ok = wait(L::bQEmpty, (q_loads & 1) ^ 1))) break;
    ptx::mbar_arrive_expect_tx(bar(L::bQFull), 2 * L::kTile);
#pragma unroll
    for (int t = 0; t < 2; ++t)
#pragma unroll
      for (int r = 0; r < kRegions; ++r)
        ptx::tma_load_4d(sbase + (t ? L::kQ1 : L::kQ0) + r * L::kRegion, &p.tm_q,
                         bar(L::bQFull), r * 64, item.q_row0 + t * kBlockM, item.h, item.b);
    DIT_TRACE(kTrQIssue, q_loads);
    ++q_loads;
    if (p.stall_kv) return;  // test-only: the consumers' first K wait will expire

    if (!(ok = load(false, item.kv0, item))) break;
    for (int j = 0; ok && j < item.ntiles; ++j) {
      if (j + 1 < item.ntiles && !(ok = load(false, item.kv0 + (j + 1) * kBlockN, item))) break;
      ok = load(true, item.kv0 + j * kBlockN, item);
    }
  }
  if (!ok) {
    raise_abort(p, abort_flag);
    // Let every copy this thread started land before the CTA can exit.
    if (q_loads > 0) ptx::mbar_wait(bar(L::bQFull), (q_loads - 1) & 1, p.wait_limit);
#pragma unroll
    for (int s = 0; s < kStages; ++s)
      if (last_bar[s] >= 0) ptx::mbar_wait(bar(last_bar[s]), last_par[s], p.wait_limit);
  }
}

// Shared-memory matrix descriptors.  The high word (stride byte offset 1024,
// version 1, 128-byte swizzle) is common to every operand; the low word holds the
// start address and the leading byte offset.  Low words are precomputed per buffer
// so that issuing one MMA costs one 32-bit add per operand.
template <int D>
struct Descs {
  static constexpr uint32_t kHi = (1024u >> 4) | (1u << 14) | (2u << 29);
  uint32_t q[2], pp[2], k[kStages], v[kStages];
  __device__ __forceinline__ static uint32_t lo(uint32_t addr, uint32_t lbo) {
    return (addr >> 4) | ((lbo >> 4) << 16);
  }
  __device__ __forceinline__ static uint64_t full(uint32_t lo_word) {
    return (static_cast<uint64_t>(kHi) << 32) | static_cast<uint64_t>(lo_word);
  }
  __device__ __forceinline__ explicit Descs(uint32_t sbase) {
    using L = AttnSmem<D>;
    q[0] = lo(sbase + L::kQ0, 16);
    q[1] = lo(sbase + L::kQ1, 16);
    pp[0] = lo(sbase + L::kP0, 16);
    pp[1] = lo(sbase + L::kP1, 16);
#pragma unroll
    for (int s = 0; s < kStages; ++s) {
      k[s] = lo(sbase + L::kKV + s * L::kTile, 16);          // K-major K tile
      v[s] = lo(sbase + L::kKV + s * L::kTile, L::kRegion);  // MN-major V tile
    }
  }
  __device__ __forceinline__ static uint32_t pick(const uint32_t (&a)[kStages], int slot) {
    uint32_t r = a[0];
#pragma unroll
    for (int s = 1; s < kStages; ++s)
      if (slot == s) r = a[s];
    return r;
  }
};

// S_t = Q_t K^T for every KV tile of every work item (warp kMmaWarp, one thread).
template <int D>
__device__ __forceinline__ void s_issuer(const AttnParams& p, uint32_t sbase, uint32_t tmem,
                                         volatile int* abort_flag) {
  using L = AttnSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBlockM, kBlockN, false, false);
  const Descs<D> ds(sbase);
  // K-major A and B, 16 of D's elements per instruction: the K-step advances 32 bytes
  // inside a 128-byte swizzle column, then moves to the next column.
  auto issue = [&](int t, int slot) {
    const uint32_t kb = Descs<D>::pick(ds.k, slot);
    const uint32_t qa = ds.q[t];
#pragma unroll
    for (int k = 0; k < D / 16; ++k) {
      const uint32_t off = ((k / 4) * L::kRegion + (k % 4) * 32) >> 4;
      ptx::mma_bf16_ss(tmem + t * kBlockN, Descs<D>::full(qa + off), Descs<D>::full(kb + off),
                       kIdesc, k > 0 ? 1u : 0u);
    }
  };
  auto wait = [&](int b, uint32_t parity) {
    return wait_or_abort(bar(b), parity, abort_flag, p.wait_limit);
  };

  uint32_t kpar = 0;  // bit s: parity of the next K_FULL[s] phase
  int g = 0;          // S tiles issued per Q tile (CTA-global)
  int li = 0;         // work items started
  int ring0 = 0;      // ring index of this item's first K/V tile
  bool ok = true;
  for (int w = blockIdx.x; ok && w < p.num_items; w += gridDim.x, ++li) {
    const int n_tiles = item_of(p, w).ntiles;
    if (!(ok = wait(L::bQFull, li & 1))) break;
    DIT_TRACE(kTrQFull, li);
    for (int j = 0; j < n_tiles; ++j, ++g) {
      const int sK = (ring0 + k_item(j)) % kStages;
      ok = wait(L::bKFull + sK, (kpar >> sK) & 1);
      kpar ^= 1u << sK;
      if (!ok) break;
      DIT_TRACE(kTrMmaK, g);
      // S_t(g) overwrites S_t: softmax t must have loaded S_t(g-1).
      if (g > 0 && !(ok = wait(L::bSEmpty + 0, (g - 1) & 1))) break;
      ptx::tc_fence_after();
      issue(0, sK);
      ptx::mma_commit(bar(L::bSFull + 0));
      DIT_TRACE(kTrMmaS0, g);
      if (g > 0 && !(ok = wait(L::bSEmpty + 1, (g - 1) & 1))) break;
      ptx::tc_fence_after();
      issue(1, sK);
      ptx::mma_commit(bar(L::bSFull + 1));
      ptx::mma_commit(bar(L::bKVEmpty + sK));
      DIT_TRACE(kTrMmaS1, g);
    }
    if (ok) ptx::mma_commit(bar(L::bQEmpty));  // Q_0/Q_1 free once these MMAs are done
    ring0 += 2 * n_tiles;
  }
  if (!ok) {
    raise_abort(p, abort_flag);
    // No MMA may still be writing tensor memory when it is released.
    ptx::mma_commit(bar(L::bDrainS));
    ptx::mbar_wait(bar(L::bDrainS), 0, p.wait_limit);
  }
}

// O_t += P_t V_j for every KV tile of every work item (warp kPvWarp, one thread).
template <int D>
__device__ __forceinline__ void pv_issuer(const AttnParams& p, uint32_t sbase, uint32_t tmem,
                                          volatile int* abort_flag) {
  using L = AttnSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  constexpr uint32_t kIdesc = ptx::idesc_bf16_f32(kBlockM, D, false, true);
  const Descs<D> ds(sbase);
  // P K-major, V MN-major (D contiguous); 16 keys (2 KB of V) per instruction.
  auto issue = [&](int t, int slot, bool acc, int half) {
    const uint32_t vb = Descs<D>::pick(ds.v, slot);
    const uint32_t pa = ds.pp[t];
#pragma unroll
    for (int k = half * 4; k < half * 4 + 4; ++k) {
      const uint32_t aoff = ((k / 4) * L::kRegion + (k % 4) * 32) >> 4;
      ptx::mma_bf16_ss(tmem + 2 * kBlockN + t * D, Descs<D>::full(pa + aoff),
                       Descs<D>::full(vb + k * 128), kIdesc, (acc || k > 0) ? 1u : 0u);
    }
  };
  auto wait = [&](int b, uint32_t parity) {
    return wait_or_abort(bar(b), parity, abort_flag, p.wait_limit);
  };

  uint32_t vpar = 0;  // bit s: parity of the next V_FULL[s] phase
  int g = 0;          // PV tiles issued per Q tile (CTA-global)
  int li = 0;
  int ring0 = 0;
  bool ok = true;
  for (int w = blockIdx.x; ok && w < p.num_items; w += gridDim.x, ++li) {
    const int n_tiles = item_of(p, w).ntiles;
    for (int j = 0; j < n_tiles; ++j, ++g) {
      const int sV = (ring0 + v_item(j, n_tiles)) % kStages;
      if (!(ok = wait(L::bPLo + 0, g & 1))) break;
      DIT_TRACE(kTrMmaP0, g);
      ok = wait(L::bVFull + sV, (vpar >> sV) & 1);
      vpar ^= 1u << sV;
      if (!ok) break;
      DIT_TRACE(kTrMmaV, g);
      // The first PV of an item overwrites O_t: the previous item's epilogue must have read it.
      if (j == 0 && li > 0 && !(ok = wait(L::bOEmpty + 0, (li - 1) & 1))) break;
      ptx::tc_fence_after();
      issue(0, sV, j > 0, 0);
      if (!(ok = wait(L::bPFull + 0, g & 1))) break;
      ptx::tc_fence_after();
      issue(0, sV, j > 0, 1);
      ptx::mma_commit(bar(L::bPVDone + 0));
      DIT_TRACE(kTrMmaPv0, g);
      if (!(ok = wait(L::bPLo + 1, g & 1))) break;
      DIT_TRACE(kTrMmaP1, g);
      if (j == 0 && li > 0 && !(ok = wait(L::bOEmpty + 1, (li - 1) & 1))) break;
      ptx::tc_fence_after();
      issue(1, sV, j > 0, 0);
      if (!(ok = wait(L::bPFull + 1, g & 1))) break;
      ptx::tc_fence_after();
      issue(1, sV, j > 0, 1);
      ptx::mma_commit(bar(L::bPVDone + 1));
      ptx::mma_commit(bar(L::bKVEmpty + sV));
      DIT_TRACE(kTrMmaPv1, g);
    }
    ring0 += 2 * n_tiles;
  }
  if (!ok) {
    raise_abort(p, abort_flag);
    ptx::mma_commit(bar(L::bDrainPV));
    ptx::mbar_wait(bar(L::bDrainPV), 0, p.wait_limit);
  }
}

// acc_lo += low bf16 of w, acc_hi += high bf16 of w (exact widening, fp32 add).
__device__ __forceinline__ void add_bf16x2(float& acc_lo, float& acc_hi, uint32_t w) {
  asm("{\n\t.reg .b16 lo, hi;\n\t"
      "mov.b32 {lo, hi}, %2;\n\t"
      "add.rn.f32.bf16 %0, lo, %0;\n\t"
      "add.rn.f32.bf16 %1, hi, %1;\n\t}"
      : "+f"(acc_lo), "+f"(acc_hi)
      : "r"(w));
}

// One butterfly stage of a warp-wide register<->lane transpose: lane bit kLaneBit and bit
// kRegBit of the register index trade meanings (each pair of registers differing in that
// register bit exchanges one value with the lane differing in that lane bit).
template <int kLaneBit, int kRegBit, int N>
__device__ __forceinline__ void swap_lane_reg_bit(uint32_t (&x)[N], int lane) {
  const bool hi = (lane >> kLaneBit) & 1;
#pragma unroll
  for (int i = 0; i < N; ++i) {
    if (i & (1 << kRegBit)) continue;
    const int j = i | (1 << kRegBit);
    const uint32_t send = hi ? x[i] : x[j];
    const uint32_t recv = __shfl_xor_sync(0xffffffffu, send, 1 << kLaneBit);
    x[i] = hi ? recv : x[i];
    x[j] = hi ? x[j] : recv;
  }
}

// 32 bytes to global memory: one 32-byte store when dst is 32-byte aligned, else two 16-byte ones.
__device__ __forceinline__ void st_global_32B(void* dst, bool align32, const uint32_t* a) {
  if (align32) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(dst), "r"(a[0]),
                 "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7])
                 : "memory");
  } else {
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(a[0]), "r"(a[1]),
                 "r"(a[2]), "r"(a[3])
                 : "memory");
    asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(static_cast<char*>(dst) + 16),
                 "r"(a[4]), "r"(a[5]), "r"(a[6]), "r"(a[7])
                 : "memory");
  }
}

// O_t of a finished short work item, drained through the (now idle) P_t buffer: every
// thread loads its row and the tensor-memory buffer is released at once.  The P tile's 32 KB
// hold the whole bf16 tile, or 64 fp32 columns: the rows are normalised and written to P_t
// in the P tile's layout (128-byte-swizzled regions of 128 bytes per row), which is the box
// layout of the output's tensor map, and one thread stores them with TMA stores once all
// rows are in.  An fp32 tile of D = 128 goes in two rounds of 64 columns: the second is
// written once the first round's stores have read P_t.  The stores drain at the SM's store
// rate while the warpgroup goes on; P_t is written again only after they have read it.
template <int D, bool kOutF32>
struct Staging {
  static constexpr int kCols = kOutF32 ? (D < 64 ? D : 64) : D;  // columns per round
  static constexpr int kRounds = D / kCols;
  static constexpr int kBoxCols = kOutF32 ? 32 : 64;               // 128 bytes per row
  static constexpr int kBoxes = kCols / kBoxCols;                  // boxes per round
};

// All of O_t into registers (o[c] = columns 32c..32c+31 of this thread's row), then O_t
// released to the next item's first PV.
template <int D>
__device__ __forceinline__ void load_o_release(uint32_t tO, uint32_t o_empty_bar,
                                               uint32_t (&o)[D / 32][32]) {
  ptx::tc_fence_after();
#pragma unroll
  for (int c = 0; c < D / 32; ++c) ptx::tmem_ld32(tO + c * 32, o[c]);
  ptx::tmem_wait_ld();
  ptx::tc_fence_before();
  ptx::mbar_arrive(o_empty_bar);
}

// Round `round` of the staging: columns [round * kCols, (round + 1) * kCols) of row r,
// scaled by inv_l, into P_t; then the generic-proxy writes are made visible to the TMA.
template <int D, bool kOutF32, int kRound>
__device__ __forceinline__ void stage_o(const uint32_t (&o)[D / 32][32], uint32_t sP, int r,
                                        float inv_l) {
  using L = AttnSmem<D>;
  using S = Staging<D, kOutF32>;
  const uint32_t sw = static_cast<uint32_t>(r & 7);
  constexpr int kPerChunk = kOutF32 ? 4 : 8;  // elements per 16-byte chunk
  constexpr int kCol0 = kRound * S::kCols;
#pragma unroll
  for (int ch = 0; ch < S::kCols / kPerChunk; ++ch) {
    const uint32_t* x = &o[(kCol0 + ch * kPerChunk) / 32][(kCol0 + ch * kPerChunk) % 32];
    uint32_t wv[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      if constexpr (kOutF32)
        wv[q] = __float_as_uint(__uint_as_float(x[q]) * inv_l);
      else
        wv[q] = ptx::pack_bf16x2(__uint_as_float(x[2 * q]) * inv_l,
                                 __uint_as_float(x[2 * q + 1]) * inv_l);
    }
    const uint32_t addr =
        sP + (ch / 8) * L::kRegion + r * 128 + ((static_cast<uint32_t>(ch % 8) ^ sw) << 4);
    asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(wv[0]), "r"(wv[1]),
                 "r"(wv[2]), "r"(wv[3])
                 : "memory");
  }
  ptx::fence_proxy_async_smem();
}

template <int D, bool kOutF32, bool kAccum, bool kLse, bool kSoftDrain>
__device__ __forceinline__ void softmax_wg(const AttnParams& p, uint32_t sbase, uint32_t tmem,
                                           int t, int warp, int lane,
                                           volatile int* abort_flag) {
  using L = AttnSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;  // row in the Q tile == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const uint32_t tS = tmem + t * kBlockN + lane_off;
  const uint32_t tO = tmem + 2 * kBlockN + t * D + lane_off;
  const uint32_t sP = sbase + (t ? L::kP1 : L::kP0);
  const uint32_t sw = static_cast<uint32_t>(r & 7);
  const float c = p.scale_log2;
  float* const hand = reinterpret_cast<float*>(__cvta_shared_to_generic(sbase + L::kInvLp));
  // Warp-uniform bounded wait.
  auto wait = [&](int b, uint32_t parity) {
    const bool ok = wait_or_abort(bar(b), parity, abort_flag, p.wait_limit);
    return __all_sync(0xffffffffu, ok);
  };

  int g = 0;   // tiles processed by this warpgroup (CTA-global)
  int li = 0;  // work items processed
  bool ok = true;
  for (int w = blockIdx.x; ok && w < p.num_items; w += gridDim.x, ++li) {
    // Only the key range is live across the tile loop; the rest of the item is
    // recomputed at its end.
    int ntiles, kv_left;  // tiles of the item, keys in its range
    {
      const Item it = item_of(p, w);
      ntiles = it.ntiles;
      kv_left = it.kv_len;
    }
    float m = -INFINITY;  // running max of scale*log2e*s (possibly stale by < 2^8)
    float l = 0.f;        // running sum of 2^(c*s - m), for the LSE
    float lp = 0.f;       // running sum of the bf16-rounded P the PV GEMM sees, for O
    for (int j = 0; j < ntiles; ++j, ++g) {
      if (!(ok = wait(L::bSFull + t, g & 1))) break;
      if (r == 0) DIT_TRACE(kTrSmFull0 + 5 * t, g);
      if (r == 0 && t == 0 && g == 0) DIT_TRACE(kTrCta, 1);
      ptx::tc_fence_after();

      // Scores into registers; the load-with-reduction form returns each 32-column
      // chunk's max as well, so a full tile's row max costs two extra instructions.
      float s[kBlockN];
      float cmax[kBlockN / 32];
#pragma unroll
      for (int cc = 0; cc < kBlockN / 32; ++cc) {
        uint32_t u[32];
        ptx::tmem_ld32_max(tS + cc * 32, u, cmax[cc]);
#pragma unroll
        for (int i = 0; i < 32; ++i) s[cc * 32 + i] = __uint_as_float(u[i]);
      }
      ptx::tmem_wait_ld();
      // S_t is in registers: the S issuer may overwrite it with the next tile.
      ptx::tc_fence_before();
      ptx::mbar_arrive(bar(L::bSEmpty + t));
      if (r == 0) DIT_TRACE(kTrSmLd0 + 5 * t, g);

      float mx = ptx::fmax3(cmax[0], cmax[1], fmaxf(cmax[2], cmax[3]));
      const int valid = kv_left - j * kBlockN;
      if (valid < kBlockN) {
        // Ragged last tile: keys past the item's range (zero-filled rows past n_kv, or the
        // next range's rows) are masked to -inf, so their P is exactly 0, and the max is
        // taken over the valid columns only.
#pragma unroll
        for (int i = 0; i < kBlockN; ++i)
          if (i >= valid) s[i] = -INFINITY;
        float a[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          a[q] = ptx::fmax3(s[16 * q], s[16 * q + 1], s[16 * q + 2]);
#pragma unroll
          for (int i = 3; i < 15; i += 2) a[q] = ptx::fmax3(a[q], s[16 * q + i], s[16 * q + i + 1]);
          a[q] = fmaxf(a[q], s[16 * q + 15]);
        }
        mx = ptx::fmax3(ptx::fmax3(a[0], a[1], a[2]), ptx::fmax3(a[3], a[4], a[5]),
                        fmaxf(a[6], a[7]));
      }
      if (r == 0) DIT_TRACE(kTrSmMax0 + 5 * t, g);
      const float m_tile = mx * c;
      const bool raise = m_tile > m + kRescaleLog2;  // always true on an item's first tile
      float alpha = 1.f;
      if (raise) {
        alpha = ptx::ex2_approx(m - m_tile);  // 0 on the first tile (m = -inf)
        m = m_tile;
      }
      l *= alpha;
      lp *= alpha;
      bool pv_prev_done = (g == 0);  // no earlier PV has read P_t
      if (j > 0 && __any_sync(0xffffffffu, raise)) {
        // O_t may only be touched once PV_t(g-1) has landed.
        if (!(ok = wait(L::bPVDone + t, (g - 1) & 1))) break;
        pv_prev_done = true;
        ptx::tc_fence_after();
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

      // P = 2^(c*s - m), two elements per packed FMA, written in two halves (keys 0-63,
      // 64-127: one 128-byte-swizzled K-major region each) so that the PV GEMM can start
      // on the first while the second is computed.
      const uint64_t c2 = ptx::f2pack(c, c);
      const uint64_t nm2 = ptx::f2pack(-m, -m);
      uint64_t acc_l[4];
      float acc_lp[8];
#pragma unroll
      for (int q = 0; q < 4; ++q) acc_l[q] = 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) acc_lp[q] = 0.f;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
#pragma unroll
        for (int i = half * 64; i < half * 64 + 64; i += 2) {
          float x0, x1;
          ptx::f2unpack(ptx::ffma2(ptx::f2pack(s[i], s[i + 1]), c2, nm2), x0, x1);
          s[i] = ptx::ex2_approx(x0);
          s[i + 1] = ptx::ex2_approx(x1);
        }
        if (half == 0) {
          if (r == 0) DIT_TRACE(kTrSmExp0 + 5 * t, g);
          // The P_t buffer is free once PV_t(g-1) has read it.
          if (!pv_prev_done && !(ok = wait(L::bPVDone + t, (g - 1) & 1))) break;
          if constexpr (kSoftDrain) {
            // ... and, at an item's first tile, once the previous item's staged O has been
            // read out of it by the TMA stores.
            if (j == 0 && li > 0) {
              if (r == 0) {
                ptx::bulk_wait_read_all();
                ptx::mbar_arrive(bar(L::bStageFree + t));
              }
              if (!(ok = wait(L::bStageFree + t,
                              Staging<D, kOutF32>::kRounds == 2 ? 1 : (li - 1) & 1)))
                break;
            }
          }
        }
        // Pack to bf16 and store row r of this half's swizzled region; accumulate the row
        // sums (unrounded for the LSE, bf16-rounded for O) in independent chains.
#pragma unroll
        for (int ch = half * 8; ch < half * 8 + 8; ++ch) {
          uint32_t wv[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float p0 = s[8 * ch + 2 * q], p1 = s[8 * ch + 2 * q + 1];
            wv[q] = ptx::pack_bf16x2(p0, p1);
            if constexpr (kLse) acc_l[q] = ptx::fadd2(acc_l[q], ptx::f2pack(p0, p1));
            add_bf16x2(acc_lp[2 * q], acc_lp[2 * q + 1], wv[q]);
          }
          const uint32_t addr = sP + half * L::kRegion + r * 128 +
                                ((static_cast<uint32_t>(ch % 8) ^ sw) << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(wv[0]),
                       "r"(wv[1]), "r"(wv[2]), "r"(wv[3])
                       : "memory");
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        ptx::mbar_arrive(bar(half == 0 ? L::bPLo + t : L::bPFull + t));
      }
      if (!ok) break;
      if (r == 0) DIT_TRACE(kTrSmArrive0 + 5 * t, g);
      {
        if constexpr (kLse) {
          const uint64_t sl =
              ptx::fadd2(ptx::fadd2(acc_l[0], acc_l[1]), ptx::fadd2(acc_l[2], acc_l[3]));
          float a0, a1;
          ptx::f2unpack(sl, a0, a1);
          l += a0 + a1;
        }
        lp += ((acc_lp[0] + acc_lp[1]) + (acc_lp[2] + acc_lp[3])) +
              ((acc_lp[4] + acc_lp[5]) + (acc_lp[6] + acc_lp[7]));
      }
    }
    if (!ok) break;

    // Hand the row's scale factors to the epilogue warpgroup and write the LSE.  O is
    // normalised by the sum of the rounded weights it was built from, so the weights
    // sum to one; the LSE uses the unrounded sum.
    constexpr float kLn2 = 0.69314718055994530942f;
    const float lse2 = m + log2f(l);  // this pass's LSE in log2 units
    const Item item = item_of(p, w);
    const int row = item.q_row0 + t * kBlockM + r;
    float* const lse_row = p.lse + item.lse_off(p) + row;
    if constexpr (kSoftDrain) {
      // Short items: this warpgroup drains its own O_t once the item's last PV has landed
      // (through P_t: load_o_release, stage_o), instead of handing it to the epilogue
      // warpgroup.
      if constexpr (kLse) {
        if (row < p.n_q) *lse_row = lse2 * kLn2;
      } else {
        (void)lse_row;
        (void)lse2;
      }
      if (!(ok = wait(L::bPVDone + t, (g - 1) & 1))) break;
      if constexpr (kSoftDrain) {
        using S = Staging<D, kOutF32>;
        const float inv_l = 1.f / lp;
        uint32_t o[D / 32][32];
        load_o_release<D>(tO, bar(L::bOEmpty + t), o);
        // STAGED completes once per round.  STAGE_FREE completes before the next item's first
        // P write and, with two rounds, also between them (once round 0's stores have read
        // P_t).  With two rounds both complete twice per item, so the parity of each wait is
        // fixed: 0 for the first completion, 1 for the second.
        auto stage_and_store = [&](auto round_tag) -> bool {
          constexpr int kRound = decltype(round_tag)::value;
          stage_o<D, kOutF32, kRound>(o, sP, r, inv_l);
          ptx::mbar_arrive(bar(L::bStaged + t));
          if (quarter == 0) {
            // All 128 rows staged: one thread stores them (rows past n_q are clipped).
            if (!wait(L::bStaged + t, S::kRounds == 2 ? kRound : (li & 1))) return false;
            if (lane == 0) {
#pragma unroll
              for (int rg = 0; rg < S::kBoxes; ++rg)
                ptx::tma_store_5d(&p.tm_o, sP + rg * L::kRegion, kRound * S::kCols + rg * S::kBoxCols,
                                  item.q_row0 + t * kBlockM, item.h, item.b, item.split);
              ptx::bulk_commit();
            }
          }
          return true;
        };
        if (!(ok = stage_and_store(std::integral_constant<int, 0>{}))) break;
        if constexpr (S::kRounds == 2) {
          // P_t takes the second half once the first half's stores have read it.
          if (r == 0) {
            ptx::bulk_wait_read_all();
            ptx::mbar_arrive(bar(L::bStageFree + t));
          }
          if (!(ok = wait(L::bStageFree + t, 0))) break;
          if (!(ok = stage_and_store(std::integral_constant<int, 1>{}))) break;
        }
      }
    } else if constexpr (!kAccum) {
      // Slot [t][r] = 1 / lp, reused once the epilogue has taken the previous item's value.
      if (li > 0 && !(ok = wait(L::bEpiTaken + t, (li - 1) & 1))) break;
      hand[t * kBlockM + r] = 1.f / lp;
      ptx::mbar_arrive(bar(L::bEpiReady + t));
      if constexpr (kLse) {
        if (row < p.n_q) *lse_row = lse2 * kLn2;
      } else {
        (void)lse_row;
        (void)lse2;
      }
    } else {
      // Accumulate mode: the epilogue merges this pass into the running (O, lse); it gets
      // (this pass's LSE in log2 units, 1 / lp) through one slot [r][2] shared by both Q
      // tiles, filled in the order tile 0, tile 1 of each item.
      (void)lse_row;
      if (t == 0) {
        if (li > 0 && !(ok = wait(L::bEpiTaken + 1, (li - 1) & 1))) break;
      } else if (!(ok = wait(L::bEpiTaken + 0, li & 1))) {
        break;
      }
      hand[2 * r] = lse2;
      hand[2 * r + 1] = 1.f / lp;
      ptx::mbar_arrive(bar(L::bEpiReady + t));
    }
  }
  if (!ok) raise_abort(p, abort_flag);
  if constexpr (kSoftDrain) {
    if (r == 0) ptx::bulk_wait_all();  // the last staged stores complete before the CTA exits
  }
}

// Epilogue warpgroup (warps 12-15): for each work item and Q tile t, waits for the
// softmax's normaliser and the tile's last PV, reads O_t out of tensor memory (then
// releases it to the next item's PV), scales it and stores it.  Off the softmax's
// critical path: the softmax warpgroups go straight on to the next item.
//
// TMEM hands each thread one row.  For fp32 output two butterfly stages (warp shuffles)
// trade lane bits 4,3 (row) with register bits 4,3 (column) of each 32-column chunk, so
// that one warp store covers 8 rows x 128 contiguous bytes rather than 32 rows x 32
// bytes: a quarter of the L1 wavefronts per byte, which keeps the burst of O stores at an
// item boundary from holding up the softmax's shared-memory P writes.  bf16 rows are
// stored from the row-per-thread layout (64 bytes per row per 32 columns), which measured
// faster there.
template <int D, bool kOutF32, bool kAccum>
__device__ __forceinline__ void epilogue_wg(const AttnParams& p, uint32_t sbase, uint32_t tmem,
                                            int warp, int lane,
                                            volatile int* abort_flag) {
  static_assert(kOutF32 || !kAccum, "the running output is fp32");
  using L = AttnSmem<D>;
  auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
  const int quarter = warp & 3;
  const int r = quarter * 32 + lane;  // row in the Q tile == TMEM lane
  const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
  const float* hand = reinterpret_cast<const float*>(__cvta_shared_to_generic(sbase + L::kInvLp));
  const int r_lo = lane & 7, cgrp = lane >> 3;  // fp32 store layout after the transpose
  auto wait = [&](int b, uint32_t parity) {
    const bool ok = wait_or_abort(bar(b), parity, abort_flag, p.wait_limit);
    return __all_sync(0xffffffffu, ok);
  };

  int li = 0;
  int g_end = 0;  // KV tiles of the items so far (CTA-global)
  bool ok = true;
  for (int w = blockIdx.x; ok && w < p.num_items; w += gridDim.x, ++li) {
    const Item item = item_of(p, w);
    g_end += item.ntiles;
    const int g_last = g_end - 1;  // CTA-global index of the item's last tile
    const size_t head_row0 = item.lse_off(p);  // LSE rows
    const size_t out_off = item.out_off(p);                           // output head
    // Accumulate mode: this item's running LSEs (read now, long before they are needed)
    // and its running-output rows brought into L2 while the item runs.
    float lse_run0 = -INFINITY, lse_run1 = -INFINITY;
    if constexpr (kAccum) {
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        const int row = item.q_row0 + t * kBlockM + r;
        if (row < p.n_q) {
          (t ? lse_run1 : lse_run0) = ptx::ld_global_f32(p.lse + head_row0 + row);
#pragma unroll
          for (int q = 0; q < D / 32; ++q) ptx::prefetch_l2(p.out_f32 + out_off + row * p.o_sn + q * 32);
        }
      }
    }
    for (int t = 0; t < 2; ++t) {
      if (!(ok = wait(L::bEpiReady + t, li & 1))) break;
      // Scale of this row's O accumulator, and in accumulate mode the weight of the
      // running output.
      float inv_l, w_run = 0.f;
      if constexpr (!kAccum) {
        inv_l = hand[t * kBlockM + r];
        ptx::mbar_arrive(bar(L::bEpiTaken + t));
      } else {
        const float lse2 = hand[2 * r], inv_lp = hand[2 * r + 1];
        ptx::mbar_arrive(bar(L::bEpiTaken + t));
        // Merge into the running (O, lse) exactly as one ring hop does:
        //   lse' = M + ln(e^(lse_run - M) + e^(lse_c - M)),  M = max(lse_run, lse_c),
        //   O'   = e^(lse_run - lse') O_run + e^(lse_c - lse') O_c.
        // A running LSE of -inf is an empty row: weight 0, its O_run is never read.
        const float run2 = (t ? lse_run1 : lse_run0) * 1.4426950408889634f;
        const float mx2 = fmaxf(run2, lse2);
        const float a = ptx::ex2_approx(run2 - mx2);
        const float b = ptx::ex2_approx(lse2 - mx2);
        const float sum = a + b;
        w_run = a / sum;
        inv_l = (b / sum) * inv_lp;
        const int row = item.q_row0 + t * kBlockM + r;
        if (row < p.n_q) p.lse[head_row0 + row] = (mx2 + log2f(sum)) * 0.69314718055994530942f;
      }
      const int row0w = item.q_row0 + t * kBlockM + quarter * 32;  // first row of this warp
      const int row = row0w + lane;
      // Accumulate mode: the next 16-column piece of this thread's own row of the running
      // output is in flight while the current one is processed; rows of weight 0 (empty)
      // or past n_q are not read (their o stays 0).
      const bool use_run = kAccum && row < p.n_q && w_run != 0.f;
      const float* const run_row = p.out_f32 + out_off + row * p.o_sn;
      uint32_t o[16];
      auto load_run = [&](int k) {
        if constexpr (kAccum) {
#pragma unroll
          for (int q = 0; q < 2; ++q) {
            ptx::U32x8 u{};
            if (use_run) u = ptx::ld_global_32B(run_row + k * 16 + q * 8, p.out_align32);
#pragma unroll
            for (int i = 0; i < 8; ++i) o[q * 8 + i] = u.v[i];
          }
        }
      };
      load_run(0);  // in flight while the last PV finishes
      if (!(ok = wait(L::bPVDone + t, g_last & 1))) break;
      ptx::tc_fence_after();
      if (r == 0 && t == 0) DIT_TRACE(kTrCta, 2 + 2 * li);
      const uint32_t tO = tmem + 2 * kBlockN + t * D + lane_off;
      auto release_if = [&](bool last) {
        if (last) {  // O_t has been read: the PV issuer may start the next item's O_t.
          ptx::tc_fence_before();
          ptx::mbar_arrive(bar(L::bOEmpty + t));
        }
      };
      if constexpr (kOutF32 && !kAccum) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t x[32];
          ptx::tmem_ld32(tO + c * 32, x);
          ptx::tmem_wait_ld();
          release_if(c == D / 32 - 1);
#pragma unroll
          for (int i = 0; i < 32; ++i) x[i] = __float_as_uint(__uint_as_float(x[i]) * inv_l);
          swap_lane_reg_bit<4, 4>(x, lane);
          swap_lane_reg_bit<3, 3>(x, lane);
          // x[8*rr + i] = (row row0w + 8*rr + r_lo, column 32*c + 8*cgrp + i)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const int row_k = row0w + rr * 8 + r_lo;
            if (row_k < p.n_q)
              st_global_32B(p.out_f32 + out_off + row_k * p.o_sn + c * 32 + cgrp * 8, p.out_align32,
                            &x[rr * 8]);
          }
        }
      } else if constexpr (kAccum) {
        // 16-column steps: O' = (1/lp)(w_c) O_acc + w_run O_run on the own row, then the
        // transpose (lane bits 4,3 <-> register bits 3,2) and 8-row x 64-byte stores.
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          uint32_t x[16];
          ptx::tmem_ld16(tO + k * 16, x);
          ptx::tmem_wait_ld();
          release_if(k == D / 16 - 1);
#pragma unroll
          for (int i = 0; i < 16; ++i)
            x[i] = __float_as_uint(fmaf(w_run, __uint_as_float(o[i]), __uint_as_float(x[i]) * inv_l));
          if (k + 1 < D / 16) load_run(k + 1);
          swap_lane_reg_bit<4, 3>(x, lane);
          swap_lane_reg_bit<3, 2>(x, lane);
          // x[4*rr + i] = (row row0w + 8*rr + r_lo, column 16*k + 4*cgrp + i)
#pragma unroll
          for (int rr = 0; rr < 4; ++rr) {
            const int row_k = row0w + rr * 8 + r_lo;
            if (row_k < p.n_q) {
              float* dst = p.out_f32 + out_off + row_k * p.o_sn + k * 16 + cgrp * 4;
              asm volatile("st.global.v4.b32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(x[rr * 4]),
                           "r"(x[rr * 4 + 1]), "r"(x[rr * 4 + 2]), "r"(x[rr * 4 + 3])
                           : "memory");
            }
          }
        }
      } else {
        __nv_bfloat16* dst = p.out_bf16 + out_off + row * p.o_sn;
#pragma unroll
        for (int half = 0; half < D / 64; ++half) {
          uint32_t wd[32];  // 64 columns of this thread's row as bf16 pairs
#pragma unroll
          for (int c = 0; c < 2; ++c) {
            uint32_t a[32];
            ptx::tmem_ld32(tO + half * 64 + c * 32, a);
            ptx::tmem_wait_ld();
            release_if(half == D / 64 - 1 && c == 1);
#pragma unroll
            for (int i = 0; i < 16; ++i)
              wd[c * 16 + i] = ptx::pack_bf16x2(__uint_as_float(a[2 * i]) * inv_l,
                                                __uint_as_float(a[2 * i + 1]) * inv_l);
          }
          if (row < p.n_q) {
#pragma unroll
            for (int i = 0; i < 32; i += 8)
              st_global_32B(dst + half * 64 + 2 * i, p.out_align32, &wd[i]);
          }
        }
      }
      if (r == 0 && t == 0) DIT_TRACE(kTrCta, 3 + 2 * li);
    }
  }
  if (!ok) raise_abort(p, abort_flag);
}

}  // namespace detail

// kLse = false: no LSE output (p.lse unused) and no unrounded row sum; O is unchanged.
// kSoftDrain: the softmax warpgroups drain O themselves (for work items of few KV tiles, where
// an item's drain would otherwise wait for the epilogue warpgroup's turn at every item).
template <int D, bool kOutF32, bool kAccum, bool kLse = true, bool kSoftDrain = false>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  static_assert(kLse || !kAccum, "the running merge needs the LSE");
  static_assert(!(kSoftDrain && kAccum), "the running merge runs in the epilogue warpgroup");
  using L = AttnSmem<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  const uint32_t sbase = ptx::smem_addr(smem);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbort);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  if (threadIdx.x == 0) {
    auto bar = [&](int i) { return sbase + L::kBars + 8u * i; };
    ptx::mbar_init(bar(L::bQFull), 1);
    ptx::mbar_init(bar(L::bQEmpty), 1);
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(bar(L::bKFull + s), 1);
      ptx::mbar_init(bar(L::bVFull + s), 1);
      ptx::mbar_init(bar(L::bKVEmpty + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      ptx::mbar_init(bar(L::bSFull + t), 1);
      ptx::mbar_init(bar(L::bSEmpty + t), kBlockM);
      ptx::mbar_init(bar(L::bPFull + t), kBlockM);
      ptx::mbar_init(bar(L::bPLo + t), kBlockM);
      ptx::mbar_init(bar(L::bPVDone + t), 1);
      ptx::mbar_init(bar(L::bOEmpty + t), kBlockM);
      ptx::mbar_init(bar(L::bEpiReady + t), kBlockM);
      ptx::mbar_init(bar(L::bEpiTaken + t), kBlockM);
      ptx::mbar_init(bar(L::bStaged + t), kBlockM);
      ptx::mbar_init(bar(L::bStageFree + t), 1);
    }
    ptx::mbar_init(bar(L::bDrainS), 1);
    ptx::mbar_init(bar(L::bDrainPV), 1);
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
  if (threadIdx.x == 0) DIT_TRACE(kTrCta, 0);

  using Regs = RegSplit<kSoftDrain>;
  if (warp < kLoadWarp) {
    ptx::setmaxnreg_inc<Regs::kSoftmax>();
    detail::softmax_wg<D, kOutF32, kAccum, kLse, kSoftDrain>(p, sbase, tmem, warp >> 2, warp, lane,
                                                              abort_flag);
  } else if (warp < kEpiWarp0) {
    ptx::setmaxnreg_dec<Regs::kIssue>();
    if (warp == kLoadWarp) {
      if (lane == 0) detail::producer<D>(p, sbase, abort_flag);
    } else if (warp == kMmaWarp) {
      if (lane == 0) detail::s_issuer<D>(p, sbase, tmem, abort_flag);
    } else if (warp == kPvWarp) {
      if (lane == 0) detail::pv_issuer<D>(p, sbase, tmem, abort_flag);
    }
    __syncwarp();
  } else {
    ptx::setmaxnreg_dec<Regs::kEpilogue>();
    if constexpr (!kSoftDrain)
      detail::epilogue_wg<D, kOutF32, kAccum>(p, sbase, tmem, warp, lane, abort_flag);
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, 512);
  }
  if (threadIdx.x == 0) DIT_TRACE(kTrCta, 63);
}

}  // namespace ditattn
