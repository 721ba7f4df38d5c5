/*
 * ditattn — non-causal DiT self-attention on GB300 (sm_103a), C ABI.
 *
 * The library computes O = softmax(scale * Q K^T) V per (batch, head) over
 * long token sequences, either in one fused pass or as p KV chunks whose
 * partial outputs and log-sum-exps are merged exactly as one Ring-attention
 * hop merges them: by a separate merge of the p stacked partials, or hop by
 * hop into a running output inside each chunk pass.  On one GPU the p chunks
 * are virtual ranks: a "hop" is a pointer to the next chunk, with no
 * communication.
 *
 * Conventions shared by every entry point:
 *  - Tensors are plain device pointers, contiguous row-major [B, H, N, D]
 *    ("BHND"), except where a head stride is passed explicitly.  Q, K, V are
 *    bf16 (IEEE binary16-brain, 2 bytes).  LSE buffers are fp32 [B, H, N].
 *  - lse is the NATURAL log of sum_j exp(scale * q_i . k_j) over the keys the
 *    call covers (the kernels work in base 2 internally and convert).
 *  - The caller owns every buffer.  The library calls no device allocator.
 *    Besides a cache of host-side TMA-descriptor encoders it holds two
 *    fixed device arrays in its own module: one status word, and the 128 MiB
 *    scratch array of dit_attn_chunk_fwd_splitkv_noalloc.  The CUDA runtime
 *    reserves them on a device when it loads the library's device code there:
 *    on the first call that uses that device under the default lazy module
 *    loading, or when the library is loaded under CUDA_MODULE_LOADING=EAGER.
 *    On a device too full to take them, that first call fails with
 *    DIT_ERR_CUDA.  Device addresses are looked up once per device number and
 *    assume the runtime's primary context (no cudaDeviceReset in between).
 *  - Calls are asynchronous on `stream` (0 = legacy default stream).  Argument
 *    errors are returned before anything is launched.  A launch failure
 *    returns DIT_ERR_CUDA.  Device-side timeouts (a bounded wait that
 *    expired) are recorded in the status word and reported by
 *    dit_attn_check(), which synchronises the stream.
 *  - Validation (before launch): B, H, N, n_kv, p >= 1; D in {64, 128} (else
 *    DIT_ERR_UNSUPPORTED); pointers non-null; q, k, v, out, partials 16-byte
 *    aligned; lse buffers 4-byte aligned; scale finite and > 0; outputs must
 *    not overlap inputs; sizes must fit the kernels' 32-bit tile coordinates
 *    (N < 2^31, B*H < 2^31).
 */
#ifndef DITATTN_H
#define DITATTN_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  DIT_OK = 0,
  DIT_ERR_INVALID_ARG = 1,  /* bad pointer, size, alignment, aliasing or scale */
  DIT_ERR_UNSUPPORTED = 2,  /* valid request the kernels do not implement (e.g. D = 96) */
  DIT_ERR_CUDA = 3,         /* a CUDA runtime/driver call failed */
  DIT_ERR_TIMEOUT = 4       /* a kernel's bounded wait expired (reported by dit_attn_check) */
} dit_status;

typedef enum { DIT_F32 = 0, DIT_BF16 = 1 } dit_dtype;

/* Opaque CUDA stream (cudaStream_t / CUstream). */
typedef void* dit_stream;

/* Element strides of a logical [B, H, N, D] view whose last dimension is
 * contiguous: with s = the strides, element (i_b, i_h, i_n, i_d) sits
 * i_b*s.b + i_h*s.h + i_n*s.n + i_d elements from the base.  Contiguous BHND
 * is {H*N*D, N*D, D}; the token-major BSND layout ([B, N, H, D] in memory) is
 * {N*H*D, D, H*D}. */
typedef struct {
  long long b, h, n;
} dit_strides;

/*
 * Fused attention over all N keys.
 * Defines: per head, s_ij = scale * q_i . k_j; o_i = sum_j softmax_j(s_ij) v_j;
 * every query sees every key (non-causal).  Pages: MindIE-SD parallelism docs,
 * "Ring Sequence Parallel" usage example (local attention = softmax of the
 * scaled scores times V); arganzheng.life multi-GPU diffusion parallelism,
 * section 4.1 Ulysses (full attention per head over all N tokens).
 *   q, k, v : device bf16 [B, H, N, D], contiguous, 16-byte aligned (read only)
 *   out     : device [B, H, N, D] of out_dtype (written)
 *   lse     : device fp32 [B, H, N] (written), or NULL when the caller needs only O:
 *             the pass then skips the LSE and its unrounded row sum (O is the same)
 *   scale   : score scale, usually 1/sqrt(D)
 */
dit_status dit_attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                        int B, int H, int N, int D, float scale, dit_dtype out_dtype,
                        dit_stream stream);

/*
 * Attention of all N_q queries against ONE KV chunk: keys/values rows
 * [0, n_kv) starting at k, v (pass pointers already offset to the chunk's
 * first row).  This is one round of Ring attention: round i of rank r uses
 * the K/V block of rank (r + i) mod p, and after p rounds every query has
 * seen every key (arganzheng.life, section 4.2 Ring).
 *   q              : device bf16 [B, H, N_q, D], contiguous
 *   k, v           : device bf16; head (b*H + h) starts kv_head_stride
 *                    elements after the previous one, rows are D elements
 *                    apart.  N*D for a view into full [B,H,N,D] tensors,
 *                    n_kv*D for a packed chunk buffer as a ring hop would
 *                    receive it.  kv_head_stride must be >= n_kv*D and a
 *                    multiple of 8 (16-byte TMA stride).
 *   out_partial    : device [B, H, N_q, D] of partial_dtype: the softmax-
 *                    normalised output over this chunk's keys
 *   lse_partial    : device fp32 [B, H, N_q]: natural log-sum-exp over this chunk
 */
dit_status dit_attn_chunk_fwd(const void* q, const void* k, const void* v, void* out_partial,
                              float* lse_partial, int B, int H, int N_q, int n_kv, int D,
                              long long kv_head_stride, float scale, dit_dtype partial_dtype,
                              dit_stream stream);

/*
 * All virtual ranks of the ring decomposition in one launch: for each of p key
 * chunks c = [chunk_starts[c], chunk_starts[c+1]) of k / v, the partial output and
 * LSE of all N_q queries against that chunk alone, exactly as dit_attn_chunk_fwd
 * defines them (a Ring round's local attention on the block a rank holds;
 * arganzheng.life, section 4.2 Ring: one KV block per round, combined by online
 * softmax).  Bitwise equal to p dit_attn_chunk_fwd calls on the chunk views; one
 * persistent launch has no per-chunk launch gaps or tails.  dit_attn_lse_merge
 * then combines the partials.
 *   q, k, v, B, H, N_q, n_kv, D, kv_head_stride, scale : as dit_attn_chunk_fwd,
 *                  k / v holding all n_kv key rows
 *   partials     : device [p, B, H, N_q, D] of partial_dtype, contiguous, 16-byte
 *                  aligned (written)
 *   lses         : device fp32 [p, B, H, N_q], contiguous (written)
 *   p            : 1 .. 64
 *   chunk_starts : HOST array of p + 1 key-row offsets, 0 <= chunk_starts[0] <
 *                  chunk_starts[1] < ... < chunk_starts[p] <= n_kv (read before the
 *                  call returns; the chunks need not cover all keys)
 * partials and lses must not overlap each other or q, k, v (DIT_ERR_INVALID_ARG).
 */
dit_status dit_attn_chunks_fwd(const void* q, const void* k, const void* v, void* partials,
                               float* lses, int B, int H, int N_q, int n_kv, int D,
                               long long kv_head_stride, int p, const int* chunk_starts,
                               float scale, dit_dtype partial_dtype, dit_stream stream);

/*
 * General-layout form of dit_attn_fwd / dit_attn_chunk_fwd: attention of N_q
 * queries against n_kv keys, each of q, k, v and out an arbitrary strided
 * [B, H, N, D] view (last dimension contiguous).  This reads and writes the
 * token-major BSND layout in which the pages' sequence-parallel code keeps its
 * activations (the MindIE-SD parallelism docs run their attention kernel on
 * BSND tensors; valdrada.cn Wan2.2, CP section: tokens are split across ranks
 * and heads kept whole) directly, with no transpose.
 *   q, k, v     : device bf16 views; NULL strides = contiguous BHND
 *   out         : device view of out_dtype (written); NULL strides = contiguous
 *   lse         : device fp32 [B, H, N_q], contiguous (written), or NULL (no LSE,
 *                 as for dit_attn_fwd)
 * Strides must be positive multiples of 8 elements (16-byte TMA strides) below
 * 2^39; out must not map two elements to one address; out and lse must not
 * overlap the address range of q, k or v (DIT_ERR_INVALID_ARG otherwise).
 */
dit_status dit_attn_fwd_strided(const void* q, const dit_strides* q_strides, const void* k,
                                const dit_strides* k_strides, const void* v,
                                const dit_strides* v_strides, void* out,
                                const dit_strides* out_strides, float* lse, int B, int H, int N_q,
                                int n_kv, int D, float scale, dit_dtype out_dtype,
                                dit_stream stream);

/*
 * One Ring-attention hop with the merge fused into the chunk pass: the attention
 * of all N_q queries against ONE KV chunk, (O_c, lse_c) exactly as
 * dit_attn_chunk_fwd defines them, is merged in place into a running output:
 *   M = max(lse_run, lse_c);  lse' = M + ln(exp(lse_run - M) + exp(lse_c - M));
 *   O' = exp(lse_run - lse') O_run + exp(lse_c - lse') O_c
 * which is the online-softmax accumulation a Ring round performs on the block it
 * receives (arganzheng.life, section 4.2 Ring).  Applying it once per chunk of
 * the keys, in any order, gives the full attention.  No stacked partials and no
 * separate merge pass.
 *   q, k, v, B, H, N_q, n_kv, D, kv_head_stride, scale : as dit_attn_chunk_fwd
 *   o_run   : device fp32 [B, H, N_q, D], 16-byte aligned (read and written)
 *   lse_run : device fp32 [B, H, N_q], 4-byte aligned (read and written)
 * A row whose lse_run is -inf is empty: its o_run is never read (it may hold
 * anything, NaN included) and the row becomes this chunk's own attention.  So a
 * running state starts either as lse_run = -inf everywhere (o_run
 * uninitialised) or as the fp32 output of dit_attn_chunk_fwd for the first
 * chunk.  o_run and lse_run must not overlap each other or q, k, v
 * (DIT_ERR_INVALID_ARG).  Rows whose lse_run is +inf or NaN propagate NaN.
 */
dit_status dit_attn_chunk_fwd_accumulate(const void* q, const void* k, const void* v, float* o_run,
                                         float* lse_run, int B, int H, int N_q, int n_kv, int D,
                                         long long kv_head_stride, float scale, dit_stream stream);

/*
 * Split-KV form of dit_attn_chunk_fwd for problems with few queries (few
 * (head, Q pair) work items for the persistent grid, e.g. a stale-KV patch or a
 * short query block against long keys): every item is split over `splits`
 * contiguous ranges of the key tiles, computed in one launch into fp32 partials
 * in `workspace`, then merged exactly (the dit_attn_lse_merge combination) into
 * out / lse by a second launch.  Same result as dit_attn_chunk_fwd up to fp32
 * rounding of the merge.  The library allocates nothing: the caller passes the
 * workspace (device memory, 256-byte aligned, at least
 * dit_attn_splitkv_workspace_bytes(B, H, N_q, D, splits) bytes, overlapping no
 * other argument); it is scratch, overwritten by every call, so two calls in
 * flight at once must not share it.
 *   arguments as dit_attn_chunk_fwd (out contiguous, of out_dtype), plus
 *   splits : 1 (no split: workspace may be NULL) to min(64, ceil(n_kv / 128))
 */
dit_status dit_attn_chunk_fwd_splitkv(const void* q, const void* k, const void* v, void* out,
                                      float* lse, int B, int H, int N_q, int n_kv, int D,
                                      long long kv_head_stride, float scale, dit_dtype out_dtype,
                                      int splits, void* workspace, size_t workspace_bytes,
                                      dit_stream stream);

/*
 * dit_attn_chunk_fwd_splitkv without a caller workspace and without any device
 * allocation: the fp32 partials live in the library's own fixed device scratch
 * array of 128 MiB (set up once per device).  The pages have no counterpart; this
 * serves callers that must not allocate.  Requests whose partials need more than
 * 128 MiB (dit_attn_splitkv_workspace_bytes > 2^27) return DIT_ERR_UNSUPPORTED;
 * splits == 1 uses no scratch.  Nothing in the scratch needs clearing: the pass
 * writes every partial before the merge reads it.  There is one scratch array per
 * device: calls that overlap in time (other streams or host threads) race on it
 * and must be serialised by the caller.
 */
dit_status dit_attn_chunk_fwd_splitkv_noalloc(const void* q, const void* k, const void* v,
                                              void* out, float* lse, int B, int H, int N_q,
                                              int n_kv, int D, long long kv_head_stride,
                                              float scale, dit_dtype out_dtype, int splits,
                                              dit_stream stream);

/* Workspace bytes a split-KV call with these sizes needs (0 when splits <= 1 or a
 * size is not positive): splits * B*H*N_q * (D + 1) * 4, the LSE part 256-byte aligned. */
size_t dit_attn_splitkv_workspace_bytes(int B, int H, int N_q, int D, int splits);

/* A split count for an N_q x n_kv problem on the current device (1 to 16, at least two
 * key tiles per split): the one with the smallest estimated time, where the estimate is the
 * persistent grid's waves of (head, Q pair, key range) items times one item's KV tiles plus
 * a fixed per-item cost, plus (for splits > 1) the merge launch and its fp32 partial
 * traffic.  Never suggests a split the estimate puts behind no split.  Reads the device's SM
 * count; returns 1 if it cannot. */
int dit_attn_splitkv_suggest(int B, int H, int N_q, int n_kv);

/*
 * Exact merge of p chunk partials (O_c, lse_c) of the same queries:
 *   M = max_c lse_c;  lse = M + ln sum_c exp(lse_c - M);  O = sum_c exp(lse_c - lse) O_c
 * which is what the Ring section's online-softmax accumulation over the p
 * rounds computes (arganzheng.life, section 4.2 Ring).  A chunk whose lse is
 * -inf contributes nothing; a row whose lse_c are all -inf gets O = 0 and
 * lse = -inf.
 *   partials : device [p, B, H, N, D] of partial_dtype (chunk c at c*B*H*N*D)
 *   lses     : device fp32 [p, B, H, N]
 *   out      : device [B, H, N, D] of out_dtype;  lse: device fp32 [B, H, N]
 */
dit_status dit_attn_lse_merge(const void* partials, const float* lses, int p, void* out,
                              float* lse, int B, int H, int N, int D, dit_dtype partial_dtype,
                              dit_dtype out_dtype, dit_stream stream);

/*
 * Stale-KV attention of one patch, as displaced patch parallelism runs it
 * (PipeFusion / DistriFusion: arganzheng.life multi-GPU diffusion parallelism,
 * section 6 PipeFusion; xllm-io review of PipeFusion, method section; TACO-DiT,
 * hybrid SP KV buffer): a KV buffer holds K, V of all N tokens from the previous
 * diffusion step; the patch's freshly computed K, V rows [row0, row0 + m)
 * overwrite their stale rows in place, then the patch's m queries attend to the
 * whole buffer (their own rows fresh, every other row stale).  Launches on
 * `stream`: the row update (K and V together), then the attention, split over
 * `splits` key ranges plus a merge when splits > 1 (as dit_attn_chunk_fwd_splitkv:
 * a patch has few queries, so splitting its long key range fills the GPU).
 *   q            : device bf16 [B, H, m, D] (the patch's queries), contiguous
 *   k_new, v_new : device bf16 [B, H, m, D], contiguous (read)
 *   k_buf, v_buf : device bf16 [B, H, N, D], contiguous (rows [row0, row0+m)
 *                  overwritten, then read)
 *   out, lse     : as dit_attn_chunk_fwd for N_q = m queries over n_kv = N keys
 *   splits, workspace, workspace_bytes : as dit_attn_chunk_fwd_splitkv (1, NULL, 0: none)
 * 0 <= row0 <= N - m; the buffers must not overlap each other or q, k_new, v_new.
 */
dit_status dit_attn_stale_kv_fwd(const void* q, const void* k_new, const void* v_new, void* k_buf,
                                 void* v_buf, void* out, float* lse, int B, int H, int m, int N,
                                 int D, int row0, float scale, dit_dtype out_dtype, int splits,
                                 void* workspace, size_t workspace_bytes, dit_stream stream);

/*
 * Copies a logical [B, H, N, D] tensor of `dtype` elements from one strided
 * view to another (last dimension contiguous in both).  This is the local, on-GPU
 * half of Ulysses sequence parallelism's re-shard around attention, where an
 * all-to-all turns each rank's token shard of all heads into all tokens of its
 * head shard (arganzheng.life multi-GPU diffusion parallelism, section 4.1
 * Ulysses; valdrada.cn Wan2.2, CP section): the token-major (BSND) <-> head-major
 * (BHND) transpose and the packing of per-rank send buffers are such copies, and
 * so is writing fresh K/V rows into a KV buffer in place (a row-range view as dst).
 *   src, dst     : device pointers, 16-byte aligned; NULL strides = contiguous BHND
 *   D            : 64 or 128 (else DIT_ERR_UNSUPPORTED)
 * Strides follow dit_attn_fwd_strided's rules; dst must not map two elements to
 * one address and the two views' address ranges must not overlap
 * (DIT_ERR_INVALID_ARG).  Bit-exact: values are moved, never converted.
 */
dit_status dit_layout_copy(const void* src, const dit_strides* src_strides, void* dst,
                           const dit_strides* dst_strides, int B, int H, int N, int D,
                           dit_dtype dtype, dit_stream stream);

/*
 * Synchronises `stream`, then reads and clears the library's device status
 * word.  Returns DIT_ERR_TIMEOUT if any kernel since the last check gave up
 * on a bounded wait, DIT_ERR_CUDA if the synchronisation failed, else DIT_OK.
 */
dit_status dit_attn_check(dit_stream stream);

/*
 * TEST ONLY: failure injection for the timeout path.  While `enable` is
 * non-zero, attention launches from this process load Q but never issue the
 * K/V copies, so the MMA warp's bounded wait on the first K tile expires
 * after `wait_limit_cycles` SM clocks (<= 0 keeps the default of about two
 * seconds); the kernel then records DIT_ERR_TIMEOUT in the status word and
 * exits cleanly, and dit_attn_check() reports it.  Nothing faults or hangs.
 * Call with enable = 0 to restore normal operation.  Not thread-safe with
 * concurrent launches from other host threads.
 */
void dit_test_inject_stall(int enable, long long wait_limit_cycles);

/*
 * TEST ONLY: caps the number of CTAs of the persistent attention kernel
 * (normally one per SM; max_ctas <= 0 restores that).  With a small cap every
 * CTA walks many work items, which exercises the cross-item pipeline on small
 * inputs.  Affects later launches from this process; results do not change.
 */
void dit_test_set_grid_limit(int max_ctas);

/* Static, human-readable name of a status code. */
const char* dit_status_string(dit_status s);

/* Library version: major * 10000 + minor * 100 + patch. */
int dit_version(void);

#ifdef __cplusplus
}
#endif

#endif /* DITATTN_H */
