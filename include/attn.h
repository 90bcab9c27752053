/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward library
 * (libattn_gb300.so).
 *
 * The library computes FlashAttention-2-style attention without ever
 * materialising the (B, H_q, N_q, N_kv) score matrix:
 *
 *     O = softmax(scale * Q K^T + mask) V,   LSE = ln(sum_j exp(scale * q.k_j))
 *
 * Notation follows "Skill: Write a Triton Attention Kernel" (Inputs the agent
 * should gather first): batch B, query heads H_q, key/value heads H_kv
 * (H_q a multiple of H_kv; GQA group = H_q / H_kv, MQA when H_kv = 1), query
 * length N_q, key/value length N_kv, head dimension D.
 *
 * Conventions shared by every call
 * --------------------------------
 * - Pointers are DEVICE pointers (cudaMalloc / PyTorch CUDA tensors) on the
 *   current CUDA device, unless stated otherwise.  The caller owns every
 *   buffer.  The library allocates no device memory of its own; it keeps only
 *   a small per-device cache of kernel attributes and function pointers.
 * - Strides are in ELEMENTS and are given in (b, h, n, d) order as int64_t[4].
 *   Any b/h/n strides are allowed (e.g. (B,H,N,D) or (B,N,H,D) memory), but
 *   the d stride must be 1, and every other stride times the element size
 *   (2 bytes) must be a multiple of 16 bytes; base pointers must be 16-byte
 *   aligned.  These are the tensor-memory-accelerator (TMA) rules.
 * - Q, K, V and O share one element type (attn_dtype_t).  LSE is always fp32,
 *   contiguous.  Accumulation is fp32 throughout.
 * - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *   Every call is stream-ordered and returns once its kernels are enqueued.
 *   The decode calls and the cache writes launch their kernels with
 *   programmatic stream serialization (each kernel may be scheduled while the
 *   preceding kernel of the stream drains, and waits for it to complete before
 *   it touches memory), which keeps stream order for the caller.
 * - Argument errors are detected on the host before anything is launched and
 *   are returned synchronously; nothing is enqueued in that case.  A failed
 *   launch returns ATTN_ERR_CUDA.
 * - Device-side failures (a pipeline wait that exceeded its time limit, or an
 *   out-of-range page id, length, position or sequence offset read from device
 *   memory by the paged and variable-length calls) are recorded in a device error word; read and clear it with
 *   attn_get_device_error().  While the word is non-zero, the library's
 *   kernels return immediately without computing.
 * - There is no CPU fallback and no other backend: every call runs the CUDA
 *   kernels of this library or returns an error.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    ATTN_OK = 0,
    ATTN_ERR_INVALID_ARG = 1,     /* null pointer, size < 1, H_q % H_kv != 0, bad scale, range error */
    ATTN_ERR_UNSUPPORTED = 2,     /* D not in {64, 128}, unknown dtype, device is not sm_103 */
    ATTN_ERR_ALIGNMENT = 3,       /* d stride != 1, pointer or stride not 16-byte aligned */
    ATTN_ERR_WORKSPACE = 4,       /* workspace missing or smaller than attn_decode_workspace_size() */
    ATTN_ERR_CUDA = 5,            /* a CUDA runtime/driver call or a launch failed */
    ATTN_ERR_DEVICE_TIMEOUT = 6,  /* a kernel gave up on a pipeline wait (see attn_get_device_error) */
    ATTN_ERR_DEVICE_INDEX = 7     /* a kernel read an out-of-range page id, length or position */
} attn_status_t;

typedef enum {
    ATTN_F16 = 0,
    ATTN_BF16 = 1
} attn_dtype_t;

/*
 * Mask, bias and position variants ("Skill: Write a Triton Attention Kernel",
 * Use this when: windowed attention, ALiBi, RoPE-fused and custom masks;
 * "Triton-FlashAttention", Deferred / explicitly out of scope: fused rotary
 * embeddings, sliding-window attention and attention biases such as ALiBi).
 * Passed to the *_ex entry points; a NULL pointer means none of them.  A
 * zero-initialised struct with window_left = window_right = -1 is the same as
 * NULL.
 *
 *   window_left   -1, or W >= 0: query i attends only to keys j >= i - W
 *   window_right  -1, or W >= 0: query i attends only to keys j <= i + W
 *                 (prefill only; with causal = 1 the bound is j <= i anyway)
 *   alibi_slopes  NULL, or a device fp32 array of H_q slopes: the score of
 *                 (i, j) gets -slopes[h] * |i - j| added before the softmax
 *   rope_theta    0, or the base theta > 0 of rotary position embeddings
 *                 (RoPE): before the scores are formed, every query and key
 *                 row at position p has each of its D/2 coordinate pairs
 *                 (x_a, x_b) rotated by the angle p * theta^(-2c/D), c the
 *                 pair's index:  x_a' = x_a cos - x_b sin,
 *                 x_b' = x_b cos + x_a sin.  The kernels rotate Q and K tiles
 *                 on chip; the caller's tensors are not modified.
 *   rope_interleaved  which coordinates form pair c: 0 pairs (c, c + D/2)
 *                 (the "rotate half" layout), 1 pairs (2c, 2c + 1)
 *   rope_rotated_keys  prefill and backward with rope_theta > 0: 1 when the keys
 *                 passed in are already rotated at their positions (for
 *                 example read back from a cache written by kv_cache_write_ex
 *                 with the same RoPE options); the kernel then rotates only
 *                 the query tiles, which costs far less than rotating every K
 *                 tile it reads.  0: the kernel rotates both.
 *   kv_ranges     prefill only: NULL, or a custom mask given as a device int32
 *                 array of key ranges, one [lo, hi) pair per query row --
 *                 (B, N_q, 2) for attn_fwd_prefill_ex and the host-buffer
 *                 call, (total_q, 2) for the variable-length call (keys
 *                 counted from the row's sequence start): query row i attends
 *                 only to keys j with lo <= j < hi, in addition to the causal
 *                 and window bounds (block-diagonal, document and prefix masks
 *                 are such ranges).  Tiles are skipped by the causal and
 *                 window bands only; the ranges mask within them.  Decode calls
 *                 return ATTN_ERR_UNSUPPORTED when it is set.
 *   num_splits    decode only: 0 lets the library choose how many parts the
 *                 cache is split into; n in [1, 64] uses at most n (1: one
 *                 pass, no workspace).  More splits than the automatic choice
 *                 need a workspace of 4 * B * H_q * n * (D + 1) bytes.
 *   prefill_kernel  attn_fwd_prefill_ex and the host-buffer call only (the
 *                 other calls accept only 0): which kernel computes it.
 *                 0 = automatic, 1 = the one-CTA kernel (every variant),
 *                 2 = the CTA-pair kernel: clusters of two CTAs on
 *                 neighbouring SMs share each tensor-core product (M = 256
 *                 rows, each CTA holding half of every K and V tile) and keep
 *                 P in shared memory; head dimension 128 without windows,
 *                 ALiBi, rotary embeddings or key ranges, else
 *                 ATTN_ERR_UNSUPPORTED.  Both compute the same function to the
 *                 same tolerances; automatic runs the one-CTA kernel, which
 *                 measures faster on GB300.
 *
 * Positions are those of the causal mask (top-left, per sequence for the
 * variable-length call); for decode the query sits at position cache_len - 1
 * (per request for the paged call) and window_right is ignored.  A query row
 * left with no key gets O = 0 and LSE = -inf.
 *
 * RoPE and the KV cache: the decode calls rotate only the query, at its
 * position; the cache must already hold rotated keys, which is what
 * kv_cache_write_ex / kv_cache_write_paged_ex write when given the same
 * rope_theta and rope_interleaved (each new key rotated at the position it is
 * written to).  The values are never rotated.
 *
 * Errors: a window below -1, a rope_theta that is negative or not finite, a
 * rope_interleaved or rope_rotated_keys other than 0 or 1, a num_splits
 * outside [0, 64], or a prefill_kernel outside [0, 2] (or not 0 where the call
 * has no choice) gives
 * ATTN_ERR_INVALID_ARG; slopes not 4-byte aligned or key ranges not 8-byte
 * aligned give ATTN_ERR_ALIGNMENT.
 * The struct is read during the call; the slope and key-range arrays are read
 * by the kernel, so they must stay valid until the work enqueued on the
 * stream has finished.
 * The caller owns both.
 */
typedef struct {
    int32_t window_left;
    int32_t window_right;
    const float *alibi_slopes;
    float rope_theta;
    int32_t rope_interleaved;
    int32_t num_splits;
    int32_t rope_rotated_keys;
    const int32_t *kv_ranges;
    int32_t prefill_kernel;
} attn_options_t;

/*
 * attn_fwd_prefill -- fused attention forward over a whole sequence.
 *
 * Follows "Skill: Write a Triton Attention Kernel", Required reasoning process
 * steps 1-9 (tiles of query rows, online softmax with running max m_i and sum
 * l_i, rescale by alpha = exp(m_old - m_new), O = O_i / l_i after the loop,
 * lse = m_i + log(l_i)), and Correctness requirements (mask before the max,
 * -inf for keys past N_kv, rows past N_q not stored).
 *
 *   q    (B, H_q,  N_q,  D) element strides q_str[4]    read
 *   k    (B, H_kv, N_kv, D) element strides k_str[4]    read
 *   v    (B, H_kv, N_kv, D) element strides v_str[4]    read
 *   o    (B, H_q,  N_q,  D) element strides o_str[4]    written (rows < N_q only)
 *   lse  (B, H_q,  N_q) fp32 contiguous, natural log, or NULL to skip it
 *   causal  0 or 1; 1 keeps key j for query i iff j <= i (top-left aligned,
 *           positions compared with no offset, as the pages write the mask)
 *   scale   softmax scale applied to Q K^T; must be finite and > 0
 *           (1/sqrt(D) is the usual value)
 *   D must be 64 or 128.  N_q, N_kv >= 1 and arbitrary (not block-aligned).
 *
 * Returns ATTN_OK after enqueueing one kernel on `stream`.
 */
attn_status_t attn_fwd_prefill(const void *q, const void *k, const void *v, void *o, float *lse,
                               attn_dtype_t dtype, int B, int H_q, int H_kv, int N_q, int N_kv, int D,
                               const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                               const int64_t o_str[4], int causal, float scale, void *stream);

/* attn_fwd_prefill with mask and bias options (see attn_options_t). */
attn_status_t attn_fwd_prefill_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                                  attn_dtype_t dtype, int B, int H_q, int H_kv, int N_q, int N_kv, int D,
                                  const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                                  const int64_t o_str[4], int causal, float scale, const attn_options_t *opts,
                                  void *stream);

/*
 * attn_fwd_prefill_varlen -- attn_fwd_prefill over a batch of sequences of
 * different lengths, packed without padding.
 *
 * Covers the variable-length batches of "Skill: Write a Triton Attention
 * Kernel" (Inputs: a CSR-style variable-length layout; Correctness
 * requirements: the KV loop of a sequence ends at that sequence's own length,
 * and padding never contributes).  Sequence b owns rows
 * [cu_seqlens_q[b], cu_seqlens_q[b+1]) of Q and O and rows
 * [cu_seqlens_k[b], cu_seqlens_k[b+1]) of K and V; masks (causal: key j kept
 * for query i iff j <= i) are per sequence, positions counted from the start
 * of the sequence.
 *
 *   q     (total_q, H_q, D)  element strides q_str[3] in (row, head, d) order   read
 *   k, v  (total_k, H_kv, D) strides k_str[3], v_str[3]                        read
 *   o     (total_q, H_q, D)  strides o_str[3]                                  written
 *   lse   (H_q, total_q) fp32 contiguous, natural log, or NULL
 *   cu_seqlens_q, cu_seqlens_k  int32 device arrays (B + 1), non-decreasing,
 *         starting at 0 and ending at total_q / total_k
 *   max_seqlen_q, max_seqlen_k  host bounds of the sequence lengths (they size
 *         the grid); a sequence with no keys gets O = 0 and LSE = -inf
 *   Rows are 16-byte aligned as for attn_fwd_prefill; d stride 1.
 *
 * A cu_seqlens entry that is out of order, past total_*, or gives a length
 * above max_seqlen_* is recorded as ATTN_ERR_DEVICE_INDEX and that sequence
 * is left unwritten.  Returns ATTN_OK after enqueueing one kernel on `stream`.
 */
attn_status_t attn_fwd_prefill_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                                      attn_dtype_t dtype, int B, int H_q, int H_kv, int D, const int32_t *cu_seqlens_q,
                                      const int32_t *cu_seqlens_k, int max_seqlen_q, int max_seqlen_k, int total_q,
                                      int total_k, const int64_t q_str[3], const int64_t k_str[3],
                                      const int64_t v_str[3], const int64_t o_str[3], int causal, float scale,
                                      void *stream);

/* attn_fwd_prefill_varlen with mask and bias options (see attn_options_t). */
attn_status_t attn_fwd_prefill_varlen_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                                         attn_dtype_t dtype, int B, int H_q, int H_kv, int D,
                                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int max_seqlen_q,
                                         int max_seqlen_k, int total_q, int total_k, const int64_t q_str[3],
                                         const int64_t k_str[3], const int64_t v_str[3], const int64_t o_str[3],
                                         int causal, float scale, const attn_options_t *opts, void *stream);

/*
 * attn_bwd_workspace_size -- bytes of scratch attn_bwd needs: one fp32 per
 * query row, 4 * B * H_q * N_q rounded up to 16.  Returns 0 on bad arguments.
 * (A sizing utility of this library; the pages define no counterpart.)
 */
size_t attn_bwd_workspace_size(int B, int H_q, int N_q);

/*
 * attn_bwd -- gradients of the fused attention forward from its saved LSE.
 *
 * The "Skill: Write a Triton Attention Kernel" page keeps lse = m + log(l)
 * precisely so that a backward pass can rebuild the attention weights
 * (P = exp(scale q.k - lse)) without storing them; "Triton-FlashAttention"
 * lists the GQA backward (dK, dV summed over the q heads of a group) among
 * its deferred work.  With dO the gradient of O:
 *   dV = P^T dO,  dP = dO V^T,  D_i = sum_d dO_id O_id,  dS = P o (dP - D),
 *   dQ = scale dS K,  dK = scale dS^T Q  (dK, dV summed over each GQA group).
 *
 *   q, k, v, o, lse  the forward's inputs, output and LSE (attn_fwd_prefill
 *                    layouts and conventions, same causal and scale)     read
 *   dout             dO, (B, H_q, N_q, D) strides do_str[4]              read
 *   dq               (B, H_q, N_q, D) strides dq_str[4]                  written
 *   dk, dv           (B, H_kv, N_kv, D) strides dk_str[4], dv_str[4]     written
 *   workspace        device scratch of attn_bwd_workspace_size() bytes, not
 *                    initialised; calls sharing one workspace must not overlap
 *
 * Deterministic (no atomics): dQ is computed per query tile, dK and dV per key
 * tile with every q head of the group.  Returns ATTN_OK after enqueueing three
 * kernels: D_i and dQ on `stream`, and dK/dV on a library-owned stream of the
 * current device that starts after D_i and that `stream` waits for (event
 * dependencies), so the two independent kernels share the GPU.  All work of the
 * call is complete once the work enqueued on `stream` so far is; a CUDA graph
 * captured on `stream` includes it (the library stream is created by the first
 * call of any kind on the device, which must precede the capture).  Concurrent
 * calls from several host threads share that stream (their dK/dV kernels run
 * one after another).
 */
attn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                       const float *lse, void *dq, void *dk, void *dv, attn_dtype_t dtype, int B, int H_q, int H_kv,
                       int N_q, int N_kv, int D, const int64_t q_str[4], const int64_t k_str[4],
                       const int64_t v_str[4], const int64_t o_str[4], const int64_t do_str[4],
                       const int64_t dq_str[4], const int64_t dk_str[4], const int64_t dv_str[4], int causal,
                       float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * attn_bwd_ex_workspace_size -- bytes of scratch attn_bwd_ex needs with these
 * options: attn_bwd_workspace_size(B, H_q, N_q), plus, with rope_theta > 0,
 * 2 * B * H_q * N_q * D for the rotated queries and -- unless
 * rope_rotated_keys -- 2 * B * H_kv * N_kv * D for the rotated keys.  Equal to
 * attn_bwd_workspace_size without rotary embeddings.  Returns 0 on bad
 * arguments or options.  (A sizing utility of this library.)
 */
size_t attn_bwd_ex_workspace_size(int B, int H_q, int H_kv, int N_q, int N_kv, int D, const attn_options_t *opts);

/*
 * attn_bwd with the forward's mask, bias and position options (see
 * attn_options_t): window_left, window_right, alibi_slopes, kv_ranges and the
 * rotary embedding (rope_theta, rope_interleaved, rope_rotated_keys), the same
 * as the attn_fwd_prefill_ex call whose O and LSE are passed in (a query row
 * the forward left without keys, O = 0 and LSE = -inf, gets dQ = 0 and adds
 * nothing to dK, dV).  The bias enters the gradients only through P.
 *
 * Rotary embeddings ("Triton-FlashAttention" names RoPE among the fused
 * extensions): with R the rotation of each row at its position, the forward
 * is attention(R Q, R K, V), so the gradients with respect to the caller's Q
 * and K are dQ = R^T dQ', dK = R^T dK', where dQ', dK' are the backward's
 * gradients with respect to the rotated rows and R^T rotates each pair by the
 * opposite angle; dV is unchanged.  The call rotates Q (and K) into the
 * workspace, runs the backward kernels on them and rotates dQ (and dK) back in
 * place: two more kernels.  With rope_rotated_keys = 1, k holds the rotated
 * keys and dk receives the gradient with respect to them (not turned back).
 *
 *   workspace        attn_bwd_ex_workspace_size() bytes with the same options
 *
 * num_splits is ignored; prefill_kernel must be 0.  Option errors as for the
 * other *_ex calls.
 */
attn_status_t attn_bwd_ex(const void *q, const void *k, const void *v, const void *o, const void *dout,
                          const float *lse, void *dq, void *dk, void *dv, attn_dtype_t dtype, int B, int H_q,
                          int H_kv, int N_q, int N_kv, int D, const int64_t q_str[4], const int64_t k_str[4],
                          const int64_t v_str[4], const int64_t o_str[4], const int64_t do_str[4],
                          const int64_t dq_str[4], const int64_t dk_str[4], const int64_t dv_str[4], int causal,
                          float scale, const attn_options_t *opts, void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * attn_decode_workspace_size -- bytes of scratch attn_fwd_decode needs.
 *
 * Split-KV decode writes one partial output (D fp32) and one partial LSE per
 * (b, q-head, split) and merges them.  The number of splits depends only on
 * B, H_q, H_kv and the current device's SM count (never on cache_len), so a
 * workspace sized once serves every cache length.  Returns 0 on bad
 * arguments.  Host-only; reads the current device's SM count.  (A sizing
 * utility of this library; the pages define no counterpart.  The split itself
 * is the decode design of attn_fwd_decode below.)
 */
size_t attn_decode_workspace_size(int B, int H_q, int H_kv, int D);

/*
 * attn_decode_splits -- number of KV splits attn_fwd_decode uses for these
 * sizes on the current device (1 means one kernel and no workspace traffic;
 * more means a split kernel plus a merge kernel).  Returns 0 on bad
 * arguments.  Host-only.  (A query utility of this library; the pages define
 * no counterpart.)
 */
int attn_decode_splits(int B, int H_q, int H_kv, int cache_len, int D);

/*
 * attn_fwd_decode -- attention of ONE new query token per (batch, q-head) over
 * a preallocated KV cache whose first cache_len positions are valid.
 *
 * Follows "Triton-FlashAttention", Phase 2 (a separate decode kernel; every
 * cached position is valid, so there is no causal loop; cache_len is a
 * runtime value, never a compile-time one), split over the KV sequence: each
 * (b, kv-head, split) streams its share of the cache once for all H_q/H_kv
 * query heads of the group and produces (O_s, lse_s); the splits are merged
 * as lse = ln sum_s exp(lse_s), O = sum_s exp(lse_s - lse) O_s.
 *
 *   q        (B, H_q, 1, D)        strides q_str[4] (n stride ignored)   read
 *   k_cache  (B, H_kv, max_len, D) strides kc_str[4]                     read rows < cache_len
 *   v_cache  (B, H_kv, max_len, D) strides vc_str[4]                     read rows < cache_len
 *   o        (B, H_q, 1, D)        strides o_str[4]                      written
 *   lse      (B, H_q) fp32 contiguous, natural log, or NULL
 *   cache_len   1 <= cache_len (rows [0, cache_len) of the cache are used)
 *   workspace   device scratch of at least attn_decode_workspace_size(B, H_q, H_kv, D)
 *               bytes (may be NULL when that size is 0); contents need not be
 *               initialised; calls sharing one workspace must not overlap
 *
 * Returns ATTN_OK after enqueueing one or two kernels on `stream`.
 */
attn_status_t attn_fwd_decode(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                              attn_dtype_t dtype, int B, int H_q, int H_kv, int cache_len, int D,
                              const int64_t q_str[4], const int64_t kc_str[4], const int64_t vc_str[4],
                              const int64_t o_str[4], float scale, void *workspace, size_t workspace_bytes,
                              void *stream);

/* attn_fwd_decode with mask and bias options (see attn_options_t); a left window
 * W limits the keys read from the cache to the last W + 1 positions. */
attn_status_t attn_fwd_decode_ex(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                                 attn_dtype_t dtype, int B, int H_q, int H_kv, int cache_len, int D,
                                 const int64_t q_str[4], const int64_t kc_str[4], const int64_t vc_str[4],
                                 const int64_t o_str[4], float scale, void *workspace, size_t workspace_bytes,
                                 const attn_options_t *opts, void *stream);

/*
 * kv_cache_write -- copy n_new tokens of K and V into a preallocated cache at
 * positions [pos, pos + n_new).
 *
 * Follows "Triton-FlashAttention", Phase 2: the cache is allocated once with
 * room for max_len positions and filled in place (no reallocation as it
 * grows), and writing into it is a call of its own, apart from attention.
 *
 *   k_cache, v_cache  (B, H_kv, max_len, D) strides kc_str / vc_str   written
 *   k_new, v_new      (B, H_kv, n_new, D)   strides kn_str / vn_str   read
 *   0 <= pos, pos + n_new <= max_len
 *
 * Returns ATTN_OK after enqueueing one kernel on `stream`.
 */
attn_status_t kv_cache_write(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                             attn_dtype_t dtype, int B, int H_kv, int n_new, int D, int pos, int max_len,
                             const int64_t kc_str[4], const int64_t vc_str[4], const int64_t kn_str[4],
                             const int64_t vn_str[4], void *stream);

/*
 * kv_cache_write_ex -- kv_cache_write with options: with rope_theta > 0 each
 * new key is rotated (rotary position embeddings, see attn_options_t) at the
 * cache position it is written to, pos + t, so that the cache holds the keys
 * that attn_fwd_decode_ex with the same rope_theta and rope_interleaved
 * expects ("Skill: Write a Triton Attention Kernel", Use this when: RoPE-fused
 * attention; "Triton-FlashAttention", Deferred: fused rotary embeddings).
 * Values are copied unchanged.  The other option fields are not used here.
 * The rotation is computed in fp32 and rounded once to the cache's type.
 */
attn_status_t kv_cache_write_ex(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                                attn_dtype_t dtype, int B, int H_kv, int n_new, int D, int pos, int max_len,
                                const int64_t kc_str[4], const int64_t vc_str[4], const int64_t kn_str[4],
                                const int64_t vn_str[4], const attn_options_t *opts, void *stream);

/*
 * attn_fwd_prefill_host -- attn_fwd_prefill_ex on host-resident tensors, with
 * the host-to-device copies, the compute and the device-to-host copies
 * pipelined.  (The pages time kernels on device-resident inputs; this entry
 * point is a convenience of this library for callers whose tensors live in
 * host memory, e.g. Grace-resident activations.)
 *
 * The problem is cut into chunks of (batch element, block of kv heads with all
 * their q heads); chunk i's inputs are copied on a library-owned stream while
 * chunk i-1 is computed on `stream` and chunk i-2's outputs are copied back on
 * a second library-owned stream (two non-blocking streams per device, created
 * on first use and kept until the process exits).  Each chunk is computed by
 * the same kernel as attn_fwd_prefill_ex on its contiguous slice, so results
 * equal those of attn_fwd_prefill_ex on the whole problem.
 *
 *   q, o  host (B, H_q, N_q, D) contiguous; k, v host (B, H_kv, N_kv, D)
 *         contiguous; lse host (B, H_q, N_q) fp32 or NULL.  Page-locked
 *         (pinned) host memory is what makes the copies asynchronous.
 *   workspace  device memory of at least attn_fwd_prefill_host_workspace_size()
 *         bytes, 256-byte aligned: staging copies of Q, K, V, O and LSE.
 *   causal, scale, opts  as for attn_fwd_prefill_ex (ALiBi slopes: a device
 *         array of H_q values).
 *
 * Ordering: the copies into the workspace start after the work enqueued on
 * `stream` before the call; `stream` waits for the last copy back, so o and
 * lse are complete once `stream` is.  The caller keeps the host buffers and
 * the workspace alive and unmodified until then.
 *
 * Errors: as attn_fwd_prefill_ex; ATTN_ERR_WORKSPACE for a missing or short
 * workspace, ATTN_ERR_ALIGNMENT for a workspace not 256-byte aligned,
 * ATTN_ERR_CUDA if a copy or stream operation fails (copies already enqueued
 * may still run: synchronise `stream` before reusing the buffers).
 */
size_t attn_fwd_prefill_host_workspace_size(attn_dtype_t dtype, int B, int H_q, int H_kv, int N_q, int N_kv, int D);
attn_status_t attn_fwd_prefill_host(const void *q, const void *k, const void *v, void *o, float *lse,
                                    attn_dtype_t dtype, int B, int H_q, int H_kv, int N_q, int N_kv, int D,
                                    int causal, float scale, const attn_options_t *opts, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * attn_fwd_decode_noalloc -- attn_fwd_decode for callers that may not allocate
 * device memory.  (The pages have no counterpart of this entry point; it is a
 * convenience of this library.)
 *
 * Some callers cannot call cudaMalloc or hand the library a workspace: a
 * plugin whose host framework owns every device allocation through its own
 * planner and forbids allocating after start-up, or a latency-critical serving
 * loop that must never hit cudaMalloc's implicit device synchronisation or an
 * out-of-memory failure in the middle of a request.  This entry point takes
 * the same arguments as attn_fwd_decode minus the workspace; the split
 * partials go to a scratch array of 4 MiB compiled into the library, which
 * every device that loads the library keeps until the process exits.  It
 * allocates nothing and calls no allocating routine.
 *
 *   Limit: the call needs 4 * B * H_q * splits * (D + 1) bytes of scratch
 *   (splits = attn_decode_splits(...), 0 bytes when splits == 1); if that
 *   exceeds 4 MiB it returns ATTN_ERR_WORKSPACE and launches nothing.
 *   Otherwise arguments, errors and results are those of attn_fwd_decode.
 *
 *   Set-up: the first call on a device looks up the device address of the
 *   scratch array (with that device current) and caches it; make that first
 *   call before capturing any stream.
 *
 *   Sharing: every call on a device uses the same scratch array, and the array
 *   keeps whatever the previous call left in it (nothing in it needs to start
 *   at zero).  Two calls whose kernels overlap on the GPU -- on different
 *   streams, or from different host threads -- race on the array and corrupt
 *   each other's results: order such calls on one stream.
 */
attn_status_t attn_fwd_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                                      attn_dtype_t dtype, int B, int H_q, int H_kv, int cache_len, int D,
                                      const int64_t q_str[4], const int64_t kc_str[4], const int64_t vc_str[4],
                                      const int64_t o_str[4], float scale, void *stream);

/*
 * attn_fwd_decode_paged -- decode for a batch of requests whose KV caches live
 * in pages of a shared pool and whose lengths differ.
 *
 * Extends attn_fwd_decode to the serving layout the "Triton-FlashAttention"
 * page lists as deferred ("Deferred / explicitly out of scope": batched, paged
 * decode across requests with differing cache lengths).  Request b's cache is
 * the sequence of pages block_table[b][0], block_table[b][1], ...; its first
 * cache_lens[b] rows are attended to by its one query token.
 *
 *   q            (B, H_q, 1, D) strides q_str[4]                            read
 *   k_pages      (num_pages, H_kv, page_size, D) strides kp_str[4], in
 *                (page, head, row, d) order                                 read
 *   v_pages      same shape, strides vp_str[4]                              read
 *   block_table  int32 device array (B, max_pages), row stride bt_stride
 *                elements (>= max_pages); entries past a request's last page
 *                are never read                                             read
 *   cache_lens   int32 device array (B); 0 <= cache_lens[b] <= max_cache_len  read
 *   max_cache_len  host upper bound of the lengths (<= max_pages * page_size);
 *                it sizes the split of each request's cache over CTAs
 *   page_size    16, 32 or a multiple of 64 (rows per page)
 *   o, lse       as attn_fwd_decode; a request of length 0 gets O = 0, LSE = -inf
 *   workspace    as attn_fwd_decode (attn_decode_workspace_size)
 *
 * A page id outside [0, num_pages) or a length outside [0, max_cache_len]
 * found on the device is recorded as ATTN_ERR_DEVICE_INDEX (the page reads as
 * zeros, the length is clamped); argument errors are returned before launch.
 */
attn_status_t attn_fwd_decode_paged(const void *q, const void *k_pages, const void *v_pages, void *o, float *lse,
                                    attn_dtype_t dtype, int B, int H_q, int H_kv, int D, int num_pages,
                                    int page_size, const int32_t *block_table, int max_pages, int64_t bt_stride,
                                    const int32_t *cache_lens, int max_cache_len, const int64_t q_str[4],
                                    const int64_t kp_str[4], const int64_t vp_str[4], const int64_t o_str[4],
                                    float scale, void *workspace, size_t workspace_bytes, void *stream);

/* attn_fwd_decode_paged with mask and bias options (see attn_options_t). */
attn_status_t attn_fwd_decode_paged_ex(const void *q, const void *k_pages, const void *v_pages, void *o, float *lse,
                                       attn_dtype_t dtype, int B, int H_q, int H_kv, int D, int num_pages,
                                       int page_size, const int32_t *block_table, int max_pages, int64_t bt_stride,
                                       const int32_t *cache_lens, int max_cache_len, const int64_t q_str[4],
                                       const int64_t kp_str[4], const int64_t vp_str[4], const int64_t o_str[4],
                                       float scale, void *workspace, size_t workspace_bytes,
                                       const attn_options_t *opts, void *stream);

/*
 * kv_cache_write_paged -- write n_new tokens per request into a paged cache.
 *
 * Token t of request b goes to position positions[b] + t of its cache, i.e. row
 * (pos % page_size) of page block_table[b][pos / page_size] (the page layout
 * of attn_fwd_decode_paged).  positions is an int32 device array (B).  A write
 * whose page index or page id is out of range is skipped and recorded as
 * ATTN_ERR_DEVICE_INDEX.
 *
 *   k_pages, v_pages  (num_pages, H_kv, page_size, D) strides kp_str / vp_str   written
 *   k_new, v_new      (B, H_kv, n_new, D) strides kn_str / vn_str               read
 */
attn_status_t kv_cache_write_paged(void *k_pages, void *v_pages, const void *k_new, const void *v_new,
                                   attn_dtype_t dtype, int B, int H_kv, int n_new, int D, int num_pages,
                                   int page_size, const int32_t *block_table, int max_pages, int64_t bt_stride,
                                   const int32_t *positions, const int64_t kp_str[4], const int64_t vp_str[4],
                                   const int64_t kn_str[4], const int64_t vn_str[4], void *stream);

/* kv_cache_write_paged with options: with rope_theta > 0 the key of token t of
 * request b is rotated at its position positions[b] + t (see kv_cache_write_ex). */
attn_status_t kv_cache_write_paged_ex(void *k_pages, void *v_pages, const void *k_new, const void *v_new,
                                      attn_dtype_t dtype, int B, int H_kv, int n_new, int D, int num_pages,
                                      int page_size, const int32_t *block_table, int max_pages, int64_t bt_stride,
                                      const int32_t *positions, const int64_t kp_str[4], const int64_t vp_str[4],
                                      const int64_t kn_str[4], const int64_t vn_str[4], const attn_options_t *opts,
                                      void *stream);

/*
 * attn_get_device_error -- synchronise `stream`, then read and clear the
 * device error word of the current device in one atomic step (a one-thread
 * kernel exchanges it with zero, so a failure recorded by a kernel still
 * running on another stream is either returned now or kept for the next
 * call, never lost).  Returns ATTN_OK if no kernel reported a failure,
 * ATTN_ERR_DEVICE_TIMEOUT if one gave up on a wait, ATTN_ERR_DEVICE_INDEX if
 * a paged or variable-length call met an out-of-range page id, length,
 * position or offset, ATTN_ERR_CUDA if a CUDA call failed.  (Error reporting
 * of this library; the pages define no counterpart.)
 */
attn_status_t attn_get_device_error(void *stream);

/*
 * attn_selftest_wait_timeout -- failure-detection self-test.  Enqueues one
 * small kernel on `stream` that waits on a shared-memory mbarrier nothing
 * ever arrives on, through the same bounded wait every pipeline wait of the
 * library uses (a wall-clock limit of 4 s, then the wait gives up, records
 * the time-out in the device error word and the kernel returns).  The next
 * attn_get_device_error() on the stream then returns ATTN_ERR_DEVICE_TIMEOUT
 * and clears the word; the CUDA context stays usable.  Returns ATTN_OK after
 * enqueueing, ATTN_ERR_UNSUPPORTED on a device other than sm_103, ATTN_ERR_CUDA
 * if the launch failed.
 */
attn_status_t attn_selftest_wait_timeout(void *stream);

/* attn_status_string -- static, human-readable name of a status code.  (A
 * utility of this library; the pages define no counterpart.) */
const char *attn_status_string(attn_status_t status);

/* attn_version -- library version as major * 10000 + minor * 100 + patch
 * (200: options with rotary embeddings and the decode split count).
 * (A utility of this library; the pages define no counterpart.) */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
