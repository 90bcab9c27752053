// attn_internal.h -- parameter blocks and launcher declarations shared by the
// host ABI (attn_api.cu) and the kernel translation units.  Not installed.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.h"

namespace attn {

// Prefill work tile: 128 query rows x 128 key/value rows per pipeline step.
constexpr int kPrefillBM = 128;
constexpr int kPrefillBN = 128;
// Decode: cache rows per shared-memory stage, and CTAs resident per SM.
constexpr int kDecodeStageTokens = 64;
constexpr int kDecodeCtasPerSm = 2;

struct PrefillParams {
  void *o;
  float *lse;               // may be null
  unsigned *err;            // device error word
  int64_t o_sb, o_sh, o_sn; // output element strides (d stride is 1)
  int Nq, Nkv, Hq, group, n_qtiles;  // n_qtiles: query-tile pairs along N_q (2 x 128 rows each)
  // Persistent schedule: n_units = H_q * B * n_qtiles pairs, numbered heads
  // fastest, then batches, then pairs (longest first under the causal mask);
  // n_ctas CTAs take them in rounds, dealt alternately forwards and backwards.
  int B, n_units, n_ctas;
  float scale_log2;         // scale * log2(e): scores are kept in base-2 units
  // Tensor-map coordinate slot (1..3) of the n, h and b coordinates for the
  // Q, K and V maps, packed as n | h << 2 | b << 4 (slot 0 is always d).
  uint32_t slots_q, slots_k, slots_v;
  // Variable-length batches only: packed Q/K/V/O rows; sequence b owns rows
  // [cu_q[b], cu_q[b+1]) of Q and O and [cu_k[b], cu_k[b+1]) of K and V; Nq / Nkv
  // then are the host's bounds on the per-sequence lengths; LSE is (H_q, total_q).
  const int32_t *cu_q, *cu_k;
  int total_q, total_k;
  // Mask and bias options: key j is kept for query i only if
  // i - window_left <= j <= i + window_right (-1: no bound on that side);
  // alibi_slopes (device fp32, one per q head) adds -slope_h |i - j| to scores.
  int window_left, window_right;
  const float *alibi_slopes;
  // Custom mask: per query row a key range [lo, hi) (int32 pairs, indexed by
  // b * Nq + row, or by the packed row for variable length); null: none.
  const int32_t *kv_ranges;
  // Rotary embeddings (ROPE builds): pair c of a row at position p turns by
  // (p * rope_f[c] mod 2^64) / 2^64 of a full turn; rope_inter selects the
  // pairs (2c, 2c + 1) instead of (c, c + D/2); rope_k = 0 when the keys come
  // already rotated (only the Q tiles are rotated then).
  int rope_inter, rope_k;
  uint64_t rope_f[64];
};

struct DecodeParams {
  const void *q, *kc, *vc;
  void *o;
  float *lse;               // may be null
  float *ws_o, *ws_lse;     // split partials (used when nsplit > 1)
  unsigned *err;
  int64_t q_sb, q_sh;
  int64_t kc_sb, kc_sh, kc_sn;
  int64_t vc_sb, vc_sh, vc_sn;
  int64_t o_sb, o_sh;
  int Hq, group, nhc, cache_len, chunk, nsplit;
  float scale_log2;
  uint32_t slots_k, slots_v;  // tensor-map coordinate slots, as for prefill
  // Paged caches only (cache_len then is the host's upper bound of the lengths):
  const int32_t *block_table;  // (B, max_pages) page ids, row stride bt_stride
  const int32_t *cache_lens;   // (B) tokens per request
  int64_t bt_stride;
  int page_size, max_pages, num_pages;
  // Mask and bias options: only keys j >= len - 1 - window_left are attended
  // (window_left < 0: all); alibi_slopes adds -slope_h (len - 1 - j).
  int window_left;
  const float *alibi_slopes;
  // Rotary embeddings: the query is rotated at its position (cache length - 1);
  // the cache holds rotated keys.  rope: 0 none, 1 rotate-half, 2 interleaved.
  int rope;
  uint64_t rope_f[64];
};

struct KvWriteParams {
  void *kc, *vc;
  const void *kn, *vn;
  int64_t kc_sb, kc_sh, kc_sn, vc_sb, vc_sh, vc_sn;
  int64_t kn_sb, kn_sh, kn_sn, vn_sb, vn_sh, vn_sn;
  int Hkv, n_new, pos, D;
  int64_t total_units;      // B * H_kv * n_new * (D / 8) 16-byte pieces per tensor
  unsigned *err;
  // Paged caches only: kc/vc are page pools (num_pages, H_kv, page_size, D);
  // token t of request b goes to position positions[b] + t.
  const int32_t *block_table;
  const int32_t *positions;
  int64_t bt_stride;
  int page_size, max_pages, num_pages;
  // Rotary embeddings: each new key is rotated at the cache position it is
  // written to.  rope: 0 none, 1 rotate-half, 2 interleaved.
  int rope;
  bool is_bf16;
  uint64_t rope_f[64];
};

// Launchers (return cudaSuccess or the launch error).
// masked: a window bound or ALiBi slopes are set (a separate kernel build, so
// that the plain kernel keeps its short softmax loop).
// rope: rotary embeddings on the Q and K tiles (two more builds).
cudaError_t launch_prefill(int D, bool causal, bool bf16, bool varlen, bool masked, bool rope, const CUtensorMap &tq,
                           const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p, int B,
                           cudaStream_t stream);
cudaError_t launch_prefill_masked(int D, bool causal, bool bf16, bool varlen, const CUtensorMap &tq,
                                  const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p, int B,
                                  cudaStream_t stream);
cudaError_t launch_prefill_rope(int D, bool causal, bool bf16, bool varlen, const CUtensorMap &tq,
                                const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p, int B,
                                cudaStream_t stream);
cudaError_t launch_prefill_rope_masked(int D, bool causal, bool bf16, bool varlen, const CUtensorMap &tq,
                                       const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p, int B,
                                       cudaStream_t stream);

// CTA-pair prefill (head dimension 128, no window, ALiBi, key ranges or
// rotary embeddings): units of 512 query rows (p.n_qtiles per (b, h)), p.n_ctas
// = 2 x clusters; tk_half has 64-row boxes (half a K tile per CTA).
cudaError_t launch_prefill_pair(bool causal, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk_half,
                                const CUtensorMap &tv, const PrefillParams &p, cudaStream_t stream);
// Clusters of two such CTAs that fit on the device at once (0: none / query failed).
int prefill_pair_max_clusters();
constexpr int kPairUnitRows = 512;  // query rows of a CTA-pair unit (two tiles of 256)

// Decode: heads served by one CTA, and launch (split kernel, plus the merge
// kernel when nsplit > 1).
int decode_heads_per_cta(int group);
cudaError_t launch_decode(int D, bool bf16, bool paged, int heads_per_cta, const CUtensorMap &tk,
                          const CUtensorMap &tv, const DecodeParams &p, int B, int Hkv, cudaStream_t stream);

cudaError_t launch_kv_cache_write(const KvWriteParams &p, bool paged, cudaStream_t stream);

// Backward.
struct BwdParams {
  const void *o, *dout;
  const float *lse;         // forward LSE (B, H_q, N_q), natural log
  float *dvec;              // workspace: D_i = rowsum(dO o O), (B, H_q, N_q)
  void *dq, *dk, *dv;
  unsigned *err;
  int64_t o_sb, o_sh, o_sn, do_sb, do_sh, do_sn;
  int64_t dq_sb, dq_sh, dq_sn, dk_sb, dk_sh, dk_sn, dv_sb, dv_sh, dv_sn;
  int Nq, Nkv, Hq, group;
  float scale, scale_log2;
  uint32_t slots_q, slots_do, slots_k, slots_v;
  // Tile order of the two tiled kernels (1-D grids): (batch, kv head) groups are
  // walked in chunks of chunk_dq / chunk_dkv groups, the longest causal tiles
  // of a chunk first, so that the CTAs in flight share a few groups' operands
  // in L2 (Q and dO of a group's heads for dK/dV, K and V for dQ).
  int B, Hkv, chunk_dq, chunk_dkv;
  // Masks and bias of the forward (masked build only), as in PrefillParams:
  // window bounds (-1: none), ALiBi slopes (device fp32, H_q), per-row key
  // ranges (device int32 pairs, (B, N_q, 2)).
  int window_left, window_right;
  const float *alibi_slopes;
  const int32_t *kv_ranges;
};
struct BwdMaps {
  CUtensorMap q, dout, k, v;  // 4-D tiled maps, 64 x 128 boxes, 128-byte swizzle
};
// masked: a window, ALiBi slopes or key ranges are set (the MASKED build).
// side: a second stream for the dK/dV kernel (null: everything on stream);
// stream waits for it before returning work.
cudaError_t launch_bwd(int D, bool causal, bool bf16, bool masked, const BwdMaps &m, const BwdParams &p, int B,
                       int Hkv, cudaStream_t stream, cudaStream_t side);
cudaError_t launch_bwd_masked(int D, bool causal, bool bf16, const BwdMaps &m, const BwdParams &p, int B, int Hkv,
                              cudaStream_t stream, cudaStream_t side);

// Rotary embedding of whole rows (rope_rows.cu): job j rotates the (B, H, N, D)
// 16-bit tensor src into dst (the same place for an in-place rotation), the row
// at sequence index n by n times each pair's turn step; sin_sign -1 applies the
// inverse rotation.  Element strides; the d stride is 1 and every row starts on
// 16 bytes.
struct RopeRowsJob {
  const void *src;
  void *dst;
  int64_t s_sb, s_sh, s_sn, d_sb, d_sh, d_sn;
  int H, N;
};
struct RopeRowsParams {
  RopeRowsJob job[2];
  int B;
  float sin_sign;
  uint64_t rope_f[64];  // pair turn steps, as in PrefillParams
};
cudaError_t launch_rope_rows(int D, bool bf16, bool interleaved, const RopeRowsParams &p, int n_jobs,
                             cudaStream_t stream);

}  // namespace attn
