// decode.cu -- split-KV decode attention and the KV-cache write, sm_103a.
//
// Decode ("Triton-FlashAttention", Phase 2): one new query token per
// (batch, q-head) attends to the first cache_len rows of a preallocated cache.
// The work is HBM-bound -- every cached K/V byte is read once per step -- so it
// runs on the CUDA cores and is organised around streaming the cache:
//
//   decode_split: one CTA per (split, kv-head [x head chunk], batch), two CTAs
//     resident per SM.  A producer warp streams the split's keys and values
//     through a 3-deep ring of 64-token shared-memory stages with TMA tensor
//     loads (128-byte swizzle), so the bytes in flight cost no registers.  The
//     CTA reads its share of the cache ONCE for all H_q/H_kv query heads of
//     the group.  Four consumer warps each take 16 tokens of a stage:
//       scores   lane = (token, half of D): one 16-byte swizzled shared load per
//                8 dimensions, packed fma.rn.f32x2 against the pre-scaled
//                query, one xor-16 shuffle to join the two halves;
//       softmax  a warp-wide max per head (xor shuffles), base-2 exponentials,
//                per-lane partial sums (reduced once at the end);
//       P . V    lane = (token slot, 16-byte slice of D), P broadcast from
//                shared memory, packed FMAs into per-lane accumulators.
//     Each warp keeps its own online-softmax state; warps merge through shared
//     memory at the end, and the result is either the output (one split) or a
//     partial (O_s, lse_s) in the workspace.
//   decode_merge: combines the partials of every (b, q-head):
//     lse = ln sum_s e^{lse_s}, O = sum_s e^{lse_s - lse} O_s.
//
// kv_cache_write: copies new tokens into cache rows [pos, pos + n) with one
// 16-byte piece per thread.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <utility>

#include "attn_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace attn {
namespace {

constexpr int kTok = kDecodeStageTokens;  // tokens per stage
constexpr int kStages = 3;
constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kTokPerWarp = kTok / kConsumerWarps;  // 16
constexpr float kLn2 = 0.693147180559945309f;
static_assert(kTokPerWarp == 16, "score mapping assumes 16 tokens per warp and stage");

template <int D, int GH>
struct DecCfg {
  static constexpr int KCH = D / 64;                  // 128-byte boxes per row
  static constexpr int CPR = D / 8;                   // 16-byte chunks per row
  static constexpr int TPI = 32 / CPR;                // tokens per P.V step of a warp
  static constexpr uint32_t BOX_BYTES = kTok * 128;   // one TMA box: kTok rows x 64 elements
  static constexpr uint32_t KV_BYTES = kTok * D * 2;  // K (or V) of one stage
  static constexpr uint32_t STAGE_BYTES = 2 * KV_BYTES;
  static constexpr uint32_t OFF_Q = kStages * STAGE_BYTES;          // fp32 [GH][D]
  static constexpr uint32_t OFF_P = OFF_Q + GH * D * 4;             // fp32 [warps][16][GH]
  static constexpr uint32_t OFF_ML = OFF_P + kConsumerWarps * kTokPerWarp * GH * 4;  // m, l [warps][GH]
  static constexpr uint32_t OFF_BAR = OFF_ML + 2 * kConsumerWarps * GH * 4;
  static constexpr uint32_t OFF_MISC = OFF_BAR + 2 * kStages * 8;
  static constexpr uint32_t SMEM_BYTES = OFF_MISC + 16 + 1024;
  // End-of-CTA merge area, placed over the (then idle) stage ring: fp32 [warps][TPI][GH][D].
  static constexpr uint32_t MERGE_BYTES = kConsumerWarps * TPI * GH * D * 4;
  static_assert(MERGE_BYTES <= kStages * STAGE_BYTES, "merge area must fit in the stage ring");
};

__device__ __forceinline__ uint64_t f2(float a, float b) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(a), "f"(b));
  return r;
}
__device__ __forceinline__ float2 unf2(uint64_t r) {
  float2 v;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(v.x), "=f"(v.y) : "l"(r));
  return v;
}
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Two 16-bit values of one 32-bit word as a packed fp32 pair (element order kept).
template <bool BF16>
__device__ __forceinline__ uint64_t widen2(uint32_t w) {
  if constexpr (BF16) {
    return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    const float2 t = __half22float2(*reinterpret_cast<const __half2 *>(&w));
    return f2(t.x, t.y);
  }
}

template <bool BF16>
__device__ __forceinline__ void store_out(void *base, int64_t idx, float x) {
  if constexpr (BF16)
    reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
  else
    reinterpret_cast<__half *>(base)[idx] = __float2half_rn(x);
}

// Byte offset of 16-byte chunk c (of CPR) of row r inside a stage tensor laid
// out as KCH boxes of [kTok rows][128 B] with the 128-byte TMA swizzle.
__device__ __forceinline__ uint32_t swz(int r, int c) {
  return static_cast<uint32_t>((c >> 3) * (kTok * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, int d, int n, int h, int b,
                                         uint32_t slots, uint32_t bar) {
  const int sn = slots & 3, sh = (slots >> 2) & 3;
  const int c1 = (sn == 1) ? n : (sh == 1) ? h : b;
  const int c2 = (sn == 2) ? n : (sh == 2) ? h : b;
  const int c3 = (sn == 3) ? n : (sh == 3) ? h : b;
  tma_load_4d(dst, map, d, c1, c2, c3, bar);
}

// PAGED: the cache is a pool of pages (num_pages, H_kv, page_size, D); request
// b's tokens sit in the pages listed by block_table[b] and its length is
// cache_lens[b].  A stage is loaded as 64 / min(page_size, 64) boxes, one per
// page it touches, and only for rows below the request's length.
template <int D, int GH, bool BF16, bool PAGED>
__global__ void __launch_bounds__(kThreads, 2)
    decode_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                        const __grid_constant__ DecodeParams p) {
  using C = DecCfg<D, GH>;
  extern __shared__ uint8_t smem_raw[];
  griddep_wait();  // before any global memory access (launched with programmatic serialization)
  if (load_volatile(p.err) != 0) return;

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (sbase - raw);
  float *sq = reinterpret_cast<float *>(smem + C::OFF_Q);
  float *sp = reinterpret_cast<float *>(smem + C::OFF_P);
  float *sm_m = reinterpret_cast<float *>(smem + C::OFF_ML);
  float *sm_l = sm_m + kConsumerWarps * GH;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto FULL = [&](int s) -> uint32_t { return bar0 + 8u * s; };
  auto EMPTY = [&](int s) -> uint32_t { return bar0 + 8u * (kStages + s); };
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC);

  const int split = blockIdx.x;
  const int hk = blockIdx.y / p.nhc, hc = blockIdx.y % p.nhc;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h_first = hk * p.group + hc * GH;
  const int nh = min(GH, p.group - hc * GH);
  int len = p.cache_len;
  if constexpr (PAGED) {
    len = p.cache_lens[b];
    if (len < 0 || len > p.cache_len) {
      if (threadIdx.x == 0) atomicOr(p.err, kErrBadIndex);
      len = len < 0 ? 0 : p.cache_len;
    }
  }
  // Sliding window: only keys t >= t_lo are attended; the splits tile the
  // range from t_lo rounded down to a whole stage (so that paged boxes stay
  // inside their pages), and keys below t_lo are masked.
  const int t_lo = p.window_left >= 0 ? max(0, len - 1 - p.window_left) : 0;
  const int t_begin = (t_lo / kTok) * kTok + split * p.chunk;
  const int t_end = min(t_begin + p.chunk, len);
  const int n_tiles = t_end > t_begin ? (t_end - t_begin + kTok - 1) / kTok : 0;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(FULL(s), 1);
      mbar_init(EMPTY(s), kConsumerWarps);
    }
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  // Query rows of this CTA's heads, pre-multiplied by scale * log2(e).
  auto q_at = [&](int i, int d) -> float {
    if (i >= nh) return 0.f;
    const int64_t off = static_cast<int64_t>(b) * p.q_sb + static_cast<int64_t>(h_first + i) * p.q_sh + d;
    if constexpr (BF16)
      return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p.q)[off]);
    else
      return __half2float(reinterpret_cast<const __half *>(p.q)[off]);
  };
  if (p.rope == 0) {
    for (int idx = threadIdx.x; idx < GH * D; idx += kThreads) sq[idx] = q_at(idx / D, idx % D) * p.scale_log2;
  } else {
    // Rotary embeddings: the query sits at position len - 1 (the keys in the
    // cache were rotated when they were written); one pair per thread.
    const uint32_t qpos = static_cast<uint32_t>(len > 0 ? len - 1 : 0);
    for (int idx = threadIdx.x; idx < GH * (D / 2); idx += kThreads) {
      const int i = idx / (D / 2), c = idx % (D / 2);
      const int da = p.rope == 2 ? 2 * c : c, db = p.rope == 2 ? 2 * c + 1 : c + D / 2;
      float sn, cs;
      rope_sincos(qpos, p.rope_f[c], &sn, &cs);
      const float xa = q_at(i, da), xb = q_at(i, db);
      sq[i * D + da] = fmaf(xa, cs, -xb * sn) * p.scale_log2;
      sq[i * D + db] = fmaf(xb, cs, xa * sn) * p.scale_log2;
    }
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < n_tiles; ++j) {
        const int st = j % kStages;
        const uint32_t dst = sbase + st * C::STAGE_BYTES;
        const int t0 = t_begin + j * kTok;
        // Paged: this stage's page ids are read before the wait for a free
        // stage, so their latency hides behind it.
        constexpr int kMaxBox = kTok / 16;
        int pg[kMaxBox];
        int rows = kTok, nbox = 1;
        if constexpr (PAGED) {
          rows = p.page_size < kTok ? p.page_size : kTok;
          nbox = (min(t_end - t0, kTok) + rows - 1) / rows;
#pragma unroll
          for (int x = 0; x < kMaxBox; ++x) {
            const int pidx = (t0 + x * rows) / p.page_size;
            pg[x] = (x < nbox && pidx < p.max_pages) ? __ldg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + pidx)
                                                    : -1;
          }
        }
        if (j >= kStages && !(ok = mbar_wait(EMPTY(st), ((j / kStages) - 1) & 1, abort_flag, p.err))) break;
        if constexpr (!PAGED) {
          mbar_arrive_expect_tx(FULL(st), C::STAGE_BYTES);
#pragma unroll
          for (int c = 0; c < C::KCH; ++c) {
            tma_tile(dst + c * C::BOX_BYTES, &tmK, c * 64, t0, hk, b, p.slots_k, FULL(st));
            tma_tile(dst + C::KV_BYTES + c * C::BOX_BYTES, &tmV, c * 64, t0, hk, b, p.slots_v, FULL(st));
          }
        } else {
          // Boxes of `rows` tokens, each inside one page; rows past the length
          // are not loaded (the consumers mask them), so the stage expects only
          // the bytes of the boxes issued.
          mbar_arrive_expect_tx(FULL(st), static_cast<uint32_t>(nbox * rows) * (2u * D * 2u));
#pragma unroll
          for (int x = 0; x < kMaxBox; ++x) {
            if (x >= nbox) break;
            int page = pg[x];
            if (page < 0 || page >= p.num_pages) {
              atomicOr(p.err, kErrBadIndex);
              page = p.num_pages;  // out of the tensor map: the box reads as zeros
            }
            const int row = (t0 + x * rows) % p.page_size;
            const uint32_t off = static_cast<uint32_t>(x * rows * 128);
#pragma unroll
            for (int c = 0; c < C::KCH; ++c) {
              tma_tile(dst + c * C::BOX_BYTES + off, &tmK, c * 64, row, hk, page, p.slots_k, FULL(st));
              tma_tile(dst + C::KV_BYTES + c * C::BOX_BYTES + off, &tmV, c * 64, row, hk, page, p.slots_v, FULL(st));
            }
          }
        }
        ++issued;
      }
      if (!ok) {
        for (int i = max(0, issued - kStages); i < issued; ++i)
          mbar_wait(FULL(i % kStages), (i / kStages) & 1, nullptr, p.err);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ consumer warps
    const int tl = lane & 15;           // token of this lane within the warp's 16 (scores)
    const int half = lane >> 4;         // which half of D this lane's score covers
    const int row = warp * kTokPerWarp + tl;
    const int slot = lane / C::CPR;     // token slot for P . V
    const int sub = lane % C::CPR;      // 16-byte slice of D for P . V
    float m[GH];
    float lpart[GH];
    float slope2[GH];  // ALiBi slope of each head, base-2 units (0 without ALiBi)
#pragma unroll
    for (int i = 0; i < GH; ++i)
      slope2[i] = (p.alibi_slopes != nullptr && i < nh) ? p.alibi_slopes[h_first + i] * 1.4426950408889634f : 0.f;
    uint64_t acc[GH][4];
#pragma unroll
    for (int i = 0; i < GH; ++i) {
      m[i] = -INFINITY;
      lpart[i] = 0.f;
#pragma unroll
      for (int e = 0; e < 4; ++e) acc[i][e] = 0;  // +0.0f, +0.0f
    }
    float *pw = sp + warp * kTokPerWarp * GH;
    bool ok = true;
    for (int j = 0; j < n_tiles; ++j) {
      const int st = j % kStages;
      ok = __all_sync(0xffffffffu, mbar_wait(FULL(st), (j / kStages) & 1, abort_flag, p.err));
      if (!ok) break;
      const uint8_t *sk = smem + st * C::STAGE_BYTES;
      const uint8_t *sv = sk + C::KV_BYTES;

      // scores of this lane's token over its half of D
      uint64_t s2[GH];
#pragma unroll
      for (int i = 0; i < GH; ++i) s2[i] = 0;
#pragma unroll
      for (int cc = 0; cc < C::CPR / 2; ++cc) {
        const int c = half * (C::CPR / 2) + cc;
        const uint4 kw = *reinterpret_cast<const uint4 *>(sk + swz(row, c));
        const uint64_t k01 = widen2<BF16>(kw.x), k23 = widen2<BF16>(kw.y);
        const uint64_t k45 = widen2<BF16>(kw.z), k67 = widen2<BF16>(kw.w);
#pragma unroll
        for (int i = 0; i < GH; ++i) {
          const ulonglong2 qa = *reinterpret_cast<const ulonglong2 *>(sq + i * D + c * 8);
          const ulonglong2 qb = *reinterpret_cast<const ulonglong2 *>(sq + i * D + c * 8 + 4);
          s2[i] = ffma2(qa.x, k01, s2[i]);
          s2[i] = ffma2(qa.y, k23, s2[i]);
          s2[i] = ffma2(qb.x, k45, s2[i]);
          s2[i] = ffma2(qb.y, k67, s2[i]);
        }
      }
      const int tok = t_begin + j * kTok + row;
      const bool valid = tok < t_end && tok >= t_lo;
      const float dist = static_cast<float>(len - 1 - tok);  // query position minus key position
      float s[GH];
#pragma unroll
      for (int i = 0; i < GH; ++i) {
        const float2 v = unf2(s2[i]);
        float x = v.x + v.y;
        x += __shfl_xor_sync(0xffffffffu, x, 16);
        s[i] = valid ? fmaf(-slope2[i], dist, x) : -INFINITY;
      }
      // online softmax over this warp's 16 tokens (both halves hold the same scores)
      float pr[GH];
#pragma unroll
      for (int i = 0; i < GH; ++i) {
        float mx = s[i];
#pragma unroll
        for (int off = 8; off >= 1; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float m_new = fmaxf(m[i], mx);
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = fast_exp2(m[i] - m_use);
        pr[i] = fast_exp2(s[i] - m_use);
        lpart[i] = lpart[i] * alpha + (half == 0 ? pr[i] : 0.f);
        const uint64_t a2 = f2(alpha, alpha);
#pragma unroll
        for (int e = 0; e < 4; ++e) acc[i][e] = fmul2(acc[i][e], a2);
        m[i] = m_new;
      }
      if (half == 0) {
#pragma unroll
        for (int i = 0; i < GH; ++i) pw[tl * GH + i] = pr[i];
      }
      __syncwarp();
      // P . V over the warp's 16 tokens
#pragma unroll
      for (int it = 0; it < kTokPerWarp / C::TPI; ++it) {
        const int t = it * C::TPI + slot;
        const int r2 = warp * kTokPerWarp + t;
        uint4 vw = *reinterpret_cast<const uint4 *>(sv + swz(r2, sub));
        if constexpr (PAGED) {
          // Rows past the length were not loaded: keep stale bytes out of P V.
          if (t_begin + j * kTok + r2 >= t_end) vw = make_uint4(0, 0, 0, 0);
        }
        const uint64_t v01 = widen2<BF16>(vw.x), v23 = widen2<BF16>(vw.y);
        const uint64_t v45 = widen2<BF16>(vw.z), v67 = widen2<BF16>(vw.w);
#pragma unroll
        for (int i = 0; i < GH; ++i) {
          const float pv = pw[t * GH + i];
          const uint64_t p2 = f2(pv, pv);
          acc[i][0] = ffma2(p2, v01, acc[i][0]);
          acc[i][1] = ffma2(p2, v23, acc[i][1]);
          acc[i][2] = ffma2(p2, v45, acc[i][2]);
          acc[i][3] = ffma2(p2, v67, acc[i][3]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(EMPTY(st));
    }
    // per-warp sum of the partial row sums
#pragma unroll
    for (int i = 0; i < GH; ++i) {
      float x = lpart[i];
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
      lpart[i] = x;
    }
    if (lane == 0) {
#pragma unroll
      for (int i = 0; i < GH; ++i) {
        sm_m[warp * GH + i] = ok ? m[i] : -INFINITY;
        sm_l[warp * GH + i] = ok ? lpart[i] : 0.f;
      }
    }
    // Every stage this CTA loaded has been consumed, so the ring is idle; wait
    // for all consumers to be past it before reusing it for the merge.
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    float *mg = reinterpret_cast<float *>(smem);  // [warps][TPI][GH][D]
#pragma unroll
    for (int i = 0; i < GH; ++i)
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 v = unf2(acc[i][e]);
        float *dst = mg + ((warp * C::TPI + slot) * GH + i) * D + sub * 8 + 2 * e;
        dst[0] = v.x;
        dst[1] = v.y;
      }
    asm volatile("bar.sync 1, %0;" ::"r"(kConsumerWarps * 32) : "memory");
    for (int idx = threadIdx.x; idx < nh * D; idx += kConsumerWarps * 32) {
      const int i = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, sm_m[w * GH + i]);
      const float M_use = (M == -INFINITY) ? 0.f : M;
      float L = 0.f, A = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float wt = fast_exp2(sm_m[w * GH + i] - M_use);
        L = fmaf(sm_l[w * GH + i], wt, L);
        float a = 0.f;
#pragma unroll
        for (int sl = 0; sl < C::TPI; ++sl) a += mg[((w * C::TPI + sl) * GH + i) * D + d];
        A = fmaf(a, wt, A);
      }
      const int hq = h_first + i;
      const float o = (L > 0.f) ? A / L : 0.f;
      const float lse = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
      if (p.nsplit == 1) {
        store_out<BF16>(p.o, static_cast<int64_t>(b) * p.o_sb + static_cast<int64_t>(hq) * p.o_sh + d, o);
        if (d == 0 && p.lse != nullptr) p.lse[static_cast<int64_t>(b) * p.Hq + hq] = lse;
      } else {
        const int64_t r = (static_cast<int64_t>(b) * p.Hq + hq) * p.nsplit + split;
        p.ws_o[r * D + d] = o;
        if (d == 0) p.ws_lse[r] = lse;
      }
    }
  }
}

// Merge of one (b, q head): O = sum_s w_s O_s / sum_s w_s and LSE = M + ln
// sum_s w_s, with w_s = exp(lse_s - M) and M the largest partial LSE.  One
// thread per output column.  Each partial LSE is read by one thread (nsplit <=
// 64 <= D) and the weights are shared, and the partial outputs are read in
// batches of 8 independent loads: a handful of memory round trips, not two
// per split.  The sums run in split order, as a plain loop would.
template <int D, bool BF16>
__global__ void __launch_bounds__(D) decode_merge_kernel(const DecodeParams p) {
  constexpr int kWarps = D / 32;
  __shared__ float w_s[64];
  __shared__ float red[kWarps];
  __shared__ int stop;
  griddep_wait();
  const int bh = blockIdx.x;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int d = threadIdx.x, lane = d & 31, warp = d >> 5;
  if (d == 0) stop = load_volatile(p.err) != 0;
  __syncthreads();
  if (stop) return;
  const int nsplit = p.nsplit;
  const float *ls = p.ws_lse + static_cast<int64_t>(bh) * nsplit;
  const float *os = p.ws_o + static_cast<int64_t>(bh) * nsplit * D;
  const float l = d < nsplit ? ls[d] : -INFINITY;
  float m = l;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) red[warp] = m;
  __syncthreads();
  float M = red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, red[w]);
  if (d < nsplit) w_s[d] = M == -INFINITY ? 0.f : expf(l - M);
  __syncthreads();
  float W = 0.f, A = 0.f;
  for (int s0 = 0; s0 < nsplit; s0 += 8) {
    float o8[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) o8[i] = s0 + i < nsplit ? os[static_cast<int64_t>(s0 + i) * D + d] : 0.f;
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      if (s0 + i < nsplit) {
        W += w_s[s0 + i];
        A = fmaf(w_s[s0 + i], o8[i], A);
      }
    }
  }
  store_out<BF16>(p.o, static_cast<int64_t>(b) * p.o_sb + static_cast<int64_t>(hq) * p.o_sh + d,
                  W > 0.f ? A / W : 0.f);
  if (d == 0 && p.lse != nullptr) p.lse[bh] = W > 0.f ? M + logf(W) : -INFINITY;
}

__global__ void __launch_bounds__(256) kv_cache_write_kernel(const KvWriteParams p) {
  griddep_wait();
  if (load_volatile(p.err) != 0) return;
  const int pieces = p.D / 8;  // 16-byte pieces per row
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < 2 * p.total_units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_v = u >= p.total_units;
    int64_t x = is_v ? u - p.total_units : u;
    const int e = static_cast<int>(x % pieces) * 8;
    x /= pieces;
    const int t = static_cast<int>(x % p.n_new);
    x /= p.n_new;
    const int hk = static_cast<int>(x % p.Hkv);
    const int64_t b = x / p.Hkv;
    const char *src;
    char *dst;
    if (!is_v) {
      src = reinterpret_cast<const char *>(p.kn) + 2 * (b * p.kn_sb + hk * p.kn_sh + t * p.kn_sn + e);
      dst = reinterpret_cast<char *>(p.kc) + 2 * (b * p.kc_sb + hk * p.kc_sh + (p.pos + t) * p.kc_sn + e);
    } else {
      src = reinterpret_cast<const char *>(p.vn) + 2 * (b * p.vn_sb + hk * p.vn_sh + t * p.vn_sn + e);
      dst = reinterpret_cast<char *>(p.vc) + 2 * (b * p.vc_sb + hk * p.vc_sh + (p.pos + t) * p.vc_sn + e);
    }
    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
  }
}

// Paged cache write: token t of request b goes to position positions[b] + t,
// i.e. row (pos % page_size) of page block_table[b][pos / page_size].  A page
// id or position out of range skips the write and records kErrBadIndex.
__global__ void __launch_bounds__(256) kv_cache_write_paged_kernel(const KvWriteParams p) {
  griddep_wait();
  if (load_volatile(p.err) != 0) return;
  const int pieces = p.D / 8;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < 2 * p.total_units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_v = u >= p.total_units;
    int64_t x = is_v ? u - p.total_units : u;
    const int e = static_cast<int>(x % pieces) * 8;
    x /= pieces;
    const int t = static_cast<int>(x % p.n_new);
    x /= p.n_new;
    const int hk = static_cast<int>(x % p.Hkv);
    const int64_t b = x / p.Hkv;
    const int pos = p.positions[b] + t;
    const int pidx = pos >= 0 ? pos / p.page_size : -1;
    const int page = (pidx >= 0 && pidx < p.max_pages) ? p.block_table[b * p.bt_stride + pidx] : -1;
    if (page < 0 || page >= p.num_pages) {
      atomicOr(p.err, kErrBadIndex);
      continue;
    }
    const int row = pos % p.page_size;
    const char *src;
    char *dst;
    if (!is_v) {
      src = reinterpret_cast<const char *>(p.kn) + 2 * (b * p.kn_sb + hk * p.kn_sh + t * p.kn_sn + e);
      dst = reinterpret_cast<char *>(p.kc) + 2 * (page * p.kc_sb + hk * p.kc_sh + row * p.kc_sn + e);
    } else {
      src = reinterpret_cast<const char *>(p.vn) + 2 * (b * p.vn_sb + hk * p.vn_sh + t * p.vn_sn + e);
      dst = reinterpret_cast<char *>(p.vc) + 2 * (page * p.vc_sb + hk * p.vc_sh + row * p.vc_sn + e);
    }
    *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
  }
}

// Cache write with rotary embeddings: new keys are rotated at the cache
// position they are written to (dense: pos + t; paged: positions[b] + t), one
// group of 8 coordinate pairs (two 16-byte pieces) per thread; values are
// copied as they are, one 16-byte piece per thread.  A paged write whose page
// index or page id is out of range is skipped and recorded as kErrBadIndex.
template <bool PAGED, bool BF16>
__global__ void __launch_bounds__(256) kv_cache_write_rope_kernel(const __grid_constant__ KvWriteParams p) {
  griddep_wait();
  if (load_volatile(p.err) != 0) return;
  const int pieces = p.D / 8;   // 16-byte pieces per row
  const int groups = p.D / 16;  // groups of 8 pairs per key row
  const int64_t rows = p.total_units / pieces;  // B * H_kv * n_new
  const int64_t k_units = rows * groups;
  const bool inter = p.rope == 2;
  for (int64_t u = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; u < k_units + p.total_units;
       u += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const bool is_v = u >= k_units;
    int64_t x = is_v ? u - k_units : u;
    const int part = static_cast<int>(x % (is_v ? pieces : groups));
    x /= is_v ? pieces : groups;
    const int t = static_cast<int>(x % p.n_new);
    x /= p.n_new;
    const int hk = static_cast<int>(x % p.Hkv);
    const int64_t b = x / p.Hkv;
    int pos = p.pos + t;
    int64_t row_c;  // cache row offset in elements (page, head, row) or (batch, head, position)
    if constexpr (PAGED) {
      pos = p.positions[b] + t;
      const int pidx = pos >= 0 ? pos / p.page_size : -1;
      const int page = (pidx >= 0 && pidx < p.max_pages) ? p.block_table[b * p.bt_stride + pidx] : -1;
      if (page < 0 || page >= p.num_pages) {
        atomicOr(p.err, kErrBadIndex);
        continue;
      }
      const int r = pos % p.page_size;
      row_c = is_v ? page * p.vc_sb + hk * p.vc_sh + r * p.vc_sn : page * p.kc_sb + hk * p.kc_sh + r * p.kc_sn;
    } else {
      row_c = is_v ? b * p.vc_sb + hk * p.vc_sh + pos * p.vc_sn : b * p.kc_sb + hk * p.kc_sh + pos * p.kc_sn;
    }
    if (is_v) {
      const char *src = reinterpret_cast<const char *>(p.vn) + 2 * (b * p.vn_sb + hk * p.vn_sh + t * p.vn_sn + part * 8);
      char *dst = reinterpret_cast<char *>(p.vc) + 2 * (row_c + part * 8);
      *reinterpret_cast<uint4 *>(dst) = *reinterpret_cast<const uint4 *>(src);
      continue;
    }
    const int ca = inter ? 2 * part : part, cb = inter ? 2 * part + 1 : part + p.D / 16;
    const char *src = reinterpret_cast<const char *>(p.kn) + 2 * (b * p.kn_sb + hk * p.kn_sh + t * p.kn_sn);
    char *dst = reinterpret_cast<char *>(p.kc) + 2 * row_c;
    uint4 A = *reinterpret_cast<const uint4 *>(src + 16 * ca), Bv = *reinterpret_cast<const uint4 *>(src + 16 * cb);
    float cs[8], sn[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) rope_sincos(static_cast<uint32_t>(pos), p.rope_f[8 * part + i], &sn[i], &cs[i]);
    if (inter) rope_rotate_group<BF16, true>(A, Bv, cs, sn);
    else rope_rotate_group<BF16, false>(A, Bv, cs, sn);
    *reinterpret_cast<uint4 *>(dst + 16 * ca) = A;
    *reinterpret_cast<uint4 *>(dst + 16 * cb) = Bv;
  }
}

// Launches with programmatic stream serialization: the kernel's blocks may be
// scheduled while the preceding kernel of the stream drains, which hides the
// launch gap between the short kernels of a decode step.  Every kernel launched
// this way calls griddep_wait() before it touches global memory, so it reads
// and writes nothing the preceding kernel is still using.
template <typename... Params, typename... Args>
cudaError_t launch_serialized(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                              Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, std::forward<Args>(args)...);
}

template <int D, int GH, bool BF16, bool PAGED>
cudaError_t launch_split(const CUtensorMap &tk, const CUtensorMap &tv, const DecodeParams &p, int B, int Hkv,
                         cudaStream_t stream) {
  using C = DecCfg<D, GH>;
  auto kern = decode_split_kernel<D, GH, BF16, PAGED>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(C::SMEM_BYTES));
  if (e != cudaSuccess) return e;
  dim3 grid(p.nsplit, Hkv * p.nhc, B);
  if (p.nsplit > 64 || p.nsplit > D) return cudaErrorInvalidValue;  // the merge holds one weight per thread
  e = launch_serialized(kern, grid, dim3(kThreads), C::SMEM_BYTES, stream, tk, tv, p);
  if (e != cudaSuccess || p.nsplit == 1) return e;
  return launch_serialized(decode_merge_kernel<D, BF16>, dim3(B * p.Hq), dim3(D), 0, stream, p);
}

}  // namespace

int decode_heads_per_cta(int group) {
  if (group <= 1) return 1;
  if (group <= 2) return 2;
  if (group <= 4) return 4;
  return 8;
}

cudaError_t launch_decode(int D, bool bf16, bool paged, int gh, const CUtensorMap &tk, const CUtensorMap &tv,
                          const DecodeParams &p, int B, int Hkv, cudaStream_t stream) {
#define ATTN_DECODE_CASE(DD, GG, BB)                                                             \
  if (D == DD && gh == GG && bf16 == BB)                                                         \
    return paged ? launch_split<DD, GG, BB, true>(tk, tv, p, B, Hkv, stream)                     \
                 : launch_split<DD, GG, BB, false>(tk, tv, p, B, Hkv, stream);
#define ATTN_DECODE_GH(DD, BB) \
  ATTN_DECODE_CASE(DD, 1, BB) ATTN_DECODE_CASE(DD, 2, BB) ATTN_DECODE_CASE(DD, 4, BB) ATTN_DECODE_CASE(DD, 8, BB)
  ATTN_DECODE_GH(128, true)
  ATTN_DECODE_GH(128, false)
  ATTN_DECODE_GH(64, true)
  ATTN_DECODE_GH(64, false)
#undef ATTN_DECODE_GH
#undef ATTN_DECODE_CASE
  return cudaErrorInvalidValue;
}

cudaError_t launch_kv_cache_write(const KvWriteParams &p, bool paged, cudaStream_t stream) {
  const int64_t work = p.rope ? p.total_units * 3 / 2 : 2 * p.total_units;
  int64_t blocks = (work + 255) / 256;
  if (blocks > 65535 * 8) blocks = 65535 * 8;
  const dim3 grid(static_cast<unsigned>(blocks));
  if (p.rope) {
    if (paged)
      return p.is_bf16 ? launch_serialized(kv_cache_write_rope_kernel<true, true>, grid, dim3(256), 0, stream, p)
                       : launch_serialized(kv_cache_write_rope_kernel<true, false>, grid, dim3(256), 0, stream, p);
    return p.is_bf16 ? launch_serialized(kv_cache_write_rope_kernel<false, true>, grid, dim3(256), 0, stream, p)
                     : launch_serialized(kv_cache_write_rope_kernel<false, false>, grid, dim3(256), 0, stream, p);
  }
  return launch_serialized(paged ? kv_cache_write_paged_kernel : kv_cache_write_kernel, grid, dim3(256), 0, stream,
                           p);
}

}  // namespace attn
