// prefill.cu -- fused attention forward (prefill) for sm_103a.
//
// One CTA computes one 128-row query tile of one (batch, q-head):
//   warp 0      TMA producer: Q tile once, then K and V tiles of 128 keys into
//               a ring of shared-memory stages (128-byte swizzled).
//   warp 1      TMEM allocator and tcgen05 MMA issuer (one thread):
//                 S_j  = Q K_j^T        (SS form, fp32 in TMEM, double-buffered)
//                 O   += P_j V_j        (TS form, P read from TMEM)
//   warps 2..5  softmax warpgroup, one thread per query row (TMEM lane):
//               mask, row max, online-softmax update, P = exp2(S - m) packed
//               to 16-bit into TMEM, rescale of O by alpha, final O / l and LSE.
//
// The algorithm is the online softmax of "Skill: Write a Triton Attention
// Kernel" (Required reasoning process, steps 4-9): running max m and sum l in
// fp32, alpha = exp(m_old - m_new) applied to O and l before the new block is
// added, O / l once after the loop, lse = m + ln l.  Scores are kept in base-2
// units (scale * log2 e folded into one multiply) so exp becomes ex2; the LSE
// is converted back to natural log on store.  The causal mask (key j kept for
// query i iff j <= i) and the key-length mask set scores to -inf before the
// max, and only tiles that straddle the diagonal or the end of the keys pay
// for it; tiles past the diagonal are never loaded (loop bound
// min(N_kv, q0 + 128)).
//
// TMEM columns (512 allocated): S0 [0,128) S1 [128,256) O [256,256+D)
// P0 [256+D, 320+D) P1 [320+D, 384+D).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kBM = kPrefillBM;
constexpr int kBN = kPrefillBN;
constexpr int kThreads = 192;
constexpr float kLn2 = 0.693147180559945309f;

template <int D>
struct Cfg {
  static constexpr int KCH = D / 64;                  // 128-byte chunks along D
  static constexpr int ST = (D == 128) ? 2 : 3;       // K/V pipeline stages
  static constexpr uint32_t CHUNK_Q = kBM * 128;      // bytes of one 64-column chunk of Q
  static constexpr uint32_t CHUNK_KV = kBN * 128;
  static constexpr uint32_t Q_BYTES = kBM * D * 2;
  static constexpr uint32_t KV_BYTES = kBN * D * 2;
  static constexpr uint32_t S_COL0 = 0, S_COL1 = 128, O_COL = 256;
  static constexpr uint32_t P_COL0 = 256 + D, P_COL1 = 256 + D + kBN / 2;
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + Q_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + ST * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + ST * KV_BYTES;
  // barrier indices
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;            // + stage
  static constexpr int B_KE = 1 + ST;       // + stage
  static constexpr int B_VF = 1 + 2 * ST;   // + stage
  static constexpr int B_VE = 1 + 3 * ST;   // + stage
  static constexpr int B_SF = 1 + 4 * ST;   // + buffer (2)
  static constexpr int B_PF = 3 + 4 * ST;   // + buffer (2)
  static constexpr int B_OR = 5 + 4 * ST;   // O += P V completed
  static constexpr int B_DONE = 6 + 4 * ST; // every MMA completed
  static constexpr int NBAR = 7 + 4 * ST;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_USED = OFF_MISC + 16;
  // + slack for 1024-byte alignment; at least 116 KB so that only one CTA (which
  // holds all 512 TMEM columns) is resident per SM.
  static constexpr uint32_t SMEM_BYTES = (SMEM_USED + 1024 > 116u * 1024) ? SMEM_USED + 1024 : 116u * 1024;
  static_assert(P_COL1 + kBN / 2 <= TMEM_COLS, "TMEM budget");
};

__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, int d, int n, int h, int b,
                                         uint32_t slots, uint32_t bar) {
  const int sn = slots & 3, sh = (slots >> 2) & 3;
  const int c1 = (sn == 1) ? n : (sh == 1) ? h : b;
  const int c2 = (sn == 2) ? n : (sh == 2) ? h : b;
  const int c3 = (sn == 3) ? n : (sh == 3) ? h : b;
  tma_load_4d(dst, map, d, c1, c2, c3, bar);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  }
}

template <int D, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const PrefillParams p) {
  using C = Cfg<D>;
  constexpr int ST = C::ST;
  extern __shared__ uint8_t smem_raw[];

  if (load_volatile(p.err) != 0) return;  // an earlier launch failed; nothing runs until it is read

  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (sbase - raw);
  const uint32_t sQ = sbase + C::OFF_Q, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qt = CAUSAL ? (p.n_qtiles - 1 - static_cast<int>(blockIdx.x)) : static_cast<int>(blockIdx.x);
  const int h = blockIdx.y, b = blockIdx.z;
  const int hk = h / p.group;
  const int q0 = qt * kBM;
  const int kv_end = CAUSAL ? min(p.Nkv, q0 + kBM) : p.Nkv;
  const int n_kv = (kv_end + kBN - 1) / kBN;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_Q), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_KE + s), 1);
      mbar_init(BAR(C::B_VF + s), 1);
      mbar_init(BAR(C::B_VE + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(C::B_SF + i), 1);
      mbar_init(BAR(C::B_PF + i), 4);  // one arrival per softmax warp
    }
    mbar_init(BAR(C::B_OR), 1);
    mbar_init(BAR(C::B_DONE), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      int issued_k = 0, issued_v = 0;
      bool ok = true;
      mbar_arrive_expect_tx(BAR(C::B_Q), C::Q_BYTES);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c)
        tma_tile(sQ + c * C::CHUNK_Q, &tmQ, c * 64, q0, h, b, p.slots_q, BAR(C::B_Q));
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % ST;
        const uint32_t ph = (j / ST) & 1;
        if (j >= ST && !(ok = mbar_wait(BAR(C::B_KE + st), ph ^ 1, abort_flag, p.err))) break;
        mbar_arrive_expect_tx(BAR(C::B_KF + st), C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_tile(sK + st * C::KV_BYTES + c * C::CHUNK_KV, &tmK, c * 64, j * kBN, hk, b, p.slots_k,
                   BAR(C::B_KF + st));
        ++issued_k;
        if (j >= ST && !(ok = mbar_wait(BAR(C::B_VE + st), ph ^ 1, abort_flag, p.err))) break;
        mbar_arrive_expect_tx(BAR(C::B_VF + st), C::KV_BYTES);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c)
          tma_tile(sV + st * C::KV_BYTES + c * C::CHUNK_KV, &tmV, c * 64, j * kBN, hk, b, p.slots_v,
                   BAR(C::B_VF + st));
        ++issued_v;
      }
      if (!ok) {
        // Let every copy already issued land before shared memory is released.
        mbar_wait(BAR(C::B_Q), 0, nullptr, p.err);
        for (int i = max(0, issued_k - ST); i < issued_k; ++i)
          mbar_wait(BAR(C::B_KF + i % ST), (i / ST) & 1, nullptr, p.err);
        for (int i = max(0, issued_v - ST); i < issued_v; ++i)
          mbar_wait(BAR(C::B_VF + i % ST), (i / ST) & 1, nullptr, p.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_qk = idesc_f16(BF16, kBM, kBN, false, false);
      constexpr uint32_t idesc_pv = idesc_f16(BF16, kBM, D, false, true);
      auto issue_pv = [&](int i) -> bool {
        const int st = i % ST;
        const int pb = i & 1;
        if (!mbar_wait(BAR(C::B_PF + pb), (i >> 1) & 1, abort_flag, p.err)) return false;
        if (!mbar_wait(BAR(C::B_VF + st), (i / ST) & 1, abort_flag, p.err)) return false;
        tc_fence_after();
        const uint32_t vbase = sV + st * C::KV_BYTES;
        const uint32_t pcol = tmem + (pb ? C::P_COL1 : C::P_COL0);
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          // V is MN-major: 16 keys per MMA = 16 rows of 128 B; D in 64-column blocks CHUNK_KV apart.
          const uint64_t bdesc = smem_desc_sw128(vbase + kk * 16 * 128, C::CHUNK_KV, 1024);
          mma_ts(tmem + C::O_COL, pcol + kk * 8, bdesc, idesc_pv, (i > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(BAR(C::B_VE + st));
        tc_commit(BAR(C::B_OR));
        return true;
      };
      bool ok = mbar_wait(BAR(C::B_Q), 0, abort_flag, p.err);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % ST;
        const int sb = j & 1;
        if (!(ok = mbar_wait(BAR(C::B_KF + st), (j / ST) & 1, abort_flag, p.err))) break;
        tc_fence_after();
        const uint32_t kbase = sK + st * C::KV_BYTES;
        const uint32_t scol = tmem + (sb ? C::S_COL1 : C::S_COL0);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          // Q and K are K-major: 16 elements (32 B) per MMA inside a 128-byte swizzle row.
          const uint64_t adesc = smem_desc_sw128(sQ + (kk / 4) * C::CHUNK_Q + (kk % 4) * 32, 16, 1024);
          const uint64_t bdesc = smem_desc_sw128(kbase + (kk / 4) * C::CHUNK_KV + (kk % 4) * 32, 16, 1024);
          mma_ss(scol, adesc, bdesc, idesc_qk, kk > 0 ? 1u : 0u);
        }
        tc_commit(BAR(C::B_SF + sb));
        tc_commit(BAR(C::B_KE + st));
        if (j > 0) ok = issue_pv(j - 1);
      }
      if (ok) issue_pv(n_kv - 1);
      tc_commit(BAR(C::B_DONE));
      mbar_wait(BAR(C::B_DONE), 0, nullptr, p.err);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroup
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                 // query row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int q_row = q0 + r;
    const float sl2 = p.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_SF + sb), (j >> 1) & 1, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      uint32_t sr[4][32];
      const uint32_t scol = tmem + lane_off + (sb ? C::S_COL1 : C::S_COL0);
#pragma unroll
      for (int i = 0; i < 4; ++i) tmem_ld_32x32b_x32(scol + i * 32, sr[i]);
      tmem_wait_ld();
#pragma unroll
      for (int i = 0; i < 4; ++i) reg_fence(sr[i]);

      const int kv0 = j * kBN;
      const bool need_mask = (kv0 + kBN > p.Nkv) || (CAUSAL && kv0 + kBN - 1 > q0);
      float mx = -INFINITY;
      if (need_mask) {
        const int lim = (CAUSAL ? min(p.Nkv, q_row + 1) : p.Nkv) - kv0;  // columns c < lim are kept
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            float x = __uint_as_float(sr[i][c]);
            x = (i * 32 + c < lim) ? x : -INFINITY;
            sr[i][c] = __float_as_uint(x);
            mx = fmaxf(mx, x);
          }
      } else {
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 32; ++c) mx = fmaxf(mx, __uint_as_float(sr[i][c]));
      }
      const float m_new = fmaxf(m, mx * sl2);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = fast_exp2(m - m_use);
      float rs = 0.f;
      uint32_t pk[2][32];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const float p0 = fast_exp2(fmaf(__uint_as_float(sr[i][c]), sl2, -m_use));
          const float p1 = fast_exp2(fmaf(__uint_as_float(sr[i][c + 1]), sl2, -m_use));
          rs += p0 + p1;
          pk[i >> 1][(i & 1) * 16 + c / 2] = pack2<BF16>(p0, p1);
        }
      l = l * alpha + rs;
      m = m_new;

      if (j > 0) {
        // O += P_{j-1} V_{j-1} must have completed before O is rescaled and before
        // this P buffer (last read by P_{j-2} V_{j-2}) is overwritten.
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_OR), (j - 1) & 1, abort_flag, p.err));
        if (!ok) break;
        tc_fence_after();
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int i = 0; i < D / 32; ++i) {
            uint32_t ov[32];
            const uint32_t ocol = tmem + lane_off + C::O_COL + i * 32;
            tmem_ld_32x32b_x32(ocol, ov);
            tmem_wait_ld();
            reg_fence(ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st_32x32b_x32(ocol, ov);
          }
        }
      }
      const uint32_t pcol = tmem + lane_off + (sb ? C::P_COL1 : C::P_COL0);
      tmem_st_32x32b_x32(pcol, pk[0]);
      tmem_st_32x32b_x32(pcol + 32, pk[1]);
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C::B_PF + sb));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_OR), (n_kv - 1) & 1, abort_flag, p.err));
    if (ok) {
      // -------------------------------------------------------- epilogue: O / l, LSE
      tc_fence_after();
      const float inv_l = 1.f / l;
      const bool row_ok = q_row < p.Nq;
      using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
      T *orow = reinterpret_cast<T *>(p.o) + static_cast<int64_t>(b) * p.o_sb + static_cast<int64_t>(h) * p.o_sh +
                static_cast<int64_t>(q_row) * p.o_sn;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(tmem + lane_off + C::O_COL + i * 32, ov);
        tmem_wait_ld();
        reg_fence(ov);
        uint32_t packed[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2)
          packed[c / 2] = pack2<BF16>(__uint_as_float(ov[c]) * inv_l, __uint_as_float(ov[c + 1]) * inv_l);
        if (row_ok) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + i * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      }
      if (p.lse != nullptr && row_ok)
        p.lse[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + q_row] = (m + __log2f(l)) * kLn2;
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_one(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p,
                       int B, cudaStream_t stream) {
  auto kern = prefill_fwd_kernel<D, CAUSAL, BF16>;
  constexpr uint32_t smem = Cfg<D>::SMEM_BYTES;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_qtiles, p.Hq, B);
  kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

}  // namespace

size_t prefill_smem_bytes(int D) { return D == 128 ? Cfg<128>::SMEM_BYTES : Cfg<64>::SMEM_BYTES; }

cudaError_t launch_prefill(int D, bool causal, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk,
                           const CUtensorMap &tv, const PrefillParams &p, int B, cudaStream_t stream) {
#define ATTN_PREFILL_CASE(DD, CC, BB) \
  if (D == DD && causal == CC && bf16 == BB) return launch_one<DD, CC, BB>(tq, tk, tv, p, B, stream);
  ATTN_PREFILL_CASE(128, true, true)
  ATTN_PREFILL_CASE(128, false, true)
  ATTN_PREFILL_CASE(128, true, false)
  ATTN_PREFILL_CASE(128, false, false)
  ATTN_PREFILL_CASE(64, true, true)
  ATTN_PREFILL_CASE(64, false, true)
  ATTN_PREFILL_CASE(64, true, false)
  ATTN_PREFILL_CASE(64, false, false)
#undef ATTN_PREFILL_CASE
  return cudaErrorInvalidValue;
}

}  // namespace attn
