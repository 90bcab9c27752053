// bwd_kernel.cuh -- attention backward from the saved log-sum-exp, sm_103a.
// Included by bwd.cu (plain causal / full attention) and bwd_masked.cu
// (sliding windows, ALiBi and per-row key ranges: the MASKED build, compiled
// as a separate translation unit so that the plain kernels keep their short
// elementwise loop).
//
// With S = scale Q K^T (masked), P = exp(S - LSE) (the forward's softmax,
// rebuilt from the saved LSE), O = P V and an incoming gradient dO:
//   dV = P^T dO,  dP = dO V^T,  D_i = sum_d dO_id O_id,  dS = P o (dP - D),
//   dQ = scale dS K,  dK = scale dS^T Q,
// and under GQA dK, dV of a kv head are summed over the q heads of its group.
// ("Skill: Write a Triton Attention Kernel" notes the backward recomputes the
// attention weights from the saved m + log(l); "Triton-FlashAttention" lists
// the GQA backward, which accumulates dK/dV over each group, as deferred.)
//
// Three kernels, no atomics, deterministic:
//   bwd_preprocess  D_i = rowsum(dO o O), fp32, into the workspace;
//   bwd_dq          one CTA per (128-row query tile, q head, b): for each KV
//                   tile, S = Q K^T and dP = dO V^T (tcgen05, SS), then
//                   dS elementwise, then dQ += dS K (TS form, dS read from
//                   TMEM, K as an MN-major operand);
//   bwd_dkdv        one CTA per (128-row key tile, kv head, b): for each q head
//                   of the group and each query tile, S^T = K Q^T and
//                   dP^T = V dO^T, then P^T and dS^T per key row, then
//                   dV += P^T dO and dK += dS^T Q (TS form), with dK and dV
//                   accumulated in TMEM over the whole group.
// Each 128-wide tile of the loop (KV tile for dQ, query tile for dK/dV) is
// computed as two 64-column halves a and b with their own TMEM columns,
// barriers and elementwise warpgroup, issued in the order
//   Sa_j dPa_j | Sb_j dPb_j | acc_a_j | Sa_{j+1} dPa_{j+1} | acc_b_j | Sb_{j+1} ...
// so that the elementwise work on one half runs while the tensor core
// computes the other half's products (the elementwise work has no row
// reduction, so the halves are independent).
// Warp roles in both tiled kernels: warp 0 TMA producer, warp 1 TMEM allocator
// and MMA issuer, warps 2-5 the elementwise warpgroup of half a, warps 6-9 the
// one of half b (one thread per TMEM lane in each).  A half writes its 16-bit
// results over the first 32 of its 64 score columns, where the following
// TS-form MMA reads them.
// MASKED: the forward's windows, ALiBi bias and key ranges (the options of
// attn_bwd_ex): the score of (query i, key j) is scale q_i . k_j -
// slope_h |i - j| and the pair is dropped outside i - window_left <= j <=
// i + window_right and the row's [lo, hi) key range; the bias enters only
// through P, and the tile loops walk only the tiles of each band.
#pragma once
#include <climits>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kT = 128;  // rows per tile (queries or keys)
constexpr int kThreads = 320;
constexpr float kLog2e = 1.4426950408889634f;

__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, int d, int n, int h, int b,
                                         uint32_t slots, uint32_t bar) {
  const int sn = slots & 3, sh = (slots >> 2) & 3;
  const int c1 = (sn == 1) ? n : (sh == 1) ? h : b;
  const int c2 = (sn == 2) ? n : (sh == 2) ? h : b;
  const int c3 = (sn == 3) ? n : (sh == 3) ? h : b;
  tma_load_4d(dst, map, d, c1, c2, c3, bar);
}

__device__ __forceinline__ int64_t max64(int64_t a, int64_t b) { return a > b ? a : b; }
__device__ __forceinline__ int64_t min64(int64_t a, int64_t b) { return a < b ? a : b; }

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

// Stores 32 fp32 accumulator columns (times s) of one row as 16-bit values.
template <bool BF16>
__device__ __forceinline__ void store_row32(void *base, int64_t off, const uint32_t (&v)[32], float s) {
  uint32_t packed[16];
#pragma unroll
  for (int c = 0; c < 32; c += 2)
    packed[c / 2] = pack2<BF16>(__uint_as_float(v[c]) * s, __uint_as_float(v[c + 1]) * s);
  uint4 *dst = reinterpret_cast<uint4 *>(reinterpret_cast<uint16_t *>(base) + off);
#pragma unroll
  for (int i = 0; i < 4; ++i) dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2], packed[4 * i + 3]);
}

// ---------------------------------------------------------------- preprocess
// 8 values of two 16-byte vectors (16-bit elements) multiplied and summed in fp32.
template <bool BF16>
__device__ __forceinline__ float dot8(const uint4 &a, const uint4 &b) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w}, bv[4] = {b.x, b.y, b.z, b.w};
  float acc = 0.f;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    float2 x, y;
    if constexpr (BF16) {
      x = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&av[i]));
      y = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162 *>(&bv[i]));
    } else {
      x = __half22float2(*reinterpret_cast<const __half2 *>(&av[i]));
      y = __half22float2(*reinterpret_cast<const __half2 *>(&bv[i]));
    }
    acc = fmaf(x.x, y.x, acc);
    acc = fmaf(x.y, y.y, acc);
  }
  return acc;
}

// D_i = sum_d dO[i, d] * O[i, d] in fp32.  D / 8 lanes per row, one 16-byte
// load of each tensor per lane and row, so a warp reads 32 / (D / 8) whole rows
// at once; each warp takes kPreRowGroups such groups of consecutive rows and
// issues all their loads before the first use (more bytes in flight per
// thread, fewer blocks).
constexpr int kPreRowGroups = 4;
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdParams p) {
  constexpr int kLanesPerRow = D / 8;
  constexpr int kRowsPerWarp = 32 / kLanesPerRow;
  if (load_volatile(p.err) != 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int row0 = (blockIdx.x * 8 + warp) * kRowsPerWarp * kPreRowGroups + lane / kLanesPerRow;
  const int part = lane % kLanesPerRow;
  const int64_t ob = static_cast<int64_t>(b) * p.o_sb + static_cast<int64_t>(h) * p.o_sh + part * 8;
  const int64_t db = static_cast<int64_t>(b) * p.do_sb + static_cast<int64_t>(h) * p.do_sh + part * 8;
  uint4 o[kPreRowGroups], g[kPreRowGroups];
#pragma unroll
  for (int it = 0; it < kPreRowGroups; ++it) {
    const int row = row0 + it * kRowsPerWarp;
    if (row < p.Nq) {
      o[it] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.o) + ob +
                                               static_cast<int64_t>(row) * p.o_sn);
      g[it] = *reinterpret_cast<const uint4 *>(reinterpret_cast<const uint16_t *>(p.dout) + db +
                                               static_cast<int64_t>(row) * p.do_sn);
    }
  }
#pragma unroll
  for (int it = 0; it < kPreRowGroups; ++it) {
    const int row = row0 + it * kRowsPerWarp;
    float acc = row < p.Nq ? dot8<BF16>(o[it], g[it]) : 0.f;
#pragma unroll
    for (int off = kLanesPerRow / 2; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    if (part == 0 && row < p.Nq) p.dvec[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + row] = acc;
  }
}

// ---------------------------------------------------------------- dQ
template <int D>
struct DqCfg {
  static constexpr int KCH = D / 64;
  static constexpr int ST = (D == 128) ? 2 : 3;
  static constexpr uint32_t CHUNK = kT * 128;      // one 64-column chunk of a 128-row tile
  static constexpr uint32_t TILE = kT * D * 2;
  static constexpr uint32_t OFF_Q = 0, OFF_DO = TILE, OFF_KV = 2 * TILE;  // stage s: K at OFF_KV + 2s TILE, V after
  static constexpr uint32_t OFF_BAR = OFF_KV + ST * 2 * TILE;
  // B_SF, B_DS: + half (2)
  static constexpr int B_QF = 0, B_KF = 1, B_KE = 1 + ST, B_SF = 1 + 2 * ST, B_DS = 3 + 2 * ST, B_DONE = 5 + 2 * ST,
                       B_MMA = 6 + 2 * ST, NBAR = 7 + 2 * ST;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_USED = OFF_MISC + 16;
  static constexpr uint32_t SMEM_BYTES = (SMEM_USED + 1024 > 116u * 1024) ? SMEM_USED + 1024 : 116u * 1024;
  // TMEM: half h's S at 128 h, its dP at 128 h + 64; dQ after both halves.
  static constexpr uint32_t DQ_COL = 256, TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t s_col(int h) { return 128u * h; }
  __host__ __device__ static constexpr uint32_t dp_col(int h) { return 128u * h + 64; }
  static constexpr uint32_t HALF_ROWS = 64 * 128;  // bytes of 64 rows in one 64-column chunk of a K or V tile
  static_assert(SMEM_BYTES <= 227u * 1024, "shared memory budget");
};

template <int D, bool CAUSAL, bool BF16, bool MASKED>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                  const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const BwdParams p) {
  using C = DqCfg<D>;
  constexpr int ST = C::ST;
  extern __shared__ uint8_t smem_raw[];
  if (load_volatile(p.err) != 0) return;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_qt = (p.Nq + kT - 1) / kT;
  // 1-D grid over (group chunk, query tile, group, q head of the group): the
  // longest causal query tiles of a chunk start first.
  int qt, h, b, hk;
  {
    const int per_group = p.group * n_qt;
    const int n_groups = p.Hkv * p.B;
    const int lin = static_cast<int>(blockIdx.x);
    const int c = lin / (p.chunk_dq * per_group);
    const int gc = min(p.chunk_dq, n_groups - c * p.chunk_dq);  // groups in this chunk
    const int r = lin - c * p.chunk_dq * per_group;
    const int tidx = r / (gc * p.group), rem = r - tidx * gc * p.group;
    const int g = c * p.chunk_dq + rem / p.group;
    qt = CAUSAL ? (n_qt - 1 - tidx) : tidx;
    hk = g % p.Hkv;
    b = g / p.Hkv;
    h = hk * p.group + rem % p.group;
  }
  const int q0 = qt * kT;
  const int nkv_all = (p.Nkv + kT - 1) / kT;
  // KV tiles [j_lo, j_lo + n_kv) of the query tile's key band: up to its
  // diagonal under the causal mask, narrowed by the windows (MASKED).
  int j_lo = 0, j_hi = CAUSAL ? min(nkv_all, qt + 1) : nkv_all;
  if constexpr (MASKED) {
    const int64_t q_last = min(p.Nq, q0 + kT) - 1;
    if (p.window_left >= 0) j_lo = static_cast<int>(max64(0, q0 - static_cast<int64_t>(p.window_left)) / kT);
    if (!CAUSAL && p.window_right >= 0)
      j_hi = static_cast<int>(min64(j_hi, min64(p.Nkv - 1, q_last + p.window_right) / kT + 1));
  }
  const int n_kv = max(0, j_hi - j_lo);

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_QF), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_KE + s), 1);
    }
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(BAR(C::B_SF + hf), 1);
      mbar_init(BAR(C::B_DS + hf), 4);  // one arrival per warp of the half's warpgroup
    }
    mbar_init(BAR(C::B_DONE), 1);
    mbar_init(BAR(C::B_MMA), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sQ = sbase + C::OFF_Q, sDO = sbase + C::OFF_DO;
  auto sK = [&](int st) { return sbase + C::OFF_KV + (2 * st) * C::TILE; };
  auto sV = [&](int st) { return sbase + C::OFF_KV + (2 * st + 1) * C::TILE; };

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(BAR(C::B_QF), 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c) {
        tma_tile(sQ + c * C::CHUNK, &tmQ, c * 64, q0, h, b, p.slots_q, BAR(C::B_QF));
        tma_tile(sDO + c * C::CHUNK, &tmDO, c * 64, q0, h, b, p.slots_do, BAR(C::B_QF));
      }
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % ST;
        if (j >= ST && !(ok = mbar_wait(BAR(C::B_KE + st), ((j / ST) - 1) & 1, abort_flag, p.err))) break;
        mbar_arrive_expect_tx(BAR(C::B_KF + st), 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c) {
          tma_tile(sK(st) + c * C::CHUNK, &tmK, c * 64, (j_lo + j) * kT, hk, b, p.slots_k, BAR(C::B_KF + st));
          tma_tile(sV(st) + c * C::CHUNK, &tmV, c * 64, (j_lo + j) * kT, hk, b, p.slots_v, BAR(C::B_KF + st));
        }
        ++issued;
      }
      if (!ok) {
        mbar_wait(BAR(C::B_QF), 0, nullptr, p.err);
        for (int i = max(0, issued - ST); i < issued; ++i)
          mbar_wait(BAR(C::B_KF + i % ST), (i / ST) & 1, nullptr, p.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(BF16, kT, 64, false, false);  // N = 64 keys (one half)
      constexpr uint32_t idesc_dq = idesc_f16(BF16, kT, D, false, true);
      // Shared-memory descriptors are formed once; each MMA adds the operand's
      // offset (in 16-byte units) to the start-address field, which never
      // carries (every operand lies below 256 KB).  The MMA thread's issue rate
      // bounds the step, so no descriptor is rebuilt per MMA.
      const uint64_t dq_k = smem_desc_sw128(sQ, 16, 1024), ddo_k = smem_desc_sw128(sDO, 16, 1024);
      const uint64_t dkv_k = smem_desc_sw128(sK(0), 16, 1024), dkv_mn = smem_desc_sw128(sK(0), C::CHUNK, 1024);
      // S_h = Q K_h^T and dP_h = dO V_h^T for keys 64 h .. 64 h + 63 of the tile in stage st.
      auto issue_sdp = [&](int hf, int st) {
        tc_fence_after();
        const uint64_t kd = dkv_k + ((2 * st * C::TILE + hf * C::HALF_ROWS) >> 4), vd = kd + (C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = ((kk / 4) * C::CHUNK + (kk % 4) * 32) >> 4;
          mma_ss(tmem + C::s_col(hf), dq_k + ko, kd + ko, idesc_s, kk > 0 ? 1u : 0u);
          mma_ss(tmem + C::dp_col(hf), ddo_k + ko, vd + ko, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(BAR(C::B_SF + hf));
      };
      // dQ += dS_h K_h: dS_h (16-bit) over the first 32 columns of S_h; K as MN-major B.
      auto issue_dq = [&](int hf, int st, bool first) {
        tc_fence_after();
        const uint64_t kd = dkv_mn + ((2 * st * C::TILE + hf * 4 * 16 * 128) >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          mma_ts(tmem + C::DQ_COL, tmem + C::s_col(hf) + kk * 8, kd + ((kk * 16 * 128) >> 4), idesc_dq,
                 (!first || kk > 0) ? 1u : 0u);
      };
      bool ok = mbar_wait(BAR(C::B_QF), 0, abort_flag, p.err);
      if (ok && n_kv > 0) {
        ok = mbar_wait(BAR(C::B_KF + 0), 0, abort_flag, p.err);
        if (ok) issue_sdp(0, 0);
      }
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % ST, sp = (j + ST - 1) % ST;
        if (j > 0) {
          // dQ += dS_b K_b of tile j-1, which then releases its stage
          if (!(ok = mbar_wait(BAR(C::B_DS + 1), (j - 1) & 1, abort_flag, p.err))) break;
          issue_dq(1, sp, false);
          tc_commit(BAR(C::B_KE + sp));
        }
        issue_sdp(1, st);
        if (!(ok = mbar_wait(BAR(C::B_DS + 0), j & 1, abort_flag, p.err))) break;
        issue_dq(0, st, j == 0);
        if (j + 1 < n_kv) {
          const int sn = (j + 1) % ST;
          if (!(ok = mbar_wait(BAR(C::B_KF + sn), ((j + 1) / ST) & 1, abort_flag, p.err))) break;
          issue_sdp(0, sn);
        }
      }
      if (ok && n_kv > 0) {
        const int sl = (n_kv - 1) % ST;
        ok = mbar_wait(BAR(C::B_DS + 1), (n_kv - 1) & 1, abort_flag, p.err);
        if (ok) {
          issue_dq(1, sl, false);
          tc_commit(BAR(C::B_KE + sl));
        }
      }
      if (ok) tc_commit(BAR(C::B_DONE));
      tc_commit(BAR(C::B_MMA));
      mbar_wait(BAR(C::B_MMA), 0, nullptr, p.err);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;  // columns half * 64 .. + 63 of each tile
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int q_row = q0 + r;
    const bool row_ok = q_row < p.Nq;
    const int64_t ri = (static_cast<int64_t>(b) * p.Hq + h) * p.Nq + q_row;
    const float lse2 = row_ok ? p.lse[ri] * kLog2e : 0.f;
    const float dv = row_ok ? p.dvec[ri] : 0.f;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = pack_f2(sl2, sl2), nl2 = pack_f2(-lse2, -lse2), nd2 = pack_f2(-dv, -dv);
    // MASKED: this row's key range and ALiBi slope (base 2).
    int64_t r_lo = INT_MIN, r_hi = INT_MAX;
    float slope2 = 0.f;
    if constexpr (MASKED) {
      if (p.kv_ranges != nullptr && row_ok) {
        const int2 rr = __ldg(reinterpret_cast<const int2 *>(p.kv_ranges) + static_cast<int64_t>(b) * p.Nq + q_row);
        r_lo = rr.x;
        r_hi = rr.y;
      }
      if (p.alibi_slopes != nullptr) slope2 = p.alibi_slopes[h] * kLog2e;
    }
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_SF + half), j & 1, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const int kv0 = (j_lo + j) * kT + half * 64;  // this half's first key
      // columns lo_c <= c < lim count
      int lim = row_ok ? ((CAUSAL ? min(p.Nkv, q_row + 1) : p.Nkv) - kv0) : 0;
      int lo_c = 0;
      if constexpr (MASKED) {
        if (p.window_left >= 0) lo_c = static_cast<int>(max64(lo_c, q_row - static_cast<int64_t>(p.window_left) - kv0));
        if (!CAUSAL && p.window_right >= 0)
          lim = static_cast<int>(min64(lim, q_row + static_cast<int64_t>(p.window_right) + 1 - kv0));
        lo_c = static_cast<int>(min64(64, max64(lo_c, r_lo - kv0)));
        lim = static_cast<int>(max64(-1, min64(lim, r_hi - kv0)));
      }
      // dS = 2^(s scale log2 e - lse2 [- slope |i - j|]) (dP - D), two columns per packed FMA / add /
      // multiply; the per-column mask (and the bias) only where some row of the warp needs it.
      auto tile = [&](auto masked) {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c0 = ch * 32;
          uint32_t sv[32], pv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::s_col(half) + c0, sv);
          tmem_ld_32x32b_x32(tmem + lane_off + C::dp_col(half) + c0, pv);
          tmem_wait_ld();
          reg_fence(sv);
          reg_fence(pv);
          uint32_t ds[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            float2 e = unpack_f2(ffma_f2(pack_f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, nl2));
            if constexpr (MASKED && decltype(masked)::value) {
              const float dq = static_cast<float>(q_row - (kv0 + c0 + c));
              e.x = fmaf(-slope2, fabsf(dq), e.x);
              e.y = fmaf(-slope2, fabsf(dq - 1.f), e.y);
            }
            float p0 = fast_exp2(e.x), p1 = fast_exp2(e.y);
            if constexpr (decltype(masked)::value) {
              if (c0 + c >= lim || c0 + c < lo_c) p0 = 0.f;
              if (c0 + c + 1 >= lim || c0 + c + 1 < lo_c) p1 = 0.f;
            }
            const float2 d = unpack_f2(
                fmul_f2(pack_f2(p0, p1), fadd_f2(pack_f2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])), nd2)));
            ds[c / 2] = pack2<BF16>(d.x, d.y);
          }
          // dS over the first 32 of this half's S columns; chunk ch only overwrites columns already read.
          tmem_st_32x32b_x16(tmem + lane_off + C::s_col(half) + ch * 16, ds);
        }
      };
      if (__all_sync(0xffffffffu, lim >= 64 && lo_c <= 0 && slope2 == 0.f))
        tile(std::false_type{});
      else
        tile(std::true_type{});
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C::B_DS + half));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_DONE), 0, abort_flag, p.err));
    if (ok) {
      tc_fence_after();
      const int64_t orow = static_cast<int64_t>(b) * p.dq_sb + static_cast<int64_t>(h) * p.dq_sh +
                           static_cast<int64_t>(q_row) * p.dq_sn;
      // each half stores half of dQ's columns
#pragma unroll
      for (int i = half * (D / 64); i < (half + 1) * (D / 64); ++i) {
        uint32_t v[32];
        if (n_kv > 0) {
          tmem_ld_32x32b_x32(tmem + lane_off + C::DQ_COL + i * 32, v);
          tmem_wait_ld();
          reg_fence(v);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = 0u;  // the row's band holds no key (windows)
        }
        if (row_ok) store_row32<BF16>(p.dq, orow + i * 32, v, p.scale);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

// ---------------------------------------------------------------- dK, dV
template <int D>
struct DkvCfg {
  static constexpr int KCH = D / 64;
  static constexpr int ST = (D == 128) ? 2 : 3;
  static constexpr uint32_t CHUNK = kT * 128;
  static constexpr uint32_t TILE = kT * D * 2;
  static constexpr uint32_t OFF_K = 0, OFF_V = TILE, OFF_QD = 2 * TILE;  // stage s: Q at OFF_QD + 2s TILE, dO after
  // [half][step parity][-lse2 | -D | key-range lo | key-range hi][64] (fp32, fp32,
  // int32, int32): the 64 queries of each half (the ranges only in MASKED builds)
  static constexpr uint32_t OFF_LD = OFF_QD + ST * 2 * TILE;
  static constexpr uint32_t OFF_BAR = OFF_LD + 2 * 2 * 4 * 64 * 4;
  // B_SF, B_DS: + half (2); B_LD: + 2 half + step parity (4)
  static constexpr int B_KVF = 0, B_QF = 1, B_QE = 1 + ST, B_SF = 1 + 2 * ST, B_DS = 3 + 2 * ST,
                       B_LD = 5 + 2 * ST, B_DONE = 9 + 2 * ST, B_MMA = 10 + 2 * ST, NBAR = 11 + 2 * ST;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_USED = OFF_MISC + 16;
  static constexpr uint32_t SMEM_BYTES = (SMEM_USED + 1024 > 116u * 1024) ? SMEM_USED + 1024 : 116u * 1024;
  // TMEM: half h's S^T at 128 h, its dP^T at 128 h + 64; dV and dK after both halves.
  static constexpr uint32_t DV_COL = 256, DK_COL = 256 + D, TMEM_COLS = 512;
  __host__ __device__ static constexpr uint32_t s_col(int h) { return 128u * h; }
  __host__ __device__ static constexpr uint32_t dp_col(int h) { return 128u * h + 64; }
  static constexpr uint32_t HALF_ROWS = 64 * 128;  // bytes of 64 rows in one 64-column chunk of a Q or dO tile
  static_assert(SMEM_BYTES <= 227u * 1024, "shared memory budget");
  static_assert(256 + 2 * D <= TMEM_COLS, "TMEM budget");
};

template <int D, bool CAUSAL, bool BF16, bool MASKED>
__global__ void __launch_bounds__(kThreads, 1)
    bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                    const BwdParams p) {
  using C = DkvCfg<D>;
  constexpr int ST = C::ST;
  extern __shared__ uint8_t smem_raw[];
  if (load_volatile(p.err) != 0) return;
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;
  uint8_t *smem = smem_raw + (sbase - raw);
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  float *sld = reinterpret_cast<float *>(smem + C::OFF_LD);  // [half][parity][lse2 | D | lo | hi][64]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kt = (p.Nkv + kT - 1) / kT;
  // 1-D grid over (group chunk, key tile, group): under the causal mask key
  // tile 0 sees every query tile, so the longest tiles of a chunk start first.
  int kt, hk, b;
  {
    const int n_groups = p.Hkv * p.B;
    const int lin = static_cast<int>(blockIdx.x);
    const int c = lin / (p.chunk_dkv * n_kt);
    const int gc = min(p.chunk_dkv, n_groups - c * p.chunk_dkv);
    const int r = lin - c * p.chunk_dkv * n_kt;
    kt = r / gc;
    const int g = c * p.chunk_dkv + (r - kt * gc);
    hk = g % p.Hkv;
    b = g / p.Hkv;
  }
  const int kv0 = kt * kT;
  const int n_qt = (p.Nq + kT - 1) / kT;
  // Query tiles that see this key tile: causal (top-left) keeps key j for query i iff j <= i;
  // windows narrow the band (MASKED).
  int i_first = CAUSAL ? min(kv0 / kT, n_qt) : 0;
  int i_end = n_qt;
  if constexpr (MASKED) {
    const int64_t kv_last = min(p.Nkv, kv0 + kT) - 1;
    if (!CAUSAL && p.window_right >= 0)
      i_first = static_cast<int>(max64(i_first, max64(0, kv0 - static_cast<int64_t>(p.window_right)) / kT));
    if (p.window_left >= 0) i_end = static_cast<int>(min64(i_end, (kv_last + p.window_left) / kT + 1));
  }
  const int n_i = max(0, i_end - i_first);
  const int n_steps = n_i * p.group;  // (q head of the group, query tile) pairs

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_KVF), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(BAR(C::B_QF + s), 1);
      mbar_init(BAR(C::B_QE + s), 1);
    }
    for (int hf = 0; hf < 2; ++hf) {
      mbar_init(BAR(C::B_SF + hf), 1);
      mbar_init(BAR(C::B_DS + hf), 4);  // one arrival per warp of the half's warpgroup
      mbar_init(BAR(C::B_LD + 2 * hf + 0), 128);
      mbar_init(BAR(C::B_LD + 2 * hf + 1), 128);
    }
    mbar_init(BAR(C::B_DONE), 1);
    mbar_init(BAR(C::B_MMA), 1);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  auto sQ = [&](int st) { return sbase + C::OFF_QD + (2 * st) * C::TILE; };
  auto sDO = [&](int st) { return sbase + C::OFF_QD + (2 * st + 1) * C::TILE; };

  if (warp == 0) {
    if (lane == 0) {
      int issued = 0;
      bool ok = true;
      mbar_arrive_expect_tx(BAR(C::B_KVF), 2 * C::TILE);
#pragma unroll
      for (int c = 0; c < C::KCH; ++c) {
        tma_tile(sK + c * C::CHUNK, &tmK, c * 64, kv0, hk, b, p.slots_k, BAR(C::B_KVF));
        tma_tile(sV + c * C::CHUNK, &tmV, c * 64, kv0, hk, b, p.slots_v, BAR(C::B_KVF));
      }
      for (int s = 0; s < n_steps; ++s) {
        const int st = s % ST;
        const int h = hk * p.group + s / n_i, i0 = (i_first + s % n_i) * kT;
        if (s >= ST && !(ok = mbar_wait(BAR(C::B_QE + st), ((s / ST) - 1) & 1, abort_flag, p.err))) break;
        mbar_arrive_expect_tx(BAR(C::B_QF + st), 2 * C::TILE);
#pragma unroll
        for (int c = 0; c < C::KCH; ++c) {
          tma_tile(sQ(st) + c * C::CHUNK, &tmQ, c * 64, i0, h, b, p.slots_q, BAR(C::B_QF + st));
          tma_tile(sDO(st) + c * C::CHUNK, &tmDO, c * 64, i0, h, b, p.slots_do, BAR(C::B_QF + st));
        }
        ++issued;
      }
      if (!ok) {
        mbar_wait(BAR(C::B_KVF), 0, nullptr, p.err);
        for (int i = max(0, issued - ST); i < issued; ++i)
          mbar_wait(BAR(C::B_QF + i % ST), (i / ST) & 1, nullptr, p.err);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_f16(BF16, kT, 64, false, false);  // N = 64 queries (one half)
      constexpr uint32_t idesc_acc = idesc_f16(BF16, kT, D, false, true);
      // S^T_h = K Q_h^T and dP^T_h = V dO_h^T for queries 64 h .. 64 h + 63 of the tile in stage st:
      // keys on the TMEM lanes, queries on the columns.
      // Descriptors formed once, per-MMA offsets added to the start-address field
      // (as in the dQ kernel).
      const uint64_t dk_k = smem_desc_sw128(sK, 16, 1024), dv_k = smem_desc_sw128(sV, 16, 1024);
      const uint64_t dqd_k = smem_desc_sw128(sQ(0), 16, 1024), dqd_mn = smem_desc_sw128(sQ(0), C::CHUNK, 1024);
      auto issue_sdp = [&](int hf, int st) {
        tc_fence_after();
        const uint64_t qd = dqd_k + ((2 * st * C::TILE + hf * C::HALF_ROWS) >> 4), dod = qd + (C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = ((kk / 4) * C::CHUNK + (kk % 4) * 32) >> 4;
          mma_ss(tmem + C::s_col(hf), dk_k + ko, qd + ko, idesc_s, kk > 0 ? 1u : 0u);
          mma_ss(tmem + C::dp_col(hf), dv_k + ko, dod + ko, idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(BAR(C::B_SF + hf));
      };
      // dV += P^T_h dO_h and dK += dS^T_h Q_h: P^T_h / dS^T_h (16-bit) over the first 32
      // columns of S^T_h / dP^T_h, dO / Q as MN-major B (queries 64 h .. of the tile).
      auto issue_acc = [&](int hf, int st, bool first) {
        tc_fence_after();
        const uint64_t qd = dqd_mn + ((2 * st * C::TILE + hf * 4 * 16 * 128) >> 4), dod = qd + (C::TILE >> 4);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
          const uint32_t bo = (kk * 16 * 128) >> 4;
          mma_ts(tmem + C::DV_COL, tmem + C::s_col(hf) + kk * 8, dod + bo, idesc_acc, (!first || kk > 0) ? 1u : 0u);
          mma_ts(tmem + C::DK_COL, tmem + C::dp_col(hf) + kk * 8, qd + bo, idesc_acc, (!first || kk > 0) ? 1u : 0u);
        }
      };
      bool ok = mbar_wait(BAR(C::B_KVF), 0, abort_flag, p.err);
      if (ok && n_steps > 0) {
        ok = mbar_wait(BAR(C::B_QF + 0), 0, abort_flag, p.err);
        if (ok) issue_sdp(0, 0);
      }
      for (int s = 0; ok && s < n_steps; ++s) {
        const int st = s % ST, sp = (s + ST - 1) % ST;
        if (s > 0) {
          // the second half of step s-1, which then releases its Q / dO stage
          if (!(ok = mbar_wait(BAR(C::B_DS + 1), (s - 1) & 1, abort_flag, p.err))) break;
          issue_acc(1, sp, false);
          tc_commit(BAR(C::B_QE + sp));
        }
        issue_sdp(1, st);
        if (!(ok = mbar_wait(BAR(C::B_DS + 0), s & 1, abort_flag, p.err))) break;
        issue_acc(0, st, s == 0);
        if (s + 1 < n_steps) {
          const int sn = (s + 1) % ST;
          if (!(ok = mbar_wait(BAR(C::B_QF + sn), ((s + 1) / ST) & 1, abort_flag, p.err))) break;
          issue_sdp(0, sn);
        }
      }
      if (ok && n_steps > 0) {
        const int sl = (n_steps - 1) % ST;
        ok = mbar_wait(BAR(C::B_DS + 1), (n_steps - 1) & 1, abort_flag, p.err);
        if (ok) {
          issue_acc(1, sl, false);
          tc_commit(BAR(C::B_QE + sl));
        }
      }
      if (ok) tc_commit(BAR(C::B_DONE));
      tc_commit(BAR(C::B_MMA));
      mbar_wait(BAR(C::B_MMA), 0, nullptr, p.err);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int half = (warp - 2) >> 2;   // query columns half * 64 .. + 63 of each tile
    const int r = quarter * 32 + lane;  // key row in the tile == TMEM lane
    const int tid = ((warp - 2) & 3) * 32 + lane;  // thread index within the warpgroup
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int kv = kv0 + r;
    const bool kv_ok = kv < p.Nkv;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = pack_f2(sl2, sl2);
    bool ok = true;
    for (int s = 0; s < n_steps; ++s) {
      const int h = hk * p.group + s / n_i, i0 = (i_first + s % n_i) * kT;
      // This step's log-sum-exp (base 2) and D of the half's 64 queries, one value
      // per thread of the warpgroup, into shared memory.
      const int q_half = i0 + half * 64;  // this half's first query
      float *buf = sld + (half * 2 + (s & 1)) * 4 * 64;
      const int *rbuf = reinterpret_cast<const int *>(buf + 128);  // key-range lo [64], hi [64]
      {
        const int qi = q_half + (tid & 63);
        const int64_t ri = (static_cast<int64_t>(b) * p.Hq + h) * p.Nq + qi;
        buf[tid] = qi < p.Nq ? ((tid < 64) ? -p.lse[ri] * kLog2e : -p.dvec[ri]) : 0.f;  // negated
        if constexpr (MASKED) {
          if (p.kv_ranges != nullptr) {
            const int2 rr = qi < p.Nq ? __ldg(reinterpret_cast<const int2 *>(p.kv_ranges) +
                                              static_cast<int64_t>(b) * p.Nq + qi)
                                      : make_int2(0, 0);
            reinterpret_cast<int *>(buf + 128)[tid] = tid < 64 ? rr.x : rr.y;
          }
        }
        mbar_arrive(BAR(C::B_LD + half * 2 + (s & 1)));
      }
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_LD + half * 2 + (s & 1)), (s >> 1) & 1, abort_flag, p.err));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_SF + half), s & 1, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      // Query columns c < hi are real queries; causal keeps query q_half+c iff kv <= q_half+c;
      // windows (MASKED): query q keeps kv iff q - window_left <= kv <= q + window_right.
      int hi = min(64, p.Nq - q_half);
      int lo = CAUSAL ? max(0, kv - q_half) : 0;
      float slope2 = 0.f;
      bool ranges = false;
      if constexpr (MASKED) {
        if (p.window_left >= 0) hi = static_cast<int>(min64(hi, kv + static_cast<int64_t>(p.window_left) - q_half + 1));
        if (!CAUSAL && p.window_right >= 0)
          lo = static_cast<int>(min64(64, max64(lo, kv - static_cast<int64_t>(p.window_right) - q_half)));
        if (p.alibi_slopes != nullptr) slope2 = p.alibi_slopes[h] * kLog2e;
        ranges = p.kv_ranges != nullptr;
      }
      // P^T = 2^(s scale log2 e - lse2), dS^T = P^T (dP^T - D), two columns per packed
      // FMA / add / multiply with the per-query values read in pairs; the mask only
      // where some key row of the warp needs it.
      auto tile = [&](auto masked) {
#pragma unroll
        for (int ch = 0; ch < 2; ++ch) {
          const int c0 = ch * 32;
          uint32_t sv[32], pv[32];
          tmem_ld_32x32b_x32(tmem + lane_off + C::s_col(half) + c0, sv);
          tmem_ld_32x32b_x32(tmem + lane_off + C::dp_col(half) + c0, pv);
          tmem_wait_ld();
          reg_fence(sv);
          reg_fence(pv);
          uint32_t pp[16], ds[16];
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const int cc = c0 + c;
            const uint64_t nl = *reinterpret_cast<const uint64_t *>(buf + cc);       // -lse2 of the two queries
            const uint64_t nd = *reinterpret_cast<const uint64_t *>(buf + 64 + cc);  // -D of the two queries
            float2 e = unpack_f2(ffma_f2(pack_f2(__uint_as_float(sv[c]), __uint_as_float(sv[c + 1])), sl2x2, nl));
            if constexpr (MASKED && decltype(masked)::value) {
              const float dq = static_cast<float>(q_half + cc - kv);
              e.x = fmaf(-slope2, fabsf(dq), e.x);
              e.y = fmaf(-slope2, fabsf(dq + 1.f), e.y);
            }
            float p0 = fast_exp2(e.x), p1 = fast_exp2(e.y);
            if constexpr (decltype(masked)::value) {
              if (!(kv_ok && cc >= lo && cc < hi)) p0 = 0.f;
              if (!(kv_ok && cc + 1 >= lo && cc + 1 < hi)) p1 = 0.f;
              if constexpr (MASKED) {
                if (ranges) {
                  if (!(kv >= rbuf[cc] && kv < rbuf[64 + cc])) p0 = 0.f;
                  if (!(kv >= rbuf[cc + 1] && kv < rbuf[64 + cc + 1])) p1 = 0.f;
                }
              }
            }
            pp[c / 2] = pack2<BF16>(p0, p1);
            const float2 d = unpack_f2(
                fmul_f2(pack_f2(p0, p1), fadd_f2(pack_f2(__uint_as_float(pv[c]), __uint_as_float(pv[c + 1])), nd)));
            ds[c / 2] = pack2<BF16>(d.x, d.y);
          }
          // P^T and dS^T over the first 32 of this half's S^T and dP^T columns;
          // only columns already read are overwritten.
          tmem_st_32x32b_x16(tmem + lane_off + C::s_col(half) + ch * 16, pp);
          tmem_st_32x32b_x16(tmem + lane_off + C::dp_col(half) + ch * 16, ds);
        }
      };
      if (__all_sync(0xffffffffu, kv_ok && lo <= 0 && hi >= 64 && slope2 == 0.f && !ranges))
        tile(std::false_type{});
      else
        tile(std::true_type{});
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C::B_DS + half));
    }
    if (ok && n_steps > 0) ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_DONE), 0, abort_flag, p.err));
    if (ok) {
      // The TMEM loads are warp-wide (.sync.aligned): every lane executes them;
      // only rows of real keys are stored.  The first warpgroup stores dV, the
      // second dK.
      tc_fence_after();
      const bool is_dk = half == 1;
      void *dst = is_dk ? p.dk : p.dv;
      const int64_t row = is_dk ? static_cast<int64_t>(b) * p.dk_sb + static_cast<int64_t>(hk) * p.dk_sh +
                                      static_cast<int64_t>(kv) * p.dk_sn
                                : static_cast<int64_t>(b) * p.dv_sb + static_cast<int64_t>(hk) * p.dv_sh +
                                      static_cast<int64_t>(kv) * p.dv_sn;
      const uint32_t col = is_dk ? C::DK_COL : C::DV_COL;
      const float mul = is_dk ? p.scale : 1.f;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        uint32_t v[32];
        if (n_steps > 0) {
          tmem_ld_32x32b_x32(tmem + lane_off + col + i * 32, v);
          tmem_wait_ld();
          reg_fence(v);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = 0u;  // no query attends to this key
        }
        if (kv_ok) store_row32<BF16>(dst, row + i * 32, v, mul);
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL, bool BF16, bool MASKED>
// The dQ and the dK/dV kernels depend only on the preprocess (D_i), not on each
// other.  Each CTA of either holds all of an SM's TMEM, so they share SMs CTA by
// CTA: with a second stream (side, if given) the dK/dV kernel runs beside the
// dQ kernel, and each fills the other's last partial waves.  The caller's stream
// waits for the side stream at the end.
cudaError_t launch_bwd_one(const BwdMaps &m, const BwdParams &p, int B, int Hkv, cudaStream_t stream,
                           cudaStream_t side) {
  constexpr int kRowsPerBlock = 8 * (32 / (D / 8)) * kPreRowGroups;
  bwd_preprocess_kernel<D, BF16><<<dim3((p.Nq + kRowsPerBlock - 1) / kRowsPerBlock, p.Hq, B), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const bool two = side != nullptr && side != stream;
  cudaEvent_t ev = nullptr;
  if (two) {
    if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    e = cudaEventRecord(ev, stream);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(side, ev, 0);
    cudaEventDestroy(ev);
    if (e != cudaSuccess) return e;
  }
  {
    auto kern = bwd_dkdv_kernel<D, CAUSAL, BF16, MASKED>;
    constexpr uint32_t smem = DkvCfg<D>::SMEM_BYTES;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
        cudaSuccess)
      return e;
    kern<<<dim3(Hkv * B * ((p.Nkv + kT - 1) / kT)), kThreads, smem, two ? side : stream>>>(m.q, m.dout, m.k, m.v,
                                                                                           p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    auto kern = bwd_dq_kernel<D, CAUSAL, BF16, MASKED>;
    constexpr uint32_t smem = DqCfg<D>::SMEM_BYTES;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
        cudaSuccess)
      return e;
    kern<<<dim3(p.Hq * B * ((p.Nq + kT - 1) / kT)), kThreads, smem, stream>>>(m.q, m.dout, m.k, m.v, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  if (two) {
    if ((e = cudaEventCreateWithFlags(&ev, cudaEventDisableTiming)) != cudaSuccess) return e;
    e = cudaEventRecord(ev, side);
    if (e == cudaSuccess) e = cudaStreamWaitEvent(stream, ev, 0);
    cudaEventDestroy(ev);
  }
  return e;
}

// Dispatch over D, causal and dtype for one value of MASKED.
template <bool MASKED>
cudaError_t launch_bwd_variant(int D, bool causal, bool bf16, const BwdMaps &m, const BwdParams &p, int B, int Hkv,
                               cudaStream_t stream, cudaStream_t side) {
#define ATTN_BWD_CASE(DD, CC, BB) \
  if (D == DD && causal == CC && bf16 == BB) return launch_bwd_one<DD, CC, BB, MASKED>(m, p, B, Hkv, stream, side);
  ATTN_BWD_CASE(128, true, true)
  ATTN_BWD_CASE(128, false, true)
  ATTN_BWD_CASE(128, true, false)
  ATTN_BWD_CASE(128, false, false)
  ATTN_BWD_CASE(64, true, true)
  ATTN_BWD_CASE(64, false, true)
  ATTN_BWD_CASE(64, true, false)
  ATTN_BWD_CASE(64, false, false)
#undef ATTN_BWD_CASE
  return cudaErrorInvalidValue;
}

}  // namespace
}  // namespace attn
