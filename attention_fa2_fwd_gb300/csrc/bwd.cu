// bwd.cu -- attention backward from the saved log-sum-exp, sm_103a.
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
//                   dS in a softmax-like warpgroup, then dQ += dS K (TS form,
//                   dS read from TMEM, K as an MN-major operand);
//   bwd_dkdv        one CTA per (128-row key tile, kv head, b): for each q head
//                   of the group and each query tile, S^T = K Q^T and
//                   dP^T = V dO^T, then P^T and dS^T per key row, then
//                   dV += P^T dO and dK += dS^T Q (TS form), with dK and dV
//                   accumulated in TMEM over the whole group.
// Warp roles in both tiled kernels: warp 0 TMA producer, warp 1 TMEM allocator
// and MMA issuer, warps 2-5 elementwise warpgroup (one thread per TMEM lane).
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kT = 128;  // rows per tile (queries or keys)
constexpr int kThreads = 192;
constexpr float kLog2e = 1.4426950408889634f;

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

template <bool BF16>
__device__ __forceinline__ float to_f(const void *p, int64_t i) {
  if constexpr (BF16)
    return __bfloat162float(reinterpret_cast<const __nv_bfloat16 *>(p)[i]);
  else
    return __half2float(reinterpret_cast<const __half *>(p)[i]);
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
template <int D, bool BF16>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const BwdParams p) {
  // One warp per row: D_i = sum_d dO[i, d] * O[i, d] in fp32.
  if (load_volatile(p.err) != 0) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int row = blockIdx.x * 8 + warp;
  if (row >= p.Nq) return;
  const int64_t oo = static_cast<int64_t>(b) * p.o_sb + static_cast<int64_t>(h) * p.o_sh + static_cast<int64_t>(row) * p.o_sn;
  const int64_t od = static_cast<int64_t>(b) * p.do_sb + static_cast<int64_t>(h) * p.do_sh + static_cast<int64_t>(row) * p.do_sn;
  float acc = 0.f;
#pragma unroll
  for (int d = lane; d < D; d += 32) acc = fmaf(to_f<BF16>(p.o, oo + d), to_f<BF16>(p.dout, od + d), acc);
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
  if (lane == 0) p.dvec[(static_cast<int64_t>(b) * p.Hq + h) * p.Nq + row] = acc;
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
  static constexpr int B_QF = 0, B_KF = 1, B_KE = 1 + ST, B_SF = 1 + 2 * ST, B_DS = 2 + 2 * ST, B_DONE = 3 + 2 * ST,
                       B_MMA = 4 + 2 * ST, NBAR = 5 + 2 * ST;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_USED = OFF_MISC + 16;
  static constexpr uint32_t SMEM_BYTES = (SMEM_USED + 1024 > 116u * 1024) ? SMEM_USED + 1024 : 116u * 1024;
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DQ_COL = 256, TMEM_COLS = 512;
  static_assert(SMEM_BYTES <= 227u * 1024, "shared memory budget");
};

template <int D, bool CAUSAL, bool BF16>
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
  // Grid (H_q, B, query tiles), heads first: under the causal mask every CTA
  // of the longest query tile starts before any shorter one.
  const int qt = CAUSAL ? (n_qt - 1 - static_cast<int>(blockIdx.z)) : static_cast<int>(blockIdx.z);
  const int h = blockIdx.x, b = blockIdx.y;
  const int hk = h / p.group;
  const int q0 = qt * kT;
  const int nkv_all = (p.Nkv + kT - 1) / kT;
  const int n_kv = CAUSAL ? min(nkv_all, qt + 1) : nkv_all;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_QF), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_KE + s), 1);
    }
    mbar_init(BAR(C::B_SF), 1);
    mbar_init(BAR(C::B_DS), 4);
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
          tma_tile(sK(st) + c * C::CHUNK, &tmK, c * 64, j * kT, hk, b, p.slots_k, BAR(C::B_KF + st));
          tma_tile(sV(st) + c * C::CHUNK, &tmV, c * 64, j * kT, hk, b, p.slots_v, BAR(C::B_KF + st));
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
      constexpr uint32_t idesc_s = idesc_f16(BF16, kT, kT, false, false);
      constexpr uint32_t idesc_dq = idesc_f16(BF16, kT, D, false, true);
      bool ok = mbar_wait(BAR(C::B_QF), 0, abort_flag, p.err);
      for (int j = 0; ok && j < n_kv; ++j) {
        const int st = j % ST;
        if (!(ok = mbar_wait(BAR(C::B_KF + st), (j / ST) & 1, abort_flag, p.err))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk / 4) * C::CHUNK + (kk % 4) * 32;
          mma_ss(tmem + C::S_COL, smem_desc_sw128(sQ + ko, 16, 1024), smem_desc_sw128(sK(st) + ko, 16, 1024),
                 idesc_s, kk > 0 ? 1u : 0u);
          mma_ss(tmem + C::DP_COL, smem_desc_sw128(sDO + ko, 16, 1024), smem_desc_sw128(sV(st) + ko, 16, 1024),
                 idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(BAR(C::B_SF));
        if (!(ok = mbar_wait(BAR(C::B_DS), j & 1, abort_flag, p.err))) break;
        tc_fence_after();
        // dQ += dS K_j: dS (16-bit) over the first 64 columns of S; K as MN-major B.
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk)
          mma_ts(tmem + C::DQ_COL, tmem + C::S_COL + kk * 8, smem_desc_sw128(sK(st) + kk * 16 * 128, C::CHUNK, 1024),
                 idesc_dq, (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit(BAR(C::B_KE + st));
      }
      if (ok) tc_commit(BAR(C::B_DONE));
      tc_commit(BAR(C::B_MMA));
      mbar_wait(BAR(C::B_MMA), 0, nullptr, p.err);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int q_row = q0 + r;
    const bool row_ok = q_row < p.Nq;
    const int64_t ri = (static_cast<int64_t>(b) * p.Hq + h) * p.Nq + q_row;
    const float lse2 = row_ok ? p.lse[ri] * kLog2e : 0.f;
    const float dv = row_ok ? p.dvec[ri] : 0.f;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int j = 0; j < n_kv; ++j) {
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_SF), j & 1, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      const int kv0 = j * kT;
      const int lim = row_ok ? ((CAUSAL ? min(p.Nkv, q_row + 1) : p.Nkv) - kv0) : 0;  // columns c < lim count
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sv[32], pv[32];
        tmem_ld_32x32b_x32(tmem + lane_off + C::S_COL + ch * 32, sv);
        tmem_ld_32x32b_x32(tmem + lane_off + C::DP_COL + ch * 32, pv);
        tmem_wait_ld();
        reg_fence(sv);
        reg_fence(pv);
        uint32_t ds[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int cc = ch * 32 + c;
          const float p0 = (cc < lim) ? fast_exp2(fmaf(__uint_as_float(sv[c]), sl2, -lse2)) : 0.f;
          const float p1 = (cc + 1 < lim) ? fast_exp2(fmaf(__uint_as_float(sv[c + 1]), sl2, -lse2)) : 0.f;
          ds[c / 2] = pack2<BF16>(p0 * (__uint_as_float(pv[c]) - dv), p1 * (__uint_as_float(pv[c + 1]) - dv));
        }
        // dS over S's first 64 columns; chunk ch only overwrites columns already read.
        tmem_st_32x32b_x16(tmem + lane_off + C::S_COL + ch * 16, ds);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C::B_DS));
    }
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_DONE), 0, abort_flag, p.err));
    if (ok) {
      tc_fence_after();
      const int64_t orow = static_cast<int64_t>(b) * p.dq_sb + static_cast<int64_t>(h) * p.dq_sh +
                           static_cast<int64_t>(q_row) * p.dq_sn;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        uint32_t v[32];
        tmem_ld_32x32b_x32(tmem + lane_off + C::DQ_COL + i * 32, v);
        tmem_wait_ld();
        reg_fence(v);
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
  static constexpr uint32_t OFF_LD = OFF_QD + ST * 2 * TILE;              // fp32 [2][2][128]: (lse2, D) per step parity
  static constexpr uint32_t OFF_BAR = OFF_LD + 2 * 2 * kT * 4;
  static constexpr int B_KVF = 0, B_QF = 1, B_QE = 1 + ST, B_SF = 1 + 2 * ST, B_DS = 2 + 2 * ST,
                       B_LD = 3 + 2 * ST /* +2 */, B_DONE = 5 + 2 * ST, B_MMA = 6 + 2 * ST, NBAR = 7 + 2 * ST;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_USED = OFF_MISC + 16;
  static constexpr uint32_t SMEM_BYTES = (SMEM_USED + 1024 > 116u * 1024) ? SMEM_USED + 1024 : 116u * 1024;
  static constexpr uint32_t S_COL = 0, DP_COL = 128, DV_COL = 256, DK_COL = 256 + D, TMEM_COLS = 512;
  static_assert(SMEM_BYTES <= 227u * 1024, "shared memory budget");
  static_assert(256 + 2 * D <= TMEM_COLS, "TMEM budget");
};

template <int D, bool CAUSAL, bool BF16>
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
  float *sld = reinterpret_cast<float *>(smem + C::OFF_LD);  // [parity][lse2 | D][128]

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_kt = (p.Nkv + kT - 1) / kT;
  // Grid (H_kv, B, key tiles), heads first: under the causal mask key tile 0
  // sees every query tile, so the longest CTAs all start first.
  const int kt = static_cast<int>(blockIdx.z);
  const int hk = blockIdx.x, b = blockIdx.y;
  const int kv0 = kt * kT;
  const int n_qt = (p.Nq + kT - 1) / kT;
  // Query tiles that see this key tile: causal (top-left) keeps key j for query i iff j <= i.
  const int i_first = CAUSAL ? min(kv0 / kT, n_qt) : 0;
  const int n_i = n_qt - i_first;
  const int n_steps = n_i * p.group;  // (q head of the group, query tile) pairs
  (void)n_kt;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_KVF), 1);
    for (int s = 0; s < ST; ++s) {
      mbar_init(BAR(C::B_QF + s), 1);
      mbar_init(BAR(C::B_QE + s), 1);
    }
    mbar_init(BAR(C::B_SF), 1);
    mbar_init(BAR(C::B_DS), 4);
    mbar_init(BAR(C::B_LD + 0), 128);
    mbar_init(BAR(C::B_LD + 1), 128);
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
      constexpr uint32_t idesc_s = idesc_f16(BF16, kT, kT, false, false);
      constexpr uint32_t idesc_acc = idesc_f16(BF16, kT, D, false, true);
      bool ok = mbar_wait(BAR(C::B_KVF), 0, abort_flag, p.err);
      for (int s = 0; ok && s < n_steps; ++s) {
        const int st = s % ST;
        if (!(ok = mbar_wait(BAR(C::B_QF + st), (s / ST) & 1, abort_flag, p.err))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t ko = (kk / 4) * C::CHUNK + (kk % 4) * 32;
          // S^T = K Q^T and dP^T = V dO^T: keys on the TMEM lanes, queries on the columns.
          mma_ss(tmem + C::S_COL, smem_desc_sw128(sK + ko, 16, 1024), smem_desc_sw128(sQ(st) + ko, 16, 1024),
                 idesc_s, kk > 0 ? 1u : 0u);
          mma_ss(tmem + C::DP_COL, smem_desc_sw128(sV + ko, 16, 1024), smem_desc_sw128(sDO(st) + ko, 16, 1024),
                 idesc_s, kk > 0 ? 1u : 0u);
        }
        tc_commit(BAR(C::B_SF));
        if (!(ok = mbar_wait(BAR(C::B_DS), s & 1, abort_flag, p.err))) break;
        tc_fence_after();
        // dV += P^T dO and dK += dS^T Q: P^T / dS^T (16-bit) from TMEM, dO / Q as MN-major B.
#pragma unroll
        for (int kk = 0; kk < kT / 16; ++kk) {
          const uint32_t bo = kk * 16 * 128;
          mma_ts(tmem + C::DV_COL, tmem + C::S_COL + kk * 8, smem_desc_sw128(sDO(st) + bo, C::CHUNK, 1024),
                 idesc_acc, (s > 0 || kk > 0) ? 1u : 0u);
          mma_ts(tmem + C::DK_COL, tmem + C::DP_COL + kk * 8, smem_desc_sw128(sQ(st) + bo, C::CHUNK, 1024),
                 idesc_acc, (s > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(BAR(C::B_QE + st));
      }
      if (ok) tc_commit(BAR(C::B_DONE));
      tc_commit(BAR(C::B_MMA));
      mbar_wait(BAR(C::B_MMA), 0, nullptr, p.err);
    }
    __syncwarp();
  } else {
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // key row in the tile == TMEM lane
    const int tid = (warp - 2) * 32 + lane;
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const int kv = kv0 + r;
    const bool kv_ok = kv < p.Nkv;
    const float sl2 = p.scale_log2;
    bool ok = true;
    for (int s = 0; s < n_steps; ++s) {
      const int h = hk * p.group + s / n_i, i0 = (i_first + s % n_i) * kT;
      // This step's per-query log-sum-exp (base 2) and D, one value per thread, into shared memory.
      float *buf = sld + (s & 1) * 2 * kT;
      {
        const int qi = i0 + tid;
        const int64_t ri = (static_cast<int64_t>(b) * p.Hq + h) * p.Nq + qi;
        buf[tid] = qi < p.Nq ? p.lse[ri] * kLog2e : 0.f;
        buf[kT + tid] = qi < p.Nq ? p.dvec[ri] : 0.f;
        mbar_arrive(BAR(C::B_LD + (s & 1)));
      }
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_LD + (s & 1)), (s >> 1) & 1, abort_flag, p.err));
      if (ok) ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_SF), s & 1, abort_flag, p.err));
      if (!ok) break;
      tc_fence_after();
      // Query columns c < hi are real queries; causal keeps query i0+c iff kv <= i0+c.
      const int hi = min(kT, p.Nq - i0);
      const int lo = CAUSAL ? max(0, kv - i0) : 0;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t sv[32], pv[32];
        tmem_ld_32x32b_x32(tmem + lane_off + C::S_COL + ch * 32, sv);
        tmem_ld_32x32b_x32(tmem + lane_off + C::DP_COL + ch * 32, pv);
        tmem_wait_ld();
        reg_fence(sv);
        reg_fence(pv);
        uint32_t pp[16], ds[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2) {
          const int cc = ch * 32 + c;
          const bool k0 = kv_ok && cc >= lo && cc < hi, k1 = kv_ok && cc + 1 >= lo && cc + 1 < hi;
          const float p0 = k0 ? fast_exp2(fmaf(__uint_as_float(sv[c]), sl2, -buf[cc])) : 0.f;
          const float p1 = k1 ? fast_exp2(fmaf(__uint_as_float(sv[c + 1]), sl2, -buf[cc + 1])) : 0.f;
          pp[c / 2] = pack2<BF16>(p0, p1);
          ds[c / 2] = pack2<BF16>(p0 * (__uint_as_float(pv[c]) - buf[kT + cc]),
                                  p1 * (__uint_as_float(pv[c + 1]) - buf[kT + cc + 1]));
        }
        // P^T over S^T's first 64 columns, dS^T over dP^T's; only columns already read are overwritten.
        tmem_st_32x32b_x16(tmem + lane_off + C::S_COL + ch * 16, pp);
        tmem_st_32x32b_x16(tmem + lane_off + C::DP_COL + ch * 16, ds);
      }
      tmem_wait_st();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(BAR(C::B_DS));
    }
    if (ok && n_steps > 0) ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_DONE), 0, abort_flag, p.err));
    if (ok) {
      // The TMEM loads are warp-wide (.sync.aligned): every lane executes them;
      // only rows of real keys are stored.
      tc_fence_after();
      const int64_t vrow = static_cast<int64_t>(b) * p.dv_sb + static_cast<int64_t>(hk) * p.dv_sh +
                           static_cast<int64_t>(kv) * p.dv_sn;
      const int64_t krow = static_cast<int64_t>(b) * p.dk_sb + static_cast<int64_t>(hk) * p.dk_sh +
                           static_cast<int64_t>(kv) * p.dk_sn;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        uint32_t v[32];
        if (n_steps > 0) {
          tmem_ld_32x32b_x32(tmem + lane_off + C::DV_COL + i * 32, v);
          tmem_wait_ld();
          reg_fence(v);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = 0u;  // no query attends to this key
        }
        if (kv_ok) store_row32<BF16>(p.dv, vrow + i * 32, v, 1.f);
      }
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        uint32_t v[32];
        if (n_steps > 0) {
          tmem_ld_32x32b_x32(tmem + lane_off + C::DK_COL + i * 32, v);
          tmem_wait_ld();
          reg_fence(v);
        } else {
#pragma unroll
          for (int c = 0; c < 32; ++c) v[c] = 0u;
        }
        if (kv_ok) store_row32<BF16>(p.dk, krow + i * 32, v, p.scale);
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

template <int D, bool CAUSAL, bool BF16>
cudaError_t launch_bwd_one(const BwdMaps &m, const BwdParams &p, int B, int Hkv, cudaStream_t stream) {
  bwd_preprocess_kernel<D, BF16><<<dim3((p.Nq + 7) / 8, p.Hq, B), 256, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  {
    auto kern = bwd_dq_kernel<D, CAUSAL, BF16>;
    constexpr uint32_t smem = DqCfg<D>::SMEM_BYTES;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
        cudaSuccess)
      return e;
    kern<<<dim3(p.Hq, B, (p.Nq + kT - 1) / kT), kThreads, smem, stream>>>(m.q, m.dout, m.k, m.v, p);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }
  {
    auto kern = bwd_dkdv_kernel<D, CAUSAL, BF16>;
    constexpr uint32_t smem = DkvCfg<D>::SMEM_BYTES;
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem))) !=
        cudaSuccess)
      return e;
    kern<<<dim3(Hkv, B, (p.Nkv + kT - 1) / kT), kThreads, smem, stream>>>(m.q, m.dout, m.k, m.v, p);
    e = cudaGetLastError();
  }
  return e;
}

}  // namespace

cudaError_t launch_bwd(int D, bool causal, bool bf16, const BwdMaps &m, const BwdParams &p, int B, int Hkv,
                       cudaStream_t stream) {
#define ATTN_BWD_CASE(DD, CC, BB) \
  if (D == DD && causal == CC && bf16 == BB) return launch_bwd_one<DD, CC, BB>(m, p, B, Hkv, stream);
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

}  // namespace attn
