// prefill_pair_kernel.cuh -- fused attention forward (prefill) for head
// dimension 128 on CTA pairs: clusters of two CTAs on neighbouring SMs whose
// matrix products are issued as one (tcgen05 cta_group::2, M = 256 rows).
//
// Why pairs.  In the one-CTA kernel P overwrites its S columns in tensor
// memory, so a tile's next S product can only start after its P V product has
// read P: the tile's step is S -> softmax -> P V -> S, and the other tile's two
// products do not fill the tensor pipe during its softmax.  Here P goes to
// shared memory (P V reads it as an ordinary operand), so S_t(j+1) is issued as
// soon as the softmax has loaded S_t(j) into registers and the tensor pipe
// always has the next product queued.  The room for P comes from the pairing:
// each CTA keeps only half of every K tile (64 of its 128 keys) and half of
// every V tile (64 of the 128 dimensions); the pair's products exchange the
// halves.
//
// A unit is 512 query rows of one (batch, q head): tile A = rows q0..q0+255,
// tile B = rows q0+256..q0+511; rank r of the pair holds rows 128 r..128 r+127
// of each tile (its TMEM lanes).  Per CTA:
//   warps 0-3   softmax of tile A, one thread per row (TMEM lane)
//   warps 4-7   softmax of tile B
//   warp 8      TMA producer: this CTA's rows of both Q tiles, its half of each
//               K tile (keys 64 r..64 r+63) and of each V tile (dimensions
//               64 r..64 r+63); every copy is counted on rank 0's barriers
//   warp 9      TMEM allocation (both CTAs, 512 columns); in rank 0 one thread
//               issues all products, per KV tile j:
//                 O_B += P_B(j-1) V_{j-1};  S_A(j+1) = Q_A K_{j+1}^T;
//                 O_A += P_A(j) V_j;        S_B(j+1) = Q_B K_{j+1}^T
//               and signals completions to both CTAs' barriers.
//   warps 10-11 idle (they keep the register split of the one-CTA kernel).
// The online softmax is that of the one-CTA kernel (base-2 scores, the running
// max raised only when a block max exceeds it by more than 8, O and l
// rescaled by alpha = 2^(m_old - m_new), O / l and lse = m + ln l at the end),
// following "Skill: Write a Triton Attention Kernel" (Required reasoning
// process, steps 4-9).  Under the causal mask rank 0's rows of a tile see one
// KV tile fewer than rank 1's; the shared product computes it and the mask
// zeroes it.
//
// TMEM columns (512, in both CTAs): S_A [0,128) S_B [128,256) O_A [256,384) O_B [384,512).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

// 12 warps: the softmax warps get 200 registers and the rest 104 (setmaxnreg
// redistributes the 384 x 168 registers of the launch: 256 x 200 + 128 x 104);
// warps 10-11 idle.
constexpr int kPairThreads = 384;
constexpr int kPairSoftmaxRegs = 200;
constexpr int kPairOtherRegs = 104;
constexpr int kPairTileRows = 128;  // rows of a tile held by one CTA
constexpr int kPairBN = 128;        // keys per KV tile
constexpr float kPairLn2 = 0.693147180559945309f;
constexpr float kPairRescale = 8.0f;  // base-2 units

struct PairCfg {
  static constexpr uint32_t CHUNK_Q = kPairTileRows * 128;  // 64 dimensions of 128 rows (128-byte rows)
  static constexpr uint32_t QT_BYTES = 2 * CHUNK_Q;          // 128 rows x 128 dimensions
  static constexpr uint32_t CHUNK_P = kPairTileRows * 128;  // 64 keys of 128 rows
  static constexpr uint32_t PT_BYTES = 2 * CHUNK_P;          // 128 rows x 128 keys
  static constexpr uint32_t CHUNK_K = 64 * 128;              // 64 dimensions of 64 keys
  static constexpr uint32_t KH_BYTES = 2 * CHUNK_K;          // half a K tile: 64 keys x 128 dimensions
  static constexpr uint32_t VH_BYTES = kPairBN * 128;        // half a V tile: 128 keys x 64 dimensions
  static constexpr int KST = 3, VST = 3;                     // ring stages
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_P = OFF_Q + 2 * QT_BYTES;
  static constexpr uint32_t OFF_K = OFF_P + 2 * PT_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KST * KH_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + VST * VH_BYTES;
  // Barriers.  Rank 0's copies of QF, KF, VF, SC and PF are the ones used (the
  // MMA thread waits on them); SF, PVD, KE and VE are signalled in both CTAs.
  static constexpr int B_QF = 0;              // Q of both CTAs landed
  static constexpr int B_KF = 1;              // + K stage: both halves landed
  static constexpr int B_KE = B_KF + KST;     // + K stage: free again
  static constexpr int B_VF = B_KE + KST;     // + V stage: both halves landed
  static constexpr int B_VE = B_VF + VST;     // + V stage: free again
  static constexpr int B_SF = B_VE + VST;     // + tile: S_t(j) computed
  static constexpr int B_SC = B_SF + 2;       // + tile: S_t(j) read by both CTAs' softmax warps (8 arrivals)
  static constexpr int B_PF = B_SC + 2;       // + tile: P_t(j) stored, O_t rescaled (8 arrivals)
  static constexpr int B_PVD = B_PF + 2;      // + tile: P_t(j) V_j completed
  static constexpr int B_DONE = B_PVD + 2;    // every product completed
  static constexpr int NBAR = B_DONE + 1;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t SMEM_USED = OFF_MISC + 16;
  static constexpr uint32_t SMEM_BYTES = SMEM_USED + 1024;  // + slack for the 1024-byte alignment
  static_assert(SMEM_BYTES <= 227u * 1024, "shared memory budget");
  static_assert(OFF_P % 1024 == 0 && OFF_K % 1024 == 0 && OFF_V % 1024 == 0, "swizzle atoms need 1024-byte alignment");
};

// One unit: 512 query rows of one (batch, q head) and the KV tiles its two
// tiles need: tile t uses KV tiles [0, hi_t), hi_A <= hi_B.
struct PairUnit {
  int h, b, hk, q0, hiA, hiB;
};

template <bool CAUSAL>
__device__ __forceinline__ PairUnit pair_unit(int u, const PrefillParams &p) {
  PairUnit U;
  const int hb = p.Hq * p.B;
  const int z = u / hb, rem = u - z * hb;
  U.h = rem % p.Hq;
  U.b = rem / p.Hq;
  U.hk = U.h / p.group;
  // Longest causal units first (see the one-CTA kernel's schedule).
  U.q0 = (CAUSAL ? (p.n_qtiles - 1 - z) : z) * kPairUnitRows;
  // Causal (top-left): row i sees keys 0..i.
  const int kmaxA = CAUSAL ? min(p.Nkv - 1, U.q0 + 255) : p.Nkv - 1;
  const int kmaxB = CAUSAL ? min(p.Nkv - 1, U.q0 + 511) : p.Nkv - 1;
  U.hiA = kmaxA / kPairBN + 1;
  U.hiB = kmaxB / kPairBN + 1;
  return U;
}

__device__ __forceinline__ int pair_unit_index(int k, int c, int g) { return k * g + ((k & 1) ? g - 1 - c : c); }

// 4-D tensor-map load into this CTA's shared memory, counted on rank 0's
// barrier `bar_c`; (d, n, h, b) placed into the map's coordinate slots.
__device__ __forceinline__ void pair_tma(uint32_t dst, const CUtensorMap *map, int d, int n, int h, int b,
                                         uint32_t slots, uint32_t bar_c, bool read_once) {
  const int sn = slots & 3, sh = (slots >> 2) & 3;
  const int c1 = (sn == 1) ? n : (sh == 1) ? h : b;
  const int c2 = (sn == 2) ? n : (sh == 2) ? h : b;
  const int c3 = (sn == 3) ? n : (sh == 3) ? h : b;
  if (read_once) tma_load_4d_pair_hint(dst, map, d, c1, c2, c3, bar_c, l2_policy_evict_first());
  else tma_load_4d_pair(dst, map, d, c1, c2, c3, bar_c);
}

template <bool BF16>
__device__ __forceinline__ uint32_t pair_pack2(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  }
}

// tmQ: 64 x 128-row boxes; tmK: 64 x 64-row boxes (half a K tile); tmV: 64 x
// 128-row boxes (half of a V tile's dimensions).  Launched as clusters of 2.
template <bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(kPairThreads, 1)
    prefill_pair_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmV, const __grid_constant__ PrefillParams p) {
  using C = PairCfg;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sbase = (raw + 1023u) & ~1023u;  // the same offset in both CTAs
  uint8_t *smem = smem_raw + (sbase - raw);
  const uint32_t sQ = sbase + C::OFF_Q, sP = sbase + C::OFF_P, sK = sbase + C::OFF_K, sV = sbase + C::OFF_V;
  const uint32_t bar0 = sbase + C::OFF_BAR;
  auto BAR = [&](int i) -> uint32_t { return bar0 + 8u * static_cast<uint32_t>(i); };
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + C::OFF_MISC);
  volatile int *abort_flag = reinterpret_cast<volatile int *>(smem + C::OFF_MISC + 4);
  volatile unsigned *stop_flag = reinterpret_cast<volatile unsigned *>(smem + C::OFF_MISC + 8);

  const uint32_t rank = cluster_cta_rank();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cid = static_cast<int>(blockIdx.x >> 1), n_cl = static_cast<int>(gridDim.x >> 1);
  const int n_units = p.n_units;
  // Rank 0's copy of barrier i, as an address in the cluster window.
  auto LEAD = [&](int i) -> uint32_t { return mapa_shared(BAR(i), 0); };

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_QF), 1);
    for (int s = 0; s < C::KST; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_KE + s), 1);
    }
    for (int s = 0; s < C::VST; ++s) {
      mbar_init(BAR(C::B_VF + s), 1);
      mbar_init(BAR(C::B_VE + s), 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(BAR(C::B_SF + t), 1);
      mbar_init(BAR(C::B_SC + t), 8);  // one arrival per softmax warp of the tile, both CTAs
      mbar_init(BAR(C::B_PF + t), 8);
      mbar_init(BAR(C::B_PVD + t), 1);
    }
    mbar_init(BAR(C::B_DONE), 1);
    *abort_flag = 0;
    // An earlier launch failed: nothing runs until the error is read.  Rank 0
    // decides for both CTAs, so that they take the same path.
    *stop_flag = (rank == 0 && load_volatile(p.err) != 0) ? 1u : 0u;
    fence_barrier_init();
  }
  cluster_sync();  // barriers initialised in both CTAs before any copy or arrival targets them
  if (ld_shared_cluster(mapa_shared(smem_u32(const_cast<unsigned *>(stop_flag)), 0)) != 0) {
    cluster_sync();  // rank 0's flag has been read by both
    return;
  }
  if (warp == 9) {
    tmem_alloc_pair(smem_u32(tmem_slot), 512);
    tmem_relinquish_pair();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' TMEM allocated before rank 0 issues a product
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t *>(tmem_slot);

  if (warp >= 8) {
   asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kPairOtherRegs));
   if (warp == 8) {
    // -------------------------------------------------------------- TMA producer
    if (lane == 0) {
      int issued_k = 0, issued_v = 0, nq = 0;
      int kst = 0, vst = 0;
      uint32_t kph = 0, vph = 0;
      int q_wait = -1;  // K stage whose release frees Q (the unit's last K tile)
      uint32_t q_phase = 0;
      bool ok = true;
      auto load_k = [&](const PairUnit &U, int j) -> bool {
        if (issued_k >= C::KST && !mbar_wait(BAR(C::B_KE + kst), kph ^ 1, abort_flag, p.err)) return false;
        if (rank == 0) mbar_arrive_expect_tx(BAR(C::B_KF + kst), 2 * C::KH_BYTES);
#pragma unroll
        for (int c = 0; c < 2; ++c)
          pair_tma(sK + kst * C::KH_BYTES + c * C::CHUNK_K, &tmK, c * 64, j * kPairBN + 64 * static_cast<int>(rank),
                   U.hk, U.b, p.slots_k, LEAD(C::B_KF + kst), false);
        ++issued_k;
        q_wait = kst;
        q_phase = kph;
        if (++kst == C::KST) {
          kst = 0;
          kph ^= 1;
        }
        return true;
      };
      auto load_v = [&](const PairUnit &U, int j) -> bool {
        if (issued_v >= C::VST && !mbar_wait(BAR(C::B_VE + vst), vph ^ 1, abort_flag, p.err)) return false;
        if (rank == 0) mbar_arrive_expect_tx(BAR(C::B_VF + vst), 2 * C::VH_BYTES);
        pair_tma(sV + vst * C::VH_BYTES, &tmV, 64 * static_cast<int>(rank), j * kPairBN, U.hk, U.b, p.slots_v,
                 LEAD(C::B_VF + vst), false);
        ++issued_v;
        if (++vst == C::VST) {
          vst = 0;
          vph ^= 1;
        }
        return true;
      };
      for (int k = 0; ok && k * n_cl < n_units; ++k) {
        const int u = pair_unit_index(k, cid, n_cl);
        if (u >= n_units) continue;
        const PairUnit U = pair_unit<CAUSAL>(u, p);
        // The previous unit's Q is free once its last S product completed: the
        // release of its last K stage (products complete in order).
        if (q_wait >= 0 && !(ok = mbar_wait(BAR(C::B_KE + q_wait), q_phase, abort_flag, p.err))) break;
        if (rank == 0) mbar_arrive_expect_tx(BAR(C::B_QF), 2 * 2 * C::QT_BYTES);
#pragma unroll
        for (int t = 0; t < 2; ++t)
#pragma unroll
          for (int c = 0; c < 2; ++c)
            pair_tma(sQ + t * C::QT_BYTES + c * C::CHUNK_Q, &tmQ, c * 64,
                     U.q0 + t * 256 + kPairTileRows * static_cast<int>(rank), U.h, U.b, p.slots_q, LEAD(C::B_QF),
                     true);
        ++nq;
        // K runs one tile ahead of V: S_A(j+1) is issued before P_A(j) V_j.
        if (!(ok = load_k(U, 0))) break;
        for (int j = 0; j < U.hiB; ++j) {
          if (j + 1 < U.hiB && !(ok = load_k(U, j + 1))) break;
          if (!(ok = load_v(U, j))) break;
        }
        if (!ok) break;
      }
      if (!ok && rank == 0) {
        // Let every copy already requested land (rank 0's barriers count both
        // CTAs' bytes) before shared memory is released.
        if (nq > 0) mbar_wait(BAR(C::B_QF), (nq - 1) & 1, nullptr, p.err);
        for (int i = max(0, issued_k - C::KST); i < issued_k; ++i)
          mbar_wait(BAR(C::B_KF + i % C::KST), (i / C::KST) & 1, nullptr, p.err);
        for (int i = max(0, issued_v - C::VST); i < issued_v; ++i)
          mbar_wait(BAR(C::B_VF + i % C::VST), (i / C::VST) & 1, nullptr, p.err);
      }
    }
    __syncwarp();
   } else if (warp == 9) {
    // -------------------------------------------------------------- MMA issuer (rank 0)
    if (rank == 0 && lane == 0) {
      constexpr uint32_t id_s = idesc_f16(BF16, 256, kPairBN, false, false);
      constexpr uint32_t id_pv = idesc_f16(BF16, 256, 128, false, true);
      const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024), dq1 = smem_desc_sw128(sQ + C::QT_BYTES, 16, 1024);
      const uint64_t dp0 = smem_desc_sw128(sP, 16, 1024), dp1 = smem_desc_sw128(sP + C::PT_BYTES, 16, 1024);
      const uint64_t dk = smem_desc_sw128(sK, 16, 1024), dv = smem_desc_sw128(sV, C::VH_BYTES, 1024);
      constexpr uint32_t kK16 = C::KH_BYTES >> 4, kV16 = C::VH_BYTES >> 4;
      const uint32_t peer = 1;
      // Completion of everything issued so far, signalled in both CTAs.
      auto commit2 = [&](int i) {
        tc_commit_pair(BAR(i));
        tc_commit_pair(mapa_shared(BAR(i), peer));
      };
      // The base descriptors pass through an empty asm so that the compiler
      // forms each product's descriptor with one add instead of holding all
      // of them in registers (the issuer has 104).
      auto issue_s = [&](int t, uint64_t qd, uint64_t kd) {
        asm volatile("" : "+l"(qd), "+l"(kd));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          // Q and K are K-major: 16 dimensions (32 B) per product inside a 128-byte row.
          mma_ss_pair(tmem + static_cast<uint32_t>(t) * 128u,
                      qd + (((kk / 4) * C::CHUNK_Q + (kk % 4) * 32) >> 4),
                      kd + (((kk / 4) * C::CHUNK_K + (kk % 4) * 32) >> 4), id_s, kk > 0 ? 1u : 0u);
        commit2(C::B_SF + t);
      };
      auto issue_pv = [&](int t, bool first, uint64_t pd, uint64_t vd) {
        asm volatile("" : "+l"(pd), "+l"(vd));
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          // P is K-major (keys along its rows); V is MN-major: 16 keys = 16 rows of 128 B.
          mma_ss_pair(tmem + 256u + static_cast<uint32_t>(t) * 128u,
                      pd + (((kk / 4) * C::CHUNK_P + (kk % 4) * 32) >> 4), vd + ((kk * 16 * 128) >> 4), id_pv,
                      (!first || kk > 0) ? 1u : 0u);
        commit2(C::B_PVD + t);
      };
      bool ok = true;
      int kst = 0, vst = 0;
      uint32_t kph = 0, vph = 0;
      uint32_t sc_par[2] = {0u, 0u}, pf_par[2] = {0u, 0u};
      bool s_any[2] = {false, false};  // an S product of tile t was issued before
      int nq = 0;
      // S_t's columns are free once both CTAs' softmax warps read the previous S_t.
      auto wait_sc = [&](int t) -> bool {
        if (!s_any[t]) {
          s_any[t] = true;
          return true;
        }
        const bool r = mbar_wait(BAR(C::B_SC + t), sc_par[t], abort_flag, p.err);
        sc_par[t] ^= 1;
        return r;
      };
      auto wait_pf = [&](int t) -> bool {
        const bool r = mbar_wait(BAR(C::B_PF + t), pf_par[t], abort_flag, p.err);
        pf_par[t] ^= 1;
        return r;
      };
      for (int k = 0; ok && k * n_cl < n_units; ++k) {
        const int u = pair_unit_index(k, cid, n_cl);
        if (u >= n_units) continue;
        const PairUnit U = pair_unit<CAUSAL>(u, p);
        const int hiA = U.hiA, hiB = U.hiB;
        if (!(ok = mbar_wait(BAR(C::B_QF), nq & 1, abort_flag, p.err))) break;
        ++nq;
        if (!(ok = mbar_wait(BAR(C::B_KF + kst), kph, abort_flag, p.err))) break;
        if (!(ok = wait_sc(0))) break;
        tc_fence_after();
        issue_s(0, dq0, dk + kst * kK16);
        if (!(ok = wait_sc(1))) break;
        tc_fence_after();
        issue_s(1, dq1, dk + kst * kK16);
        commit2(C::B_KE + kst);
        if (++kst == C::KST) {
          kst = 0;
          kph ^= 1;
        }
        bool firstA = true, firstB = true;
        int vprev = 0;
        uint32_t vprev_ph = 0;
        bool vprev_waited = false;
        for (int j = 0; j < hiB; ++j) {
          const bool uA = j < hiA, uA1 = j + 1 < hiA, uB1 = j + 1 < hiB;
          if (j > 0) {
            // O_B += P_B(j-1) V_{j-1}; tile B is the last reader of V_{j-1}.
            if (!(ok = wait_pf(1))) break;
            if (!vprev_waited && !(ok = mbar_wait(BAR(C::B_VF + vprev), vprev_ph, abort_flag, p.err))) break;
            tc_fence_after();
            issue_pv(1, firstB, dp1, dv + vprev * kV16);
            firstB = false;
            commit2(C::B_VE + vprev);
          }
          bool k_waited = false;
          if (uA1) {
            // S_A(j+1)
            if (!(ok = wait_sc(0))) break;
            if (!(ok = mbar_wait(BAR(C::B_KF + kst), kph, abort_flag, p.err))) break;
            k_waited = true;
            tc_fence_after();
            issue_s(0, dq0, dk + kst * kK16);
          }
          vprev_waited = false;
          if (uA) {
            // O_A += P_A(j) V_j
            if (!(ok = wait_pf(0))) break;
            if (!(ok = mbar_wait(BAR(C::B_VF + vst), vph, abort_flag, p.err))) break;
            vprev_waited = true;
            tc_fence_after();
            issue_pv(0, firstA, dp0, dv + vst * kV16);
            firstA = false;
          }
          if (uB1) {
            // S_B(j+1); tile B is the last reader of K_{j+1}.
            if (!(ok = wait_sc(1))) break;
            if (!k_waited && !(ok = mbar_wait(BAR(C::B_KF + kst), kph, abort_flag, p.err))) break;
            tc_fence_after();
            issue_s(1, dq1, dk + kst * kK16);
            commit2(C::B_KE + kst);
            if (++kst == C::KST) {
              kst = 0;
              kph ^= 1;
            }
          }
          vprev = vst;
          vprev_ph = vph;
          if (++vst == C::VST) {
            vst = 0;
            vph ^= 1;
          }
        }
        if (!ok) break;
        // O_B += P_B(hiB-1) V_{hiB-1}
        if (!(ok = wait_pf(1))) break;
        if (!vprev_waited && !(ok = mbar_wait(BAR(C::B_VF + vprev), vprev_ph, abort_flag, p.err))) break;
        tc_fence_after();
        issue_pv(1, firstB, dp1, dv + vprev * kV16);
        commit2(C::B_VE + vprev);
      }
      // Every product (which reads the other CTA's shared memory and writes its
      // TMEM) completes before this CTA reaches the final cluster barrier.
      tc_commit_pair(BAR(C::B_DONE));
      mbar_wait(BAR(C::B_DONE), 0, nullptr, p.err);
    }
    __syncwarp();
   }
  } else {
    // -------------------------------------------------------------- softmax warps
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kPairSoftmaxRegs));
    const int t = warp >> 2;
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;  // row within this CTA's part of the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const uint32_t scol = tmem + lane_off + static_cast<uint32_t>(t) * 128u;
    const uint32_t ocol = tmem + lane_off + 256u + static_cast<uint32_t>(t) * 128u;
    const uint32_t sc_bar = LEAD(C::B_SC + t), pf_bar = LEAD(C::B_PF + t);
    // Row r of P_t: keys 8c..8c+7 are 16-byte piece c % 8 of 128-byte chunk c / 8, swizzled.
    const uint32_t prow = sP + static_cast<uint32_t>(t) * C::PT_BYTES + static_cast<uint32_t>(r) * 128u;
    const uint32_t psw = static_cast<uint32_t>(r & 7);
    const float sl2 = p.scale_log2;
    const int Nkv = p.Nkv;
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    bool ok = true;
    uint32_t sf = 0, pvd = 0;
    for (int k = 0; ok && k * n_cl < n_units; ++k) {
      const int u = pair_unit_index(k, cid, n_cl);
      if (u >= n_units) continue;
      int q_tile0, jhi;
      {
        const PairUnit U = pair_unit<CAUSAL>(u, p);
        q_tile0 = U.q0 + t * 256 + kPairTileRows * static_cast<int>(rank);
        jhi = t == 0 ? U.hiA : U.hiB;
      }
      const int q_row = q_tile0 + r;
      float m = -INFINITY, l = 0.f;
      for (int j = 0; j < jhi; ++j) {
        ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_SF + t), sf, abort_flag, p.err));
        sf ^= 1;
        if (!ok) break;
        tc_fence_after();
        uint32_t sr[4][32];
#pragma unroll
        for (int i = 0; i < 4; ++i) tmem_ld_32x32b_x32(scol + i * 32, sr[i]);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 4; ++i) reg_fence(sr[i]);
        // S_t(j) is in registers: the next S_t may overwrite its columns.
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(sc_bar);

        const int kv0 = j * kPairBN;
        const bool need_mask = (kv0 + kPairBN > Nkv) || (CAUSAL && kv0 + kPairBN - 1 > q_tile0);
        if (need_mask) {
          const int hi_c = (CAUSAL ? min(Nkv, q_row + 1) : Nkv) - kv0;  // columns c < hi_c are kept
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (i * 32 + c >= hi_c) sr[i][c] = __float_as_uint(-INFINITY);
        }
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 32; c += 8)
#pragma unroll
            for (int w = 0; w < 4; ++w)
              mq[w] = fmax3(mq[w], __uint_as_float(sr[i][c + 2 * w]), __uint_as_float(sr[i][c + 2 * w + 1]));
        const float mx = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
        const float mb = mx * sl2;
        const bool raise = (m == -INFINITY) || (mb > m + kPairRescale);
        const float m_new = raise ? fmaxf(m, mb) : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = raise ? fast_exp2(m - m_use) : 1.f;
        if (j > 0) {
          // P_t(j-1) V_{j-1} has completed: its P buffer may be overwritten and O_t is stable.
          ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_PVD + t), pvd, abort_flag, p.err));
          pvd ^= 1;
          if (!ok) break;
          tc_fence_after();
        }
        // P = 2^(s * scale * log2 e - m), two columns per packed FMA, stored as
        // 16-bit pairs straight into the shared-memory operand; row sum in four
        // packed partial sums.
        const uint64_t sl2x2 = pack_f2(sl2, sl2), negm2 = pack_f2(-m_use, -m_use);
        uint64_t rs2[4] = {0, 0, 0, 0};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c8 = 0; c8 < 4; ++c8) {
            uint32_t w[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int c = c8 * 8 + q * 2;
              const float2 e = unpack_f2(
                  ffma_f2(pack_f2(__uint_as_float(sr[i][c]), __uint_as_float(sr[i][c + 1])), sl2x2, negm2));
              const float p0 = fast_exp2(e.x), p1 = fast_exp2(e.y);
              rs2[q] = fadd_f2(rs2[q], pack_f2(p0, p1));
              w[q] = pair_pack2<BF16>(p0, p1);
            }
            const uint32_t piece = static_cast<uint32_t>(i * 4 + c8);  // keys 8 piece .. 8 piece + 7
            const uint32_t addr = prow + (piece >> 3) * C::CHUNK_P + (((piece & 7u) ^ psw) << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(w[0]), "r"(w[1]), "r"(w[2]),
                         "r"(w[3])
                         : "memory");
          }
        const float2 r01 = unpack_f2(fadd_f2(rs2[0], rs2[1])), r23 = unpack_f2(fadd_f2(rs2[2], rs2[3]));
        l = l * alpha + ((r01.x + r01.y) + (r23.x + r23.y));
        m = m_new;
        // O_t *= alpha before P_t(j) V_j adds to it (S is no longer held here).
        const bool rescale = j > 0 && __any_sync(0xffffffffu, alpha != 1.f);
        if (rescale) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint32_t ov[32];
            tmem_ld_32x32b_x32(ocol + i * 32, ov);
            tmem_wait_ld();
            reg_fence(ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st_32x32b_x32(ocol + i * 32, ov);
          }
        }
        fence_proxy_async_smem();  // the tensor core reads P through the async proxy
        if (rescale) tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive_cluster(pf_bar);
      }
      if (!ok) break;
      // The unit's last P_t V completes O_t.
      ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_PVD + t), pvd, abort_flag, p.err));
      pvd ^= 1;
      if (!ok) break;
      // ------------------------------------------------------------ epilogue: O / l, LSE
      tc_fence_after();
      const PairUnit U = pair_unit<CAUSAL>(u, p);
      const float inv_l = 1.f / l;  // every row sees key 0, so l >= 1
      const bool row_ok = q_row < p.Nq;
      T *orow = reinterpret_cast<T *>(p.o) + static_cast<int64_t>(U.b) * p.o_sb + static_cast<int64_t>(U.h) * p.o_sh +
                static_cast<int64_t>(q_row) * p.o_sn;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(ocol + i * 32, ov);
        tmem_wait_ld();
        reg_fence(ov);
        uint32_t packed[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2)
          packed[c / 2] = pair_pack2<BF16>(__uint_as_float(ov[c]) * inv_l, __uint_as_float(ov[c + 1]) * inv_l);
        if (row_ok) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + i * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      }
      if (p.lse != nullptr && row_ok)
        p.lse[(static_cast<int64_t>(U.b) * p.Hq + U.h) * p.Nq + q_row] = (m + __log2f(l)) * kPairLn2;
      // O_t is read: the next unit's first P_t V may overwrite it once this
      // warp's next P-ready arrival says so.
    }
  }

  // After a timed-out wait, copies this CTA requested may still be landing in
  // its shared memory (rank 0 cannot wait for them all): give them time.
  if (*abort_flag != 0) {
    const uint64_t t0 = globaltimer_ns();
    while (globaltimer_ns() - t0 < 1000000ull) __nanosleep(1000);
  }
  tc_fence_before();
  cluster_sync();  // no product, copy or arrival of either CTA is still aimed at the other
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc_pair(tmem, 512);
  }
}

template <bool CAUSAL, bool BF16>
cudaError_t pair_launch_one(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv,
                            const PrefillParams &p, cudaStream_t stream) {
  auto kern = prefill_pair_kernel<CAUSAL, BF16>;
  constexpr uint32_t smem = PairCfg::SMEM_BYTES;
  // setmaxnreg redistributes the registers the CTA was launched with; refuse a
  // split larger than that pool (it would never be granted).
  cudaFuncAttributes fa{};
  cudaError_t e = cudaFuncGetAttributes(&fa, kern);
  if (e != cudaSuccess) return e;
  if (fa.numRegs * kPairThreads < 256 * kPairSoftmaxRegs + (kPairThreads - 256) * kPairOtherRegs)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(p.n_ctas));
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, tq, tk, tv, p);
}

template <bool CAUSAL, bool BF16>
int pair_clusters_one() {
  auto kern = prefill_pair_kernel<CAUSAL, BF16>;
  constexpr uint32_t smem = PairCfg::SMEM_BYTES;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem)) != cudaSuccess)
    return 0;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) != cudaSuccess) return 0;
  return n;
}

}  // namespace
}  // namespace attn
