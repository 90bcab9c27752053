// prefill_kernel.cuh -- fused attention forward (prefill) kernel for sm_103a.
//
// Included by prefill.cu (plain causal / full masks), prefill_masked.cu
// (sliding windows and ALiBi), prefill_rope.cu and prefill_rope_masked.cu
// (the same two with rotary position embeddings), which instantiate it with
// MASKED and ROPE false / true in separate translation units compiled in
// parallel.
//
// Persistent: one CTA per SM walks a sequence of units; a unit is TWO 128-row
// query tiles (rows q0..q0+255) of one (batch, q-head), so the tensor core
// always has one tile's matrix products to run while the other tile's softmax
// is computed:
//   warps 0-3   softmax warpgroup of tile 0, one thread per query row (TMEM lane)
//   warps 4-7   softmax warpgroup of tile 1
//   warp 8      TMA producer: both Q tiles once, then K and V tiles of 128 keys
//               into a ring of shared-memory stages (128-byte swizzle)
//   warp 9      TMEM allocator and tcgen05 MMA issuer (one thread), per KV tile j:
//                 S0_j = Q0 K_j^T;  O1 += P1_{j-1} V_{j-1};  S1_j = Q1 K_j^T;  O0 += P0_j V_j
//               (SS form for Q K^T, TS form with P read from TMEM for P V)
//   warps 10-11 rotary embeddings only (ROPE builds): rotate both Q tiles and
//               every K tile in shared memory once TMA has landed them, before
//               the MMA thread may read them
//   warp 10     variable length: also zeroes the rows past a sequence's end in
//               its last V tile before P V reads it (otherwise idle, like warp 11)
//
// The algorithm is the online softmax of "Skill: Write a Triton Attention
// Kernel" (Required reasoning process, steps 4-9): running max m and sum l in
// fp32, O and l rescaled by alpha = exp(m_old - m_new) before a block is
// added, O / l once after the loop, lse = m + ln l.  Details of this kernel:
//   * scores are kept in base-2 units (scale * log2 e folded into one FMA), so
//     the exponential is one ex2; the LSE is converted back on store;
//   * the running max of a row is only raised when the block max exceeds it
//     by more than 8 (base 2).  P = 2^(s - m) then stays below 2^8, the rescale
//     of O (TMEM load, multiply, store) is skipped for most blocks, and O / l is
//     unchanged because O and l always share the same m;
//   * the causal mask (key j kept for query i iff j <= i) and the key-length
//     mask set scores to -inf before the max; only tiles that straddle the
//     diagonal or the end of the keys pay for it, and KV tiles past the
//     diagonal of a query tile are never computed for it;
//   * P (16-bit) overwrites the first half of its S columns in TMEM; in-order
//     execution of the MMAs keeps the next S from landing before P V has read P,
//     and makes P_i(j-1) V_{j-1} complete before S_i(j) is signalled, so the
//     softmax warpgroup may rescale O_i as soon as it sees S_i(j).
//
// TMEM columns (512): S0/P0 [0,128) S1/P1 [128,256) O0 [256,256+D) O1 [256+D,256+2D).
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <type_traits>

#include "attn_internal.h"
#include "ptx.cuh"
#include "rope.cuh"

namespace attn {
namespace {

constexpr int kBM = kPrefillBM;  // rows per query tile
constexpr int kBN = kPrefillBN;  // keys per KV tile
// 12 warps in every build.  (A 14-warp rotary build with four rotation
// warps was tried: its launch caps every thread at 128 registers and the
// warps then spill.)
template <bool ROPE>
constexpr int kThreadsFor = 384;
template <bool ROPE>
constexpr int kRopeWarps = 2;
constexpr float kLn2 = 0.693147180559945309f;
constexpr float kRescaleThreshold = 8.0f;  // base-2 units
constexpr int kSoftmaxRegs = 200;
constexpr int kUnlimited = 0x3fffffff;  // "no window bound" (large, yet safe to add small offsets to)
// Registers of the non-softmax warps after setmaxnreg: what is left of the
// launch's pool after the two softmax warpgroups.
template <bool ROPE>
constexpr int kOtherRegsFor = 96;

template <int D, bool CAUSAL, bool ROPE>
struct Cfg {
  static constexpr int KCH = D / 64;                  // 128-byte chunks along D
  // Shared-memory stages of the K and V rings.  The causal and the rotary
  // builds keep the K ring one stage deeper than the V ring and load K one
  // tile ahead of V, so that K_{j+1} has landed (and, rotary, been rotated)
  // before the MMA thread waits for it ahead of P0_j V_j (D = 128: 3 x 32 KB of
  // K + 2 x 32 KB of V + 64 KB of Q fit in 227 KB).  Measured A/B on one GPU:
  // causal N = 8192 +2 % at D = 128 and +1-2 % at D = 64 (+2-6 % at N = 2048),
  // while at D = 128 non-causal and the cross-attention workload ran 3-4 %
  // slower (V then arrives later), so the plain non-causal builds keep equal
  // rings.
  static constexpr int KST = (D == 128) ? ((CAUSAL || ROPE) ? 3 : 2) : ((CAUSAL || ROPE) ? 4 : 3);
  static constexpr int VST = (D == 128) ? 2 : 3;
  static constexpr bool SPLIT = KST != VST;           // the two rings advance separately
  static constexpr uint32_t CHUNK_Q = kBM * 128;      // bytes of one 64-column chunk of a Q tile
  static constexpr uint32_t CHUNK_KV = kBN * 128;
  static constexpr uint32_t QT_BYTES = kBM * D * 2;   // one Q tile
  static constexpr uint32_t KV_BYTES = kBN * D * 2;
  // TMEM column of S_t / P_t and of O_t for query tile t
  static __device__ __forceinline__ uint32_t s_col(int t) { return static_cast<uint32_t>(t) * 128u; }
  static __device__ __forceinline__ uint32_t o_col(int t) { return 256u + static_cast<uint32_t>(t) * D; }
  static constexpr uint32_t TMEM_COLS = 512;
  static constexpr uint32_t OFF_Q = 0;
  static constexpr uint32_t OFF_K = OFF_Q + 2 * QT_BYTES;
  static constexpr uint32_t OFF_V = OFF_K + KST * KV_BYTES;
  static constexpr uint32_t OFF_BAR = OFF_V + VST * KV_BYTES;
  // barrier indices
  static constexpr int B_Q = 0;
  static constexpr int B_KF = 1;                       // + K stage
  // K stage released: K_j is free, and so is V_{j-1} (every product that
  // reads V_{j-1} is issued before the release of K_j, so one commit frees both)
  static constexpr int B_KE = B_KF + KST;              // + K stage
  static constexpr int B_VF = B_KE + KST;              // + V stage
  static constexpr int B_SF = B_VF + VST;              // + tile (2): S_i(j) computed
  static constexpr int B_PF = B_SF + 2;                // + tile (2): P_i(j) stored (and O_i rescaled)
  static constexpr int B_OD = B_PF + 2;                // + tile (2): last P_i V done
  static constexpr int B_DONE = B_OD + 2;              // every MMA completed
  static constexpr int B_VZ = B_DONE + 1;              // variable length: V rows past the sequence zeroed
  static constexpr int B_VT = B_VZ + 1;                // variable length: the tail V tile has landed
  static constexpr int B_QR = B_VT + 1;                // + Q tile (2): rotary: Q tile rotated
  static constexpr int B_KR = B_QR + 2;                // + K stage: rotary: K tile rotated
  static constexpr int NBAR = B_KR + KST;
  static constexpr uint32_t OFF_MISC = OFF_BAR + NBAR * 8;
  static constexpr uint32_t OFF_ROPE = (OFF_MISC + 16 + 7) & ~7u;  // rotary turn steps, uint64 [D/2]
  static constexpr uint32_t SMEM_USED = OFF_ROPE + (D / 2) * 8;
  // + slack for 1024-byte alignment; at least 116 KB so that only one CTA (which
  // holds all 512 TMEM columns) is resident per SM.
  static constexpr uint32_t SMEM_BYTES = (SMEM_USED + 1024 > 116u * 1024) ? SMEM_USED + 1024 : 116u * 1024;
  static_assert(256 + 2 * D <= TMEM_COLS, "TMEM budget");
  static_assert(SMEM_BYTES <= 227u * 1024, "shared memory budget");
};

__device__ __forceinline__ void tma_tile(uint32_t dst, const CUtensorMap *map, int d, int n, int h, int b,
                                         uint32_t slots, uint32_t bar) {
  const int sn = slots & 3, sh = (slots >> 2) & 3;
  const int c1 = (sn == 1) ? n : (sh == 1) ? h : b;
  const int c2 = (sn == 2) ? n : (sh == 2) ? h : b;
  const int c3 = (sn == 3) ? n : (sh == 3) ? h : b;
  tma_load_4d(dst, map, d, c1, c2, c3, bar);
}
// tma_tile for data read once (Q): evicted from L2 first, so that the K and V
// tiles every query tile of a head group re-reads stay resident.
__device__ __forceinline__ void tma_tile_once(uint32_t dst, const CUtensorMap *map, int d, int n, int h, int b,
                                              uint32_t slots, uint32_t bar) {
  const int sn = slots & 3, sh = (slots >> 2) & 3;
  const int c1 = (sn == 1) ? n : (sh == 1) ? h : b;
  const int c2 = (sn == 2) ? n : (sh == 2) ? h : b;
  const int c3 = (sn == 3) ? n : (sh == 3) ? h : b;
  tma_load_4d_hint(dst, map, d, c1, c2, c3, bar, l2_policy_evict_first());
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

template <int N>
__device__ __forceinline__ void setmaxnreg_inc() {
  asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(N));
}
template <int N>
__device__ __forceinline__ void setmaxnreg_dec() {
  asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(N));
}

// One unit of work: a pair of 128-row query tiles of one (batch, q head), with
// the KV tiles each tile needs.
struct Unit {
  int h, b, hk, q0, q_base, k_base, Nq, Nkv, bc;  // bc: batch coordinate of the tensor maps
  int lo0, hi0, lo1, hi1, J0, J1, j_tail;         // KV tile bands [lo_t, hi_t) and their hull [J0, J1)
  bool zero_v;                                    // variable length: tail V tile to be zeroed
  int kind;
};
constexpr int kRun = 0;    // compute the unit
constexpr int kSkip = 1;   // nothing to do (variable length: pair past the sequence, or bad offsets)
constexpr int kEmpty = 2;  // variable length, no keys: O = 0 and LSE = -inf
constexpr int kBadIndex = 4;  // with kSkip: the sequence offsets were out of range

// Every role of the CTA derives the same units in the same order, so the
// pipelines (TMA ring, S/P/O barriers) stay in step across units.
template <bool CAUSAL, bool VARLEN>
__device__ __forceinline__ Unit make_unit(int u, const PrefillParams &p, int win_l, int win_r) {
  Unit U;
  const int hb = p.Hq * p.B;
  const int z = u / hb, rem = u - z * hb;
  U.h = rem % p.Hq;
  U.b = rem / p.Hq;
  const int pair = CAUSAL ? (p.n_qtiles - 1 - z) : z;
  U.hk = U.h / p.group;
  U.q0 = pair * 2 * kBM;
  U.q_base = 0;
  U.k_base = 0;
  U.Nq = p.Nq;
  U.Nkv = p.Nkv;
  U.bc = U.b;
  U.kind = kRun;
  if constexpr (VARLEN) {
    const int qs = p.cu_q[U.b], qe = p.cu_q[U.b + 1], ks = p.cu_k[U.b], ke = p.cu_k[U.b + 1];
    if (qs < 0 || qe < qs || qe > p.total_q || qe - qs > p.Nq || ks < 0 || ke < ks || ke > p.total_k ||
        ke - ks > p.Nkv) {
      U.kind = kSkip | kBadIndex;
      U.Nq = U.Nkv = 0;
    } else {
      U.q_base = qs;
      U.k_base = ks;
      U.Nq = qe - qs;
      U.Nkv = ke - ks;
      U.bc = 0;
      if (U.q0 >= U.Nq) U.kind = kSkip;
      else if (U.Nkv == 0) U.kind = kEmpty;
    }
  }
  // Key band of a query row i: i - win_l <= j <= i + win_r (kUnlimited: no
  // bound on that side); causal fixes win_r at 0.  Query tile t needs KV tiles
  // [lo_t, hi_t); tiles outside the band are never loaded or computed.  Tile 1
  // lies at or after tile 0 (lo0 <= lo1, hi0 <= hi1).
  int lo[2] = {0, 0}, hi[2] = {0, 0};
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int qa = U.q0 + t * kBM;  // first row of the tile
    const int kmin = win_l == kUnlimited ? 0 : max(0, qa - win_l);
    const int kmax = win_r == kUnlimited ? U.Nkv - 1 : min(U.Nkv - 1, qa + kBM - 1 + win_r);
    lo[t] = kmin / kBN;
    hi[t] = kmax < kmin ? lo[t] : kmax / kBN + 1;
  }
  U.lo0 = lo[0];
  U.hi0 = hi[0];
  U.lo1 = lo[1];
  U.hi1 = hi[1];
  const bool has_t0 = lo[0] < hi[0], has_t1 = lo[1] < hi[1];
  U.J0 = has_t0 ? (has_t1 ? min(lo[0], lo[1]) : lo[0]) : (has_t1 ? lo[1] : 0);
  U.J1 = has_t0 ? (has_t1 ? max(hi[0], hi[1]) : hi[0]) : (has_t1 ? hi[1] : 0);
  if (U.kind != kRun) U.J1 = U.J0;
  const int nkv_all = (U.Nkv + kBN - 1) / kBN;
  // Variable length: the last KV tile runs past the sequence and is used here.
  U.j_tail = nkv_all - 1;
  U.zero_v = VARLEN && U.kind == kRun && (U.Nkv % kBN) != 0 && U.J1 == nkv_all && U.J0 <= U.j_tail;
  return U;
}

// The unit a CTA runs in round k: rounds of gridDim.x units in longest-first
// order, dealt alternately forwards and backwards over the CTAs, which evens
// out the CTAs' total work (the sum of the causal lengths).
__device__ __forceinline__ int unit_index(int k, int c, int g) { return k * g + ((k & 1) ? g - 1 - c : c); }

// Persistent: one CTA per SM walks rounds of units (longest first).
// While the softmax warps store one unit's O, the next unit's Q is already
// loaded and its first Q K^T product runs: Q is reloaded as soon as the last
// S product of a unit completed, and a tile's O columns are only
// overwritten by the next unit's first P V, which waits for that tile's
// softmax warps -- the same warps that ran the epilogue.
//
// VARLEN: the batch is packed; sequence b's rows are found through cu_q / cu_k
// (see PrefillParams), tensor maps span the packed tensors, and the last V tile
// of a sequence -- whose tail rows belong to the next sequence -- gets those
// rows zeroed by warp 10 before P V reads it, so nothing from another sequence
// (not even a non-finite value times a zero weight) reaches the result.
// ROPE: warps 10 and 11 rotate the Q tiles and each K tile in shared memory
// (rows at their positions within the sequence); the MMA thread waits on the
// "rotated" barriers instead of the TMA ones.
template <int D, bool CAUSAL, bool BF16, bool VARLEN, bool MASKED, bool ROPE>
__global__ void __launch_bounds__(kThreadsFor<ROPE>, 1)
    prefill_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                       const __grid_constant__ CUtensorMap tmV, const __grid_constant__ PrefillParams p) {
  using C = Cfg<D, CAUSAL, ROPE>;
  constexpr int KST = C::KST, VST = C::VST;
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
  // Without MASKED both bounds are compile-time constants and the band code
  // folds away (the plain kernel keeps its shorter softmax loop).
  const int win_l = (!MASKED || p.window_left < 0) ? kUnlimited : p.window_left;
  const int win_r = CAUSAL ? 0 : ((!MASKED || p.window_right < 0) ? kUnlimited : p.window_right);
  const int u_first = blockIdx.x, u_step = gridDim.x, n_units = p.n_units;

  if (threadIdx.x == 0) {
    mbar_init(BAR(C::B_Q), 1);
    for (int s = 0; s < KST; ++s) {
      mbar_init(BAR(C::B_KF + s), 1);
      mbar_init(BAR(C::B_KE + s), 1);
    }
    for (int s = 0; s < VST; ++s) mbar_init(BAR(C::B_VF + s), 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(BAR(C::B_SF + i), 1);
      mbar_init(BAR(C::B_PF + i), 4);  // one arrival per softmax warp
      mbar_init(BAR(C::B_OD + i), 1);
    }
    mbar_init(BAR(C::B_DONE), 1);
    mbar_init(BAR(C::B_VZ), 1);
    mbar_init(BAR(C::B_VT), 1);
    mbar_init(BAR(C::B_QR), kRopeWarps<ROPE>);  // one arrival per rotating warp
    mbar_init(BAR(C::B_QR + 1), kRopeWarps<ROPE>);
    for (int s = 0; s < KST; ++s) mbar_init(BAR(C::B_KR + s), kRopeWarps<ROPE>);
    *abort_flag = 0;
    fence_barrier_init();
    fence_proxy_async_smem();
  }
  if (warp == 9) {
    tmem_alloc(smem_u32(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  if (warp == 8 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if constexpr (ROPE) {
    uint64_t *fs = reinterpret_cast<uint64_t *>(smem + C::OFF_ROPE);
    for (int i = threadIdx.x; i < D / 2; i += kThreadsFor<ROPE>) fs[i] = p.rope_f[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp >= 8) {
    setmaxnreg_dec<kOtherRegsFor<ROPE>>();
    if (warp == 8) {
      // ---------------------------------------------------------- TMA producer
      if (lane == 0) {
        int issued_k = 0, issued_v = 0, nq = 0;  // K, V tiles and Q pairs issued so far
        int kst = 0, vst = 0;                    // ring stages of the next K and V tiles
        uint32_t kph = 0, vph = 0;               // their phases
        int q_wait = -1;                         // what frees Q: -1 nothing, -2 the last Q load, else KE stage
        uint32_t q_phase = 0;
        bool ok = true;
        // K (or V) tile j of unit U into the next stage of its ring, once the
        // stage's previous tile (KST or VST loads back) has been released.
        auto load_k = [&](const Unit &U, int j) -> bool {
          if (issued_k >= KST && !mbar_wait(BAR(C::B_KE + kst), kph ^ 1, abort_flag, p.err)) return false;
          mbar_arrive_expect_tx(BAR(C::B_KF + kst), C::KV_BYTES);
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            tma_tile(sK + kst * C::KV_BYTES + c * C::CHUNK_KV, &tmK, c * 64, U.k_base + j * kBN, U.hk, U.bc,
                     p.slots_k, BAR(C::B_KF + kst));
          ++issued_k;
          q_wait = kst;
          q_phase = kph;
          if (++kst == KST) {
            kst = 0;
            kph ^= 1;
          }
          return true;
        };
        // V tile number issued_v (counted over the whole walk) reuses the stage
        // of V tile issued_v - VST, which is released with K tile m =
        // issued_v - VST + 1 (already loaded: K runs level with or ahead of V).
        // Its release barrier cannot be a phase further on: that would need K
        // tile m + KST, which is not loaded yet.
        auto load_v = [&](const Unit &U, int j) -> bool {
          if (issued_v >= VST) {
            const int m = issued_v - VST + 1;
            if (!mbar_wait(BAR(C::B_KE + m % KST), (m / KST) & 1, abort_flag, p.err)) return false;
          }
          mbar_arrive_expect_tx(BAR(C::B_VF + vst), C::KV_BYTES);
#pragma unroll
          for (int c = 0; c < C::KCH; ++c)
            tma_tile(sV + vst * C::KV_BYTES + c * C::CHUNK_KV, &tmV, c * 64, U.k_base + j * kBN, U.hk, U.bc,
                     p.slots_v, BAR(C::B_VF + vst));
          ++issued_v;
          if (++vst == VST) {
            vst = 0;
            vph ^= 1;
          }
          return true;
        };
        for (int k = 0; ok && k * u_step < n_units; ++k) {
          const int u = unit_index(k, u_first, u_step);
          if (u >= n_units) continue;
          const Unit U = make_unit<CAUSAL, VARLEN>(u, p, win_l, win_r);
          if (U.kind != kRun) continue;
          // With windows (MASKED), a unit without KV tiles (every row's band
          // empty) has no product that reads Q, so it gets no Q load.  Each Q load
          // is then followed by S products, and the release below implies the MMA
          // thread has passed its wait for the previous Q: the Q barrier never
          // runs two phases ahead of that wait.  Without windows every unit has
          // KV tiles.
          if constexpr (MASKED) {
            if (U.J0 == U.J1) continue;
          }
          // The previous unit's Q is free once its last S product completed: the
          // release of its last K stage (in-order MMAs: every S product before it
          // is complete too), or -- for a unit without KV tiles -- once its Q landed.
          if (q_wait >= 0) ok = mbar_wait(BAR(C::B_KE + q_wait), q_phase, abort_flag, p.err);
          else if (q_wait == -2) ok = mbar_wait(BAR(C::B_Q), (nq - 1) & 1, abort_flag, p.err);
          if (!ok) break;
          mbar_arrive_expect_tx(BAR(C::B_Q), 2 * C::QT_BYTES);
#pragma unroll
          for (int t = 0; t < 2; ++t)
#pragma unroll
            for (int c = 0; c < C::KCH; ++c)
              tma_tile_once(sQ + t * C::QT_BYTES + c * C::CHUNK_Q, &tmQ, c * 64, U.q_base + U.q0 + t * kBM, U.h,
                            U.bc, p.slots_q, BAR(C::B_Q));
          ++nq;
          if constexpr (C::SPLIT) {
            // The K ring is deeper: K_{j+1} is requested before V_j, so each K
            // tile lands (and is rotated) well before its first product.
            if (U.J0 < U.J1 && !(ok = load_k(U, U.J0))) break;
            for (int j = U.J0; j < U.J1; ++j) {
              if (j + 1 < U.J1 && !(ok = load_k(U, j + 1))) break;
              if (!(ok = load_v(U, j))) break;
            }
          } else {
            for (int j = U.J0; j < U.J1; ++j) {
              if (!(ok = load_k(U, j))) break;
              if (!(ok = load_v(U, j))) break;
            }
          }
          if (!ok) break;
          if (U.J0 == U.J1) q_wait = -2;
        }
        if (!ok) {
          // Let every copy already issued land before shared memory is released.
          if (nq > 0) mbar_wait(BAR(C::B_Q), (nq - 1) & 1, nullptr, p.err);
          for (int i = max(0, issued_k - KST); i < issued_k; ++i)
            mbar_wait(BAR(C::B_KF + i % KST), (i / KST) & 1, nullptr, p.err);
          for (int i = max(0, issued_v - VST); i < issued_v; ++i)
            mbar_wait(BAR(C::B_VF + i % VST), (i / VST) & 1, nullptr, p.err);
        }
      }
      __syncwarp();
    } else if (warp == 9) {
      // ---------------------------------------------------------- MMA issuer
      if (lane == 0) {
        constexpr uint32_t idesc_qk = idesc_f16(BF16, kBM, kBN, false, false);
        constexpr uint32_t idesc_pv = idesc_f16(BF16, kBM, D, false, true);
        // Shared-memory descriptors are formed once; each MMA adds a compile-time
        // offset (in 16-byte units) to the start-address field.  All operands lie
        // below 256 KB, so the 14-bit field never carries into the next one.
        const uint64_t dq0 = smem_desc_sw128(sQ, 16, 1024), dq1 = smem_desc_sw128(sQ + C::QT_BYTES, 16, 1024);
        const uint64_t dk = smem_desc_sw128(sK, 16, 1024), dv = smem_desc_sw128(sV, C::CHUNK_KV, 1024);
        constexpr uint32_t kStage16 = C::KV_BYTES >> 4;
        auto issue_s = [&](int t, uint64_t qd, uint64_t kd) {
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            // Q and K are K-major: 16 elements (32 B) per MMA inside a 128-byte swizzle row.
            mma_ss(tmem + C::s_col(t), qd + (((kk / 4) * C::CHUNK_Q + (kk % 4) * 32) >> 4),
                   kd + (((kk / 4) * C::CHUNK_KV + (kk % 4) * 32) >> 4), idesc_qk, kk > 0 ? 1u : 0u);
          }
          tc_commit(BAR(C::B_SF + t));
        };
        auto issue_pv = [&](int t, bool first, uint64_t vd) {
#pragma unroll
          for (int kk = 0; kk < kBN / 16; ++kk) {
            // V is MN-major: 16 keys per MMA = 16 rows of 128 B; D in 64-column blocks CHUNK_KV apart.
            mma_ts(tmem + C::o_col(t), tmem + C::s_col(t) + kk * 8, vd + ((kk * 16 * 128) >> 4), idesc_pv,
                   (!first || kk > 0) ? 1u : 0u);
          }
        };
        // Q and K may be read once they landed (or, with rotary embeddings,
        // once warps 10-11 rotated them).
        constexpr int kQReady = ROPE ? C::B_QR : C::B_Q;
        const int kKReady = (ROPE && p.rope_k) ? C::B_KR : C::B_KF;
        bool ok = true;
        int kst = 0;                // K ring stage of the next KV tile
        uint32_t kph = 0;           // its phase
        // V ring stage and phase of the next KV tile: the same variables as K's
        // unless the rings have different depths.
        int vst_own = 0;
        uint32_t vph_own = 0;
        int &vst = C::SPLIT ? vst_own : kst;
        uint32_t &vph = C::SPLIT ? vph_own : kph;
        uint32_t pf0 = 0, pf1 = 0;  // parities of the P-ready barriers
        uint32_t q_par = 0;         // parity of the current unit's Q barriers
        bool q1_wait = false;       // rotary: Q1's barrier not yet waited for in this unit
        int nq = 0, nvz = 0;        // units started; tail V tiles zeroed
        for (int k = 0; ok && k * u_step < n_units; ++k) {
          const int u = unit_index(k, u_first, u_step);
          if (u >= n_units) continue;
          const Unit U = make_unit<CAUSAL, VARLEN>(u, p, win_l, win_r);
          if (U.kind != kRun) continue;
          const int lo0 = U.lo0, hi0 = U.hi0, lo1 = U.lo1, hi1 = U.hi1, J0 = U.J0, J1 = U.J1;
          // V of KV tile j (ring stage s, phase f) has landed (and, for a sequence's
          // tail tile, been zeroed past the end: this thread, which follows the stage
          // phases in order, tells warp 10 when the tail tile is in and waits for it
          // to clear the rows).
          auto wait_v = [&](int j, int s, uint32_t f) -> bool {
            if (!mbar_wait(BAR(C::B_VF + s), f, abort_flag, p.err)) return false;
            if (!(U.zero_v && j == U.j_tail)) return true;
            mbar_arrive(BAR(C::B_VT));
            const bool zeroed = mbar_wait(BAR(C::B_VZ), nvz & 1, abort_flag, p.err);
            ++nvz;
            return zeroed;
          };
          if constexpr (MASKED) {
            // A unit without KV tiles gets no Q load (see the producer) and must
            // not wait for one: the next unit's Q may already have landed, so not
            // even the Q barrier's previous phase can be waited for.  It waits
            // instead on the all-done barrier's (never incomplete) phase before
            // its first, which passes at once.
            const bool has_kv = J0 < J1;
            q_par = nq & 1;
            q1_wait = ROPE && has_kv;
            if (!(ok = mbar_wait(BAR(has_kv ? kQReady : C::B_DONE), has_kv ? q_par : 1u, abort_flag, p.err)))
              break;
            nq += has_kv ? 1 : 0;
          } else {
            q_par = nq & 1;
            q1_wait = ROPE;
            if (!(ok = mbar_wait(BAR(kQReady), q_par, abort_flag, p.err))) break;
            ++nq;
          }
          // Rotary: Q1 is signalled after Q0 and waited for before the first S1
          // product, once per Q load.  A unit without S1 products waits for it
          // at once: the next unit's Q can only be loaded after this unit's last
          // S product, so waiting here keeps the barrier within one phase of
          // this wait (a wait left to the unit's end could see it two ahead).
          auto wait_q1 = [&]() -> bool {
            if (!q1_wait) return true;
            q1_wait = false;
            return mbar_wait(BAR(C::B_QR + 1), q_par, abort_flag, p.err);
          };
          if (ROPE && lo1 >= hi1 && !(ok = wait_q1())) break;
          bool v_waited = false;  // V of tile j-1 already waited for (by P0 V)
          bool h1p = false;       // tile 1 uses KV tile j-1
          bool first0 = true, first1 = true;
          int vsp = 0;            // V ring stage of j-1
          uint32_t vpph = 0;      // and its phase
          // S0_j is issued at the end of step j-1, right behind P0_{j-1} V_{j-1} (K_j
          // having been waited for before P0_{j-1}): the thread's next tcgen05
          // instruction after a P V product is the following S product, so the
          // tensor pipe gets no gap there.
          if (J0 < J1) {
            ok = mbar_wait(BAR(kKReady + kst), kph, abort_flag, p.err);
            if (ok && J0 >= lo0 && J0 < hi0) {
              tc_fence_after();
              issue_s(0, dq0, dk + kst * kStage16);
            }
          }
          for (int j = J0; ok && j < J1; ++j) {
            const bool h0 = j >= lo0 && j < hi0, h1 = j >= lo1 && j < hi1;
            const int kst1 = kst + 1 == KST ? 0 : kst + 1;    // K ring stage of j + 1
            const uint32_t kph1 = kst1 == 0 ? kph ^ 1 : kph;  // and its phase
            const bool h0n = j + 1 >= lo0 && j + 1 < hi0;  // tile 0 uses KV tile j + 1
            if (h1p) {
              // O1 += P1_{j-1} V_{j-1}: tile 1 is the last user of V_{j-1} (released with K_j below)
              if (!(ok = mbar_wait(BAR(C::B_PF + 1), pf1, abort_flag, p.err))) break;
              pf1 ^= 1;
              if (!v_waited && !(ok = wait_v(j - 1, vsp, vpph))) break;
              tc_fence_after();
              issue_pv(1, first1, dv + vsp * kStage16);
              first1 = false;
            }
            if (h1) {
              if constexpr (ROPE) {
                if (!(ok = wait_q1())) break;
              }
              tc_fence_after();
              issue_s(1, dq1, dk + kst * kStage16);
            }
            tc_commit(BAR(C::B_KE + kst));  // both S products that read K_j, and every P V of V_{j-1}, are issued
            v_waited = false;
            if (j + 1 < J1 && !(ok = mbar_wait(BAR(kKReady + kst1), kph1, abort_flag, p.err))) break;
            if (h0) {
              // O0 += P0_j V_j
              if (!(ok = mbar_wait(BAR(C::B_PF + 0), pf0, abort_flag, p.err))) break;
              pf0 ^= 1;
              if (!(ok = wait_v(j, vst, vph))) break;
              v_waited = true;
              tc_fence_after();
              issue_pv(0, first0, dv + vst * kStage16);
              first0 = false;
              if (j == hi0 - 1) tc_commit(BAR(C::B_OD + 0));
            } else if (!h1) {
              // A tile between the two bands: nothing reads V_j.  Its copy must land
              // before the stage is handed back (with K_{j+1}) for the next one.
              if (!(ok = wait_v(j, vst, vph))) break;
            }
            if (j + 1 < J1 && h0n) {
              tc_fence_after();
              issue_s(0, dq0, dk + kst1 * kStage16);  // S0_{j+1}
            }
            h1p = h1;
            vsp = vst;
            vpph = vph;
            if constexpr (C::SPLIT) {
              if (++vst == VST) {
                vst = 0;
                vph ^= 1;
              }
            }
            kst = kst1;
            kph = kph1;
          }
          if (ok && h1p) {
            // the last P1 V of tile 1 (its band ends the ring)
            ok = mbar_wait(BAR(C::B_PF + 1), pf1, abort_flag, p.err) && (v_waited || wait_v(J1 - 1, vsp, vpph));
            if (ok) {
              pf1 ^= 1;
              tc_fence_after();
              issue_pv(1, first1, dv + vsp * kStage16);
              tc_commit(BAR(C::B_OD + 1));
            }
          }
          if (!ok) break;
          // With windows (MASKED), a query tile whose band holds no key gets no
          // product and no O-done signal: its softmax warps store zeros without
          // waiting.  (Signalled here, a run of such units would let this thread
          // complete the barrier's phases faster than the softmax warps consume
          // them.)  Without windows no band is empty.
          if constexpr (!MASKED) {
            if (lo0 >= hi0) tc_commit(BAR(C::B_OD + 0));
            if (lo1 >= hi1) tc_commit(BAR(C::B_OD + 1));
          }
        }
        tc_commit(BAR(C::B_DONE));
        mbar_wait(BAR(C::B_DONE), 0, nullptr, p.err);
      }
      __syncwarp();
    } else {
      // ---------------------------------------------------------- warps 10-11
      // Rotary embeddings (ROPE): both warps rotate each unit's Q tiles and then
      // its K tiles, in the order the producer loads them.  Variable length:
      // warp 10 then zeroes the rows past the sequence in the unit's tail V tile.
      constexpr int NT = kRopeWarps<ROPE> * 32;  // rotating threads
      constexpr int G = D / 16;             // groups of 8 pairs per row
      constexpr int RPT = kBM * G / NT;     // consecutive rows per thread in a 128-row tile
      const int tid = threadIdx.x - 320;    // 0 .. NT - 1
      const int g = tid % G, rb = tid / G;  // this thread's pair group and row block
      float c1[8], s1[8];                   // cos and sin of one position's angle of the group's 8 pairs
      const uint64_t *fs = reinterpret_cast<const uint64_t *>(smem + C::OFF_ROPE);
      if constexpr (ROPE) {
#pragma unroll
        for (int i = 0; i < 8; ++i) rope_sincos(1u, fs[8 * g + i], &s1[i], &c1[i]);
      }
      // Rotates rows [rb * RPT, rb * RPT + RPT) of the 128-row tile at `tile`
      // (64-column blocks CHUNK bytes apart, 128-byte swizzle); row r sits at
      // position pos0 + r.
      auto rotate_rows = [&](auto inter, uint8_t *tile, uint32_t chunk_bytes, int pos0) {
        constexpr bool IL = decltype(inter)::value;
        int ca, cb;
        rope_group_chunks<D, IL>(g, &ca, &cb);
        float cs[8], sn[8];
        const uint32_t r0 = static_cast<uint32_t>(rb * RPT);
#pragma unroll
        for (int i = 0; i < 8; ++i) rope_sincos(static_cast<uint32_t>(pos0) + r0, fs[8 * g + i], &sn[i], &cs[i]);
        RopeWalk wk;
        wk.start(cs, sn);
        uint8_t *ta = tile + (ca >> 3) * chunk_bytes + r0 * 128, *tb = tile + (cb >> 3) * chunk_bytes + r0 * 128;
        ca &= 7;
        cb &= 7;
#pragma unroll 2
        for (int rr = 0; rr < RPT; ++rr) {
          const uint32_t sw = (r0 + rr) & 7;  // 128-byte swizzle of the row
          uint4 *pa = reinterpret_cast<uint4 *>(ta + rr * 128 + ((ca ^ sw) << 4));
          uint4 *pb = reinterpret_cast<uint4 *>(tb + rr * 128 + ((cb ^ sw) << 4));
          uint4 A = *pa, Bv = *pb;
          rope_rotate_group<BF16, IL>(A, Bv, wk.cs, wk.sn);
          *pa = A;
          *pb = Bv;
          wk.step(c1, s1);
        }
      };
      auto rotate_tile = [&](uint8_t *tile, uint32_t chunk_bytes, int pos0) {
        if (p.rope_inter) rotate_rows(std::true_type{}, tile, chunk_bytes, pos0);
        else rotate_rows(std::false_type{}, tile, chunk_bytes, pos0);
      };
      const bool rope_k = p.rope_k != 0;     // K tiles rotated here (else given rotated)
      int st = 0, nq = 0, pos = 0, nvz = 0;  // K ring stage, Q loads, V ring position, tails zeroed
      uint32_t ph = 0;
      bool ok = true;
      for (int k = 0; ok && k * u_step < n_units; ++k) {
        if constexpr (!ROPE && !VARLEN) break;
        const int u = unit_index(k, u_first, u_step);
        if (u >= n_units) continue;
        const Unit U = make_unit<CAUSAL, VARLEN>(u, p, win_l, win_r);
        if (U.kind != kRun) continue;
        if constexpr (ROPE) {
          if (U.J0 < U.J1) {  // the producer loads Q only for units with KV tiles
            ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_Q), nq & 1, abort_flag, p.err));
            ++nq;
            if (!ok) break;
            // Tile 0 first, signalled on its own: the unit's first product (S0)
            // needs only Q0 and can run while Q1 is rotated.
            rotate_tile(smem + C::OFF_Q, C::CHUNK_Q, U.q0);
            fence_proxy_async_smem();  // the tensor core reads the rotated rows
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::B_QR));
            rotate_tile(smem + C::OFF_Q + C::QT_BYTES, C::CHUNK_Q, U.q0 + kBM);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::B_QR + 1));
          }
          for (int j = U.J0; ok && rope_k && j < U.J1; ++j) {
            ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_KF + st), ph, abort_flag, p.err));
            if (!ok) break;
            rotate_tile(smem + C::OFF_K + st * C::KV_BYTES, C::CHUNK_KV, j * kBN);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::B_KR + st));
            if (++st == KST) {
              st = 0;
              ph ^= 1;
            }
          }
          if (!ok) break;
        }
        if constexpr (VARLEN) {
          if (warp == 10 && U.zero_v) {
            const int st_t = (pos + U.j_tail - U.J0) % VST;  // V ring stage of the tail tile
            const bool landed = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_VT), nvz & 1, abort_flag, p.err));
            ++nvz;
            if (!landed) break;
            const int r0 = U.Nkv % kBN;  // rows r0..127 of the tile lie past the sequence
            uint8_t *vt = smem + C::OFF_V + st_t * C::KV_BYTES;
            const int pieces = (kBN - r0) * 8;  // 16-byte pieces per 128-byte row chunk
            for (int c = 0; c < C::KCH; ++c)
              for (int i = lane; i < pieces; i += 32)
                *reinterpret_cast<uint4 *>(vt + c * C::CHUNK_KV + (r0 + i / 8) * 128 + (i % 8) * 16) =
                    make_uint4(0, 0, 0, 0);
            fence_proxy_async_smem();  // make the zeros visible to the tensor core
            __syncwarp();
            if (lane == 0) mbar_arrive(BAR(C::B_VZ));
          }
          pos += U.J1 - U.J0;
        }
      }
      __syncwarp();
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    setmaxnreg_inc<kSoftmaxRegs>();
    const int t = warp >> 2;                            // query tile of this warpgroup
    const int quarter = warp & 3;
    const int r = quarter * 32 + lane;                  // row in the tile == TMEM lane
    const uint32_t lane_off = static_cast<uint32_t>(quarter * 32) << 16;
    const float sl2 = p.scale_log2;
    const uint32_t scol = tmem + lane_off + C::s_col(t);
    const uint32_t ocol = tmem + lane_off + C::o_col(t);
    using T = typename std::conditional<BF16, __nv_bfloat16, __half>::type;
    bool ok = true;
    uint32_t sf = 0, od = 0;  // parities of this tile's S-ready and O-done barriers
    for (int k = 0; ok && k * u_step < n_units; ++k) {
      const int u = unit_index(k, u_first, u_step);
      if (u >= n_units) continue;
      int q_tile0, Nkv, jlo, jhi;
      const int2 *krow = nullptr;  // custom mask: this row's key range [lo, hi), or null
      float slope2;
      {
        // Only what the step loop needs stays live through it; the epilogue
        // derives the unit again (cheap integer work, fewer registers held).
        const Unit U = make_unit<CAUSAL, VARLEN>(u, p, win_l, win_r);
        q_tile0 = U.q0 + t * kBM;
        Nkv = U.Nkv;
        jlo = t == 0 ? U.lo0 : U.lo1;
        jhi = t == 0 ? U.hi0 : U.hi1;
        // ALiBi: score += -slope_h |i - j|, in base-2 units.
        slope2 = (MASKED && p.alibi_slopes != nullptr && U.kind == kRun)
                     ? p.alibi_slopes[U.h] * 1.4426950408889634f : 0.f;
        if (MASKED && p.kv_ranges != nullptr && U.kind == kRun) {
          // A row past N_q (computed, never stored) reads row 0's range.
          const int row = q_tile0 + r < U.Nq ? q_tile0 + r : 0;
          const int64_t ri = VARLEN ? static_cast<int64_t>(U.q_base) + row : static_cast<int64_t>(U.b) * p.Nq + row;
          krow = reinterpret_cast<const int2 *>(p.kv_ranges) + ri;
        }
        if (U.kind != kRun) {
          const int q_row = q_tile0 + r;
          if ((U.kind & kBadIndex) && threadIdx.x == 0) atomicOr(p.err, kErrBadIndex);
          if (U.kind == kEmpty && q_row < U.Nq) {
            // No keys: O = 0 and LSE = -inf for this row.
            T *orow = reinterpret_cast<T *>(p.o) + static_cast<int64_t>(U.h) * p.o_sh +
                      static_cast<int64_t>(U.q_base + q_row) * p.o_sn;
            for (int d = 0; d < D; d += 8) *reinterpret_cast<uint4 *>(orow + d) = make_uint4(0, 0, 0, 0);
            if (p.lse != nullptr) p.lse[static_cast<int64_t>(U.h) * p.total_q + U.q_base + q_row] = -INFINITY;
          }
          continue;
        }
      }
      const int q_row = q_tile0 + r;
      const bool alibi = MASKED && p.alibi_slopes != nullptr;
      float m = -INFINITY, l = 0.f;
      for (int j = jlo; j < jhi; ++j) {
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

        const int kv0 = j * kBN;
        // Masked only where the tile crosses the end of the keys or a band edge
        // (or, with key ranges, some row's range edge).
        bool need_mask = (kv0 + kBN > Nkv) || (win_r != kUnlimited && kv0 + kBN - 1 > q_tile0 + win_r) ||
                         (win_l != kUnlimited && kv0 < q_tile0 + kBM - 1 - win_l);
        int2 kr = make_int2(0, kUnlimited);
        if (MASKED && krow != nullptr) {
          kr = __ldg(krow);
          need_mask = need_mask || __any_sync(0xffffffffu, kr.x > kv0 || kr.y < kv0 + kBN);
        }
        if (need_mask) {
          // columns lo_c <= c < hi_c are kept
          int hi_c = (win_r == kUnlimited ? Nkv : min(Nkv, q_row + win_r + 1)) - kv0;
          int lo_c = win_l == kUnlimited ? 0 : q_row - win_l - kv0;
          if constexpr (MASKED) {
            hi_c = min(hi_c, kr.y - kv0);
            lo_c = max(lo_c, kr.x - kv0);
          }
#pragma unroll
          for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int c = 0; c < 32; ++c)
              if (i * 32 + c >= hi_c || i * 32 + c < lo_c) sr[i][c] = __float_as_uint(-INFINITY);
        }
        float sl_eff = sl2;     // factor from the values in sr to base-2 scores
        float row_bias = 0.f;   // base-2 term every score of the row gets after the max
        if (alibi) {
          const float dq = static_cast<float>(q_row - kv0);
          // A tile wholly left of every row's diagonal (or wholly right of it) has
          // |i - j| = side * (i - j) with one sign: the bias splits into a column
          // term, two columns per packed multiply-add, and a row term added later.
          // Tiles that straddle a diagonal take |i - j| per element.
          const int side = (kv0 + kBN - 1 <= q_tile0) ? 1 : (kv0 >= q_tile0 + kBM - 1) ? -1 : 0;
          if (side != 0) {
            const float cs = static_cast<float>(side) * slope2;
            const uint64_t cs2 = pack_f2(cs, cs), sl2x2 = pack_f2(sl2, sl2);
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int c = 0; c < 32; c += 2) {
                const uint64_t col = pack_f2(static_cast<float>(i * 32 + c), static_cast<float>(i * 32 + c + 1));
                const float2 v = unpack_f2(ffma_f2(pack_f2(__uint_as_float(sr[i][c]), __uint_as_float(sr[i][c + 1])),
                                                   sl2x2, fmul_f2(col, cs2)));
                sr[i][c] = __float_as_uint(v.x);
                sr[i][c + 1] = __float_as_uint(v.y);
              }
            row_bias = -cs * dq;
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
              for (int c = 0; c < 32; ++c)
                sr[i][c] = __float_as_uint(
                    fmaf(__uint_as_float(sr[i][c]), sl2, -slope2 * fabsf(dq - static_cast<float>(i * 32 + c))));
          }
          sl_eff = 1.f;
        }
        // Row max: four independent chains of 3-input maxima.
        float mq[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 32; c += 8)
#pragma unroll
            for (int w = 0; w < 4; ++w)
              mq[w] = fmax3(mq[w], __uint_as_float(sr[i][c + 2 * w]), __uint_as_float(sr[i][c + 2 * w + 1]));
        const float mx = fmax3(mq[0], mq[1], fmaxf(mq[2], mq[3]));
        // Raise the running max only when the block max exceeds it by more than
        // the threshold; otherwise keep it (alpha = 1, no rescale of O).
        const float mb = mx * sl_eff + row_bias;
        const bool raise = (m == -INFINITY) || (mb > m + kRescaleThreshold);
        const float m_new = raise ? fmaxf(m, mb) : m;
        const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
        const float alpha = raise ? fast_exp2(m - m_use) : 1.f;
        // P = 2^(s * scale * log2 e - m), two columns per packed FMA; row sum in
        // four packed partial sums.
        const uint64_t sl2x2 = pack_f2(sl_eff, sl_eff), negm2 = pack_f2(row_bias - m_use, row_bias - m_use);
        uint64_t rs2[4] = {0, 0, 0, 0};
        uint32_t pk[2][32];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
          for (int c = 0; c < 32; c += 2) {
            const uint64_t e2 =
                ffma_f2(pack_f2(__uint_as_float(sr[i][c]), __uint_as_float(sr[i][c + 1])), sl2x2, negm2);
            const float2 e = unpack_f2(e2);
            const float p0 = fast_exp2(e.x), p1 = fast_exp2(e.y);
            rs2[(c >> 1) & 3] = fadd_f2(rs2[(c >> 1) & 3], pack_f2(p0, p1));
            pk[i >> 1][(i & 1) * 16 + c / 2] = pack2<BF16>(p0, p1);
          }
        const float2 r01 = unpack_f2(fadd_f2(rs2[0], rs2[1])), r23 = unpack_f2(fadd_f2(rs2[2], rs2[3]));
        const float rs = (r01.x + r01.y) + (r23.x + r23.y);
        l = l * alpha + rs;
        m = m_new;
        // P_i(j) over the first 64 columns of S_i (S_i(j) is already in registers).
        tmem_st_32x32b_x32(scol, pk[0]);
        tmem_st_32x32b_x32(scol + 32, pk[1]);
        // P_i(j-1) V_{j-1} completed before S_i(j) was signalled: O_i is stable.
        if (j > jlo && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
          for (int i = 0; i < D / 32; ++i) {
            uint32_t ov[32];
            tmem_ld_32x32b_x32(ocol + i * 32, ov);
            tmem_wait_ld();
            reg_fence(ov);
#pragma unroll
            for (int c = 0; c < 32; ++c) ov[c] = __float_as_uint(__uint_as_float(ov[c]) * alpha);
            tmem_st_32x32b_x32(ocol + i * 32, ov);
          }
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(BAR(C::B_PF + t));
      }
      // O-done comes only for a tile with keys (MASKED: one phase per such
      // unit); the MMA thread cannot signal the next one before these warps'
      // next P-ready arrival, so the barrier stays within one phase of this wait.
      if (!MASKED || jlo < jhi) {
        if (ok) ok = __all_sync(0xffffffffu, mbar_wait(BAR(C::B_OD + t), od, abort_flag, p.err));
        od ^= 1;
      }
      if (!ok) break;
      // -------------------------------------------------------- epilogue: O / l, LSE
      tc_fence_after();
      const Unit U = make_unit<CAUSAL, VARLEN>(u, p, win_l, win_r);
      // A row whose band holds no key (possible with windows) gets O = 0, LSE = -inf.
      const bool any_key = l > 0.f;
      const float inv_l = any_key ? 1.f / l : 0.f;
      const bool row_ok = q_row < U.Nq;
      T *orow = reinterpret_cast<T *>(p.o) + static_cast<int64_t>(U.bc) * p.o_sb +
                static_cast<int64_t>(U.h) * p.o_sh + static_cast<int64_t>(U.q_base + q_row) * p.o_sn;
#pragma unroll
      for (int i = 0; i < D / 32; ++i) {
        uint32_t ov[32];
        tmem_ld_32x32b_x32(ocol + i * 32, ov);
        tmem_wait_ld();
        reg_fence(ov);
        uint32_t packed[16];
#pragma unroll
        for (int c = 0; c < 32; c += 2)
          packed[c / 2] = pack2<BF16>(any_key ? __uint_as_float(ov[c]) * inv_l : 0.f,
                                      any_key ? __uint_as_float(ov[c + 1]) * inv_l : 0.f);
        if (row_ok) {
          uint4 *dst = reinterpret_cast<uint4 *>(orow + i * 32);
#pragma unroll
          for (int v = 0; v < 4; ++v)
            dst[v] = make_uint4(packed[4 * v], packed[4 * v + 1], packed[4 * v + 2], packed[4 * v + 3]);
        }
      }
      if (p.lse != nullptr && row_ok)
        p.lse[VARLEN ? static_cast<int64_t>(U.h) * p.total_q + U.q_base + q_row
                     : (static_cast<int64_t>(U.b) * p.Hq + U.h) * p.Nq + q_row] =
            any_key ? (m + __log2f(l)) * kLn2 : -INFINITY;
      // The O columns are read: the next unit's first P V may overwrite them once
      // this warp's next P-ready arrival (after tc_fence_before) says so.
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 9) {
    tc_fence_after();
    tmem_dealloc(tmem, C::TMEM_COLS);
  }
}

template <int D, bool CAUSAL, bool BF16, bool VARLEN, bool MASKED, bool ROPE>
cudaError_t launch_one(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p,
                       int B, cudaStream_t stream) {
  auto kern = prefill_fwd_kernel<D, CAUSAL, BF16, VARLEN, MASKED, ROPE>;
  constexpr uint32_t smem = Cfg<D, CAUSAL, ROPE>::SMEM_BYTES;
  // setmaxnreg redistributes the registers the CTA was launched with; a split
  // larger than that pool would never be granted, so refuse to launch then.
  cudaFuncAttributes attr{};
  cudaError_t e = cudaFuncGetAttributes(&attr, kern);
  if (e != cudaSuccess) return e;
  constexpr int kThreads = kThreadsFor<ROPE>;
  if (attr.numRegs * kThreads < 256 * kSoftmaxRegs + (kThreads - 256) * kOtherRegsFor<ROPE>)
    return cudaErrorInvalidConfiguration;
  e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  dim3 grid(p.n_ctas);  // persistent: at most one CTA per SM (n_ctas <= number of SMs)
  kern<<<grid, kThreads, smem, stream>>>(tq, tk, tv, p);
  return cudaGetLastError();
}

// Dispatch over D, causal, dtype and varlen for one value of MASKED and ROPE.
template <bool MASKED, bool ROPE>
cudaError_t launch_prefill_variant(int D, bool causal, bool bf16, bool varlen, const CUtensorMap &tq,
                                   const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p, int B,
                                   cudaStream_t stream) {
#define ATTN_PREFILL_CASE(DD, CC, BB)                                                           \
  if (D == DD && causal == CC && bf16 == BB)                                                    \
    return varlen ? launch_one<DD, CC, BB, true, MASKED, ROPE>(tq, tk, tv, p, B, stream)        \
                  : launch_one<DD, CC, BB, false, MASKED, ROPE>(tq, tk, tv, p, B, stream);
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

}  // namespace
}  // namespace attn
