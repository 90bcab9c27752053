// attn_api.cu -- the extern "C" boundary of libattn_gb300.so.
//
// Host-side work only: argument validation (before anything is launched),
// TMA tensor-map encoding, split-count selection for decode, the device error
// word, and dispatch to the kernels (prefill_kernel.cuh through prefill.cu and
// prefill_masked.cu, decode.cu, bwd.cu).
#include <algorithm>
#include <climits>
#include <cmath>
#include <cstring>
#include <mutex>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kMaxDevices = 64;

__device__ unsigned g_device_error = 0;
// Where attn_get_device_error's one-thread kernel leaves the word it took.
__device__ unsigned g_device_error_taken = 0;

__global__ void take_error_kernel(unsigned *err, unsigned *out) { *out = atomicExch(err, 0u); }

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int sm_count = 0;
  int pair_clusters = 0;  // CTA-pair prefill clusters resident at once (0: pair kernel not used)
  unsigned *err = nullptr;
  unsigned *taken = nullptr;
  // Library-owned stream on which the backward's dK/dV kernel runs beside its
  // dQ kernel (event-ordered against the caller's stream).  Created with the
  // rest of the per-device state, so that a backward captured into a CUDA graph
  // after any earlier call on the device creates nothing during the capture.
  cudaStream_t side = nullptr;
};

std::mutex g_mutex;
DeviceState g_state[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Per-device setup with the device current: SM count, architecture check and
// the address of the device error word.
attn_status_t device_state(const DeviceState **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceState &s = g_state[dev];
  if (!s.ready) {
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    s.supported = (major == 10 && minor == 3);
    s.sm_count = sms;
    if (s.supported) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return ATTN_ERR_CUDA;
      s.err = static_cast<unsigned *>(p);
      if (cudaGetSymbolAddress(&p, g_device_error_taken) != cudaSuccess) return ATTN_ERR_CUDA;
      s.taken = static_cast<unsigned *>(p);
      if (g_encode == nullptr) {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess || fn == nullptr)
          return ATTN_ERR_CUDA;
        g_encode = reinterpret_cast<EncodeTiledFn>(fn);
      }
      s.pair_clusters = prefill_pair_max_clusters();
      if (cudaStreamCreateWithFlags(&s.side, cudaStreamNonBlocking) != cudaSuccess) return ATTN_ERR_CUDA;
    }
    s.ready = true;
  }
  if (!s.supported) return ATTN_ERR_UNSUPPORTED;
  *out = &s;
  return ATTN_OK;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// (b, h, n, d) element strides of a tensor with sizes sz: d stride 1, every
// stride of an extent > 1 positive and a multiple of 8 elements (16 bytes).
attn_status_t check_strides(const int64_t s[4], const int64_t sz[4]) {
  if (s == nullptr) return ATTN_ERR_INVALID_ARG;
  if (sz[3] > 1 && s[3] != 1) return ATTN_ERR_ALIGNMENT;
  for (int i = 0; i < 3; ++i) {
    if (sz[i] <= 1) continue;
    if (s[i] <= 0) return ATTN_ERR_INVALID_ARG;
    if (s[i] % 8 != 0) return ATTN_ERR_ALIGNMENT;
  }
  return ATTN_OK;
}

// Encodes a 4-D tensor map over (d, n, h, b) with a box of 64 x box_n x 1 x 1
// and 128-byte swizzling.  The three outer dimensions are ordered by stride
// (smallest first) as the encoder expects; `slots` records where n, h and b
// went.  Extent-1 dimensions get a harmless stride.
attn_status_t make_map(CUtensorMap *map, const void *base, bool bf16, const int64_t sz[4], const int64_t st[4],
                       int box_n, uint32_t *slots) {
  struct Dim {
    int which;  // 0 = b, 1 = h, 2 = n
    uint64_t size, stride_bytes;
  } dims[3];
  uint64_t span = static_cast<uint64_t>(sz[3]) * 2;
  for (int i = 0; i < 3; ++i) span = std::max<uint64_t>(span, static_cast<uint64_t>(sz[i]) * st[i] * 2);
  span = (span + 15) & ~uint64_t(15);
  const int order[3] = {2, 1, 0};  // n, h, b (indices into the (b, h, n, d) arrays)
  for (int k = 0; k < 3; ++k) {
    const int i = order[k];
    dims[k].which = i;
    dims[k].size = static_cast<uint64_t>(sz[i]);
    dims[k].stride_bytes = sz[i] > 1 ? static_cast<uint64_t>(st[i]) * 2 : span;
  }
  std::stable_sort(dims, dims + 3, [](const Dim &a, const Dim &b) { return a.stride_bytes < b.stride_bytes; });
  cuuint64_t gdim[4] = {static_cast<cuuint64_t>(sz[3]), dims[0].size, dims[1].size, dims[2].size};
  cuuint64_t gstride[3] = {dims[0].stride_bytes, dims[1].stride_bytes, dims[2].stride_bytes};
  cuuint32_t box[4] = {64, 1, 1, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  uint32_t sn = 0, sh = 0, sb = 0;
  for (int k = 0; k < 3; ++k) {
    if (dims[k].which == 2) {
      sn = k + 1;
      box[k + 1] = static_cast<cuuint32_t>(box_n);
    } else if (dims[k].which == 1) {
      sh = k + 1;
    } else {
      sb = k + 1;
    }
  }
  for (int k = 0; k < 3; ++k)
    if (gstride[k] % 16 != 0 || gstride[k] >= (1ull << 40)) return ATTN_ERR_ALIGNMENT;
  *slots = sn | (sh << 2) | (sb << 4);
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                        const_cast<void *>(base), gdim, gstride, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ATTN_OK : ATTN_ERR_CUDA;
}

// Number of KV splits decode uses on long caches for these sizes on this
// device: the fewest splits that give at least one full wave of resident
// CTAs (kDecodeCtasPerSm per SM) with the last wave at least 85 % full;
// failing that, the split count (<= 64) whose last wave is fullest.
int decode_max_splits(int B, int H_q, int H_kv, int sm_count) {
  const int group = H_q / H_kv;
  const int gh = decode_heads_per_cta(group);
  const int nhc = (group + gh - 1) / gh;
  const double ctas = static_cast<double>(B) * H_kv * nhc;
  const double slots = static_cast<double>(kDecodeCtasPerSm) * sm_count;
  int best = 1;
  double best_eff = -1.0;
  for (int s = 1; s <= 64; ++s) {
    const double waves = ctas * s / slots;
    const double eff = waves / std::ceil(waves);
    if (waves >= 1.0 && eff >= 0.85) return s;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = s;
    }
  }
  return best;
}

// Split plan of one decode call: every split holds a multiple of the stage
// size in keys (except the last), at least kMinChunk keys, and none is empty.
// forced > 0 (a caller's num_splits) replaces the automatic split count as
// the upper bound and drops the minimum split length (down to one stage).
void decode_plan(int B, int H_q, int H_kv, int cache_len, int D, int sm_count, int *nsplit_out, int *chunk_out,
                 int forced = 0) {
  constexpr int kMinChunk = 256;
  (void)D;
  const int step = kDecodeStageTokens;
  int nsplit;
  if (forced > 0) {
    nsplit = std::min<int>(forced, (cache_len + step - 1) / step);
  } else {
    const int max_splits = decode_max_splits(B, H_q, H_kv, sm_count);
    nsplit = std::min<int>(max_splits, (cache_len + kMinChunk - 1) / kMinChunk);
  }
  nsplit = std::max(nsplit, 1);
  int chunk = (cache_len + nsplit - 1) / nsplit;
  chunk = (chunk + step - 1) / step * step;
  *nsplit_out = (cache_len + chunk - 1) / chunk;
  *chunk_out = chunk;
}

size_t decode_ws_bytes(int B, int H_q, int D, int splits) {
  if (splits <= 1) return 0;
  return static_cast<size_t>(B) * H_q * splits * (D + 1) * sizeof(float);
}

bool valid_dtype(attn_dtype_t dt) { return dt == ATTN_F16 || dt == ATTN_BF16; }

// Mask, bias, position and split options (NULL: none of them).
struct Opts {
  int wl = -1, wr = -1;          // window bounds (-1: unbounded)
  const float *slopes = nullptr; // ALiBi slopes (device, H_q)
  float rope_theta = 0.f;        // 0: no rotary embedding
  int rope_interleaved = 0;      // 0: pairs (c, c + D/2); 1: pairs (2c, 2c + 1)
  int num_splits = 0;            // decode: 0 automatic, else at most this many KV splits
  int rope_rotated_keys = 0;     // prefill: the keys come already rotated
  const int32_t *kv_ranges = nullptr;  // prefill: per-row key ranges
  int prefill_kernel = 0;        // dense prefill: 0 automatic, 1 one-CTA, 2 CTA pair
};
constexpr int kMaxDecodeSplits = 64;

// kernel_choice: the call can run either prefill kernel (else prefill_kernel
// must be 0).
attn_status_t read_opts(const attn_options_t *opts, Opts *o, bool kernel_choice = false) {
  *o = Opts{};
  if (opts == nullptr) return ATTN_OK;
  if (opts->prefill_kernel < 0 || opts->prefill_kernel > 2 || (!kernel_choice && opts->prefill_kernel != 0))
    return ATTN_ERR_INVALID_ARG;
  if (opts->window_left < -1 || opts->window_right < -1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(opts->rope_theta) || opts->rope_theta < 0.f) return ATTN_ERR_INVALID_ARG;
  if (opts->rope_interleaved != 0 && opts->rope_interleaved != 1) return ATTN_ERR_INVALID_ARG;
  if (opts->num_splits < 0 || opts->num_splits > kMaxDecodeSplits) return ATTN_ERR_INVALID_ARG;
  if (opts->rope_rotated_keys != 0 && opts->rope_rotated_keys != 1) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(opts->alibi_slopes) & 3) != 0) return ATTN_ERR_ALIGNMENT;
  if ((reinterpret_cast<uintptr_t>(opts->kv_ranges) & 7) != 0) return ATTN_ERR_ALIGNMENT;
  o->wl = opts->window_left;
  o->wr = opts->window_right;
  o->slopes = opts->alibi_slopes;
  o->rope_theta = opts->rope_theta;
  o->rope_interleaved = opts->rope_interleaved;
  o->num_splits = opts->num_splits;
  o->rope_rotated_keys = opts->rope_rotated_keys;
  o->kv_ranges = opts->kv_ranges;
  o->prefill_kernel = opts->prefill_kernel;
  return ATTN_OK;
}

// Turn steps of rotary embeddings as 64-bit fractions of a full turn:
// f_c = frac(theta^(-2c/D) / (2 pi)) * 2^64.  Computed in double precision,
// whose error (about 1e-16 of a turn per unit position) stays far below fp32
// resolution for any position an int can hold.
void fill_rope_steps(float theta, int D, uint64_t *f) {
  constexpr double kTwoPi = 6.283185307179586476925286766559;
  for (int c = 0; c < D / 2; ++c) {
    const double inv = std::pow(static_cast<double>(theta), -2.0 * c / D);
    double t = inv / kTwoPi;
    t -= std::floor(t);  // in [0, 1)
    const double scaled = std::ldexp(t, 64);
    f[c] = scaled >= 18446744073709551615.0 ? ~uint64_t(0) : static_cast<uint64_t>(scaled);
  }
  for (int c = D / 2; c < 64; ++c) f[c] = 0;
}

// Failure-detection self-test: one thread waits on an mbarrier that nothing
// ever arrives on.  The bounded wait gives up after its wall-clock limit,
// records kErrWaitTimeout in the device error word and returns.
__global__ void selftest_wait_kernel(unsigned *err) {
  __shared__ __align__(8) uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, err);
}

// Persistent prefill schedule: units = query-row blocks x heads x batches,
// walked by at most `slots` workers (CTAs, or CTA pairs) resident at once.
attn_status_t prefill_schedule(PrefillParams *p, int B, int H_q, int slots) {
  const int64_t units = static_cast<int64_t>(H_q) * B * p->n_qtiles;
  // The kernel walks units in rounds of up to `slots`; every index it forms
  // (round * workers + worker) stays below units + slots, which must fit an int.
  if (units + slots > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
  p->B = B;
  p->n_units = static_cast<int>(units);
  p->n_ctas = static_cast<int>(units < slots ? units : slots);
  return ATTN_OK;
}

// Groups per chunk of the backward's tile order: as many (batch, kv head)
// groups as keep the operands the CTAs in flight share within ~48 MB of L2 (Q
// and dO of the group's heads for dK/dV, K and V for dQ).  Under the causal
// mask a dK/dV tile's cost falls from the whole group's queries (key tile 0)
// to one tile, and the longest tiles must start early: at most two chunks
// there, so that the second chunk's longest tiles start about half way.
// (Measured, B = 2, H_q = 32, H_kv = 8, N = 8192: chunks of 5 groups cut the
// dK/dV kernel's DRAM reads from 1088 to 393 MB but stretched it from 1.65 to
// 1.91 ms; dQ in chunks of 11 read 349 instead of 606 MB in 1.39 instead of
// 1.42 ms.)
void bwd_chunks(BwdParams *p, int D, bool causal) {
  const int n_groups = p->Hkv * p->B;
  const double budget = 48e6;
  auto fit = [&](double group_bytes) {
    return std::max(1, std::min(static_cast<int>(budget / group_bytes), n_groups));
  };
  p->chunk_dq = fit(2.0 * p->Nkv * D * 2);
  p->chunk_dkv = fit(2.0 * p->group * p->Nq * D * 2);
  if (causal) p->chunk_dkv = std::max(p->chunk_dkv, (n_groups + 1) / 2);
}

// Whether a prefill needs the masked kernel build: a left window, a right
// window that the causal mask does not already imply, or ALiBi slopes.
bool prefill_masked(const PrefillParams &p, bool causal) {
  return p.window_left >= 0 || (!causal && p.window_right >= 0) || p.alibi_slopes != nullptr ||
         p.kv_ranges != nullptr;
}

// Keys decode streams for a cache of `len` rows under a left window: the
// window plus the rounding of its start down to a whole stage.
int decode_span(int len, int wl) {
  if (wl < 0) return len;
  const int64_t span = static_cast<int64_t>(wl) + kDecodeStageTokens;
  return static_cast<int>(span < len ? span : len);
}

// Argument checks of attn_fwd_decode (everything but the options and the
// workspace), in the order that call applies them: pointers and sizes, then
// the type and head dimension, then alignment and strides.
attn_status_t decode_check_args(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                                attn_dtype_t dtype, int B, int H_q, int H_kv, int cache_len, int D,
                                const int64_t q_str[4], const int64_t kc_str[4], const int64_t vc_str[4],
                                const int64_t o_str[4], float scale) {
  if (!q || !k_cache || !v_cache || !o || !q_str || !kc_str || !vc_str || !o_str) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H_q < 1 || H_kv < 1 || cache_len < 1 || D < 1 || H_q % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f) || B > 65535) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3)))
    return ATTN_ERR_ALIGNMENT;
  const int64_t qsz[4] = {B, H_q, 1, D}, csz[4] = {B, H_kv, cache_len, D};
  attn_status_t st;
  if ((st = check_strides(q_str, qsz)) || (st = check_strides(kc_str, csz)) || (st = check_strides(vc_str, csz)) ||
      (st = check_strides(o_str, qsz)))
    return st;
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

using namespace attn;

extern "C" {

attn_status_t attn_fwd_prefill(const void *q, const void *k, const void *v, void *o, float *lse, attn_dtype_t dtype,
                               int B, int H_q, int H_kv, int N_q, int N_kv, int D, const int64_t q_str[4],
                               const int64_t k_str[4], const int64_t v_str[4], const int64_t o_str[4], int causal,
                               float scale, void *stream) {
  return attn_fwd_prefill_ex(q, k, v, o, lse, dtype, B, H_q, H_kv, N_q, N_kv, D, q_str, k_str, v_str, o_str, causal,
                             scale, nullptr, stream);
}

attn_status_t attn_fwd_prefill_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                                  attn_dtype_t dtype, int B, int H_q, int H_kv, int N_q, int N_kv, int D,
                                  const int64_t q_str[4], const int64_t k_str[4], const int64_t v_str[4],
                                  const int64_t o_str[4], int causal, float scale, const attn_options_t *opts,
                                  void *stream) {
  if (!q || !k || !v || !o || !q_str || !k_str || !v_str || !o_str) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H_q < 1 || H_kv < 1 || N_q < 1 || N_kv < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (H_q % H_kv != 0 || (causal != 0 && causal != 1)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (B > 65535 || H_q > 65535) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || (lse && (reinterpret_cast<uintptr_t>(lse) & 3)))
    return ATTN_ERR_ALIGNMENT;
  const int64_t qsz[4] = {B, H_q, N_q, D}, kvsz[4] = {B, H_kv, N_kv, D};
  attn_status_t st;
  if ((st = check_strides(q_str, qsz)) || (st = check_strides(k_str, kvsz)) || (st = check_strides(v_str, kvsz)) ||
      (st = check_strides(o_str, qsz)))
    return st;

  PrefillParams p{};
  Opts op;
  if ((st = read_opts(opts, &op, true)) != ATTN_OK) return st;
  p.window_left = op.wl;
  p.window_right = op.wr;
  p.alibi_slopes = op.slopes;
  p.kv_ranges = op.kv_ranges;
  const bool rope = op.rope_theta > 0.f;
  if (rope) {
    p.rope_inter = op.rope_interleaved;
    p.rope_k = op.rope_rotated_keys ? 0 : 1;
    fill_rope_steps(op.rope_theta, D, p.rope_f);
  }
  const DeviceState *dev = nullptr;
  if ((st = device_state(&dev)) != ATTN_OK) return st;
  const bool bf16 = dtype == ATTN_BF16;
  const bool masked = prefill_masked(p, causal != 0);
  // The CTA-pair kernel (on request only): head dimension 128 without
  // windows, ALiBi, key ranges or rotary embeddings; each CTA loads half of
  // every K tile (64-row boxes).
  const bool pair = op.prefill_kernel == 2;
  if (pair && (D != 128 || masked || rope || dev->pair_clusters <= 0)) return ATTN_ERR_UNSUPPORTED;
  CUtensorMap tq, tk, tv;
  if ((st = make_map(&tq, q, bf16, qsz, q_str, kPrefillBM, &p.slots_q)) ||
      (st = make_map(&tk, k, bf16, kvsz, k_str, pair ? kPrefillBN / 2 : kPrefillBN, &p.slots_k)) ||
      (st = make_map(&tv, v, bf16, kvsz, v_str, kPrefillBN, &p.slots_v)))
    return st;
  p.o = o;
  p.lse = lse;
  p.err = dev->err;
  p.o_sb = o_str[0];
  p.o_sh = o_str[1];
  p.o_sn = o_str[2];
  p.Nq = N_q;
  p.Nkv = N_kv;
  p.Hq = H_q;
  p.group = H_q / H_kv;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  cudaError_t e;
  if (pair) {
    p.n_qtiles = (N_q + kPairUnitRows - 1) / kPairUnitRows;
    if ((st = prefill_schedule(&p, B, H_q, dev->pair_clusters)) != ATTN_OK) return st;
    p.n_ctas *= 2;  // clusters of two CTAs
    e = launch_prefill_pair(causal != 0, bf16, tq, tk, tv, p, static_cast<cudaStream_t>(stream));
  } else {
    p.n_qtiles = (N_q + 2 * kPrefillBM - 1) / (2 * kPrefillBM);
    if ((st = prefill_schedule(&p, B, H_q, dev->sm_count)) != ATTN_OK) return st;
    e = launch_prefill(D, causal != 0, bf16, false, masked, rope, tq, tk, tv, p, B, static_cast<cudaStream_t>(stream));
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_fwd_prefill_varlen(const void *q, const void *k, const void *v, void *o, float *lse,
                                      attn_dtype_t dtype, int B, int H_q, int H_kv, int D, const int32_t *cu_seqlens_q,
                                      const int32_t *cu_seqlens_k, int max_seqlen_q, int max_seqlen_k, int total_q,
                                      int total_k, const int64_t q_str[3], const int64_t k_str[3],
                                      const int64_t v_str[3], const int64_t o_str[3], int causal, float scale,
                                      void *stream) {
  return attn_fwd_prefill_varlen_ex(q, k, v, o, lse, dtype, B, H_q, H_kv, D, cu_seqlens_q, cu_seqlens_k, max_seqlen_q,
                                    max_seqlen_k, total_q, total_k, q_str, k_str, v_str, o_str, causal, scale, nullptr,
                                    stream);
}

attn_status_t attn_fwd_prefill_varlen_ex(const void *q, const void *k, const void *v, void *o, float *lse,
                                         attn_dtype_t dtype, int B, int H_q, int H_kv, int D,
                                         const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int max_seqlen_q,
                                         int max_seqlen_k, int total_q, int total_k, const int64_t q_str[3],
                                         const int64_t k_str[3], const int64_t v_str[3], const int64_t o_str[3],
                                         int causal, float scale, const attn_options_t *opts, void *stream) {
  if (!q || !k || !v || !o || !cu_seqlens_q || !cu_seqlens_k || !q_str || !k_str || !v_str || !o_str)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H_q < 1 || H_kv < 1 || D < 1 || max_seqlen_q < 1 || max_seqlen_k < 1 || total_q < 1 || total_k < 1)
    return ATTN_ERR_INVALID_ARG;
  if (max_seqlen_q > total_q || max_seqlen_k > total_k) return ATTN_ERR_INVALID_ARG;
  if (H_q % H_kv != 0 || (causal != 0 && causal != 1)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f) || B > 65535 || H_q > 65535) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3)) || (reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3) ||
      (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3))
    return ATTN_ERR_ALIGNMENT;
  // Packed tensors seen as (1, H, total, D) with (b, h, n, d) strides.
  const int64_t qsz[4] = {1, H_q, total_q, D}, kvsz[4] = {1, H_kv, total_k, D};
  const int64_t q4[4] = {0, q_str[1], q_str[0], q_str[2]}, k4[4] = {0, k_str[1], k_str[0], k_str[2]};
  const int64_t v4[4] = {0, v_str[1], v_str[0], v_str[2]}, o4[4] = {0, o_str[1], o_str[0], o_str[2]};
  attn_status_t st;
  if ((st = check_strides(q4, qsz)) || (st = check_strides(k4, kvsz)) || (st = check_strides(v4, kvsz)) ||
      (st = check_strides(o4, qsz)))
    return st;
  PrefillParams p{};
  Opts op;
  if ((st = read_opts(opts, &op)) != ATTN_OK) return st;
  p.window_left = op.wl;
  p.window_right = op.wr;
  p.alibi_slopes = op.slopes;
  p.kv_ranges = op.kv_ranges;
  const bool rope = op.rope_theta > 0.f;
  if (rope) {
    p.rope_inter = op.rope_interleaved;
    p.rope_k = op.rope_rotated_keys ? 0 : 1;
    fill_rope_steps(op.rope_theta, D, p.rope_f);
  }
  const DeviceState *dev = nullptr;
  if ((st = device_state(&dev)) != ATTN_OK) return st;
  const bool bf16 = dtype == ATTN_BF16;
  CUtensorMap tq, tk, tv;
  if ((st = make_map(&tq, q, bf16, qsz, q4, kPrefillBM, &p.slots_q)) ||
      (st = make_map(&tk, k, bf16, kvsz, k4, kPrefillBN, &p.slots_k)) ||
      (st = make_map(&tv, v, bf16, kvsz, v4, kPrefillBN, &p.slots_v)))
    return st;
  p.o = o;
  p.lse = lse;
  p.err = dev->err;
  p.o_sb = 0;
  p.o_sh = o4[1];
  p.o_sn = o4[2];
  p.Nq = max_seqlen_q;
  p.Nkv = max_seqlen_k;
  p.Hq = H_q;
  p.group = H_q / H_kv;
  p.n_qtiles = (max_seqlen_q + 2 * kPrefillBM - 1) / (2 * kPrefillBM);
  if ((st = prefill_schedule(&p, B, H_q, dev->sm_count)) != ATTN_OK) return st;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.cu_q = cu_seqlens_q;
  p.cu_k = cu_seqlens_k;
  p.total_q = total_q;
  p.total_k = total_k;
  cudaError_t e = launch_prefill(D, causal != 0, bf16, true, prefill_masked(p, causal != 0), rope, tq, tk, tv, p, B,
                                 static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_bwd_workspace_size(int B, int H_q, int N_q) {
  if (B < 1 || H_q < 1 || N_q < 1) return 0;
  return (static_cast<size_t>(B) * H_q * N_q * sizeof(float) + 15) & ~size_t(15);
}

namespace {
// Backward workspace: D_i (fp32 per query row), then, with rotary embeddings,
// the rotated queries Q' (B, H_q, N_q, D) and -- unless the keys come rotated
// -- the rotated keys K' (B, H_kv, N_kv, D), both contiguous 16-bit rows.
struct BwdWorkspace {
  size_t q_off, k_off, total;
};
BwdWorkspace bwd_workspace(int B, int H_q, int H_kv, int N_q, int N_kv, int D, bool rope, bool rotate_k) {
  BwdWorkspace w;
  w.q_off = attn_bwd_workspace_size(B, H_q, N_q);
  w.k_off = w.q_off + (rope ? static_cast<size_t>(B) * H_q * N_q * D * 2 : 0);
  w.total = w.k_off + (rope && rotate_k ? static_cast<size_t>(B) * H_kv * N_kv * D * 2 : 0);
  return w;
}
}  // namespace

size_t attn_bwd_ex_workspace_size(int B, int H_q, int H_kv, int N_q, int N_kv, int D, const attn_options_t *opts) {
  if (B < 1 || H_q < 1 || H_kv < 1 || N_q < 1 || N_kv < 1 || H_q % H_kv != 0 || (D != 64 && D != 128)) return 0;
  Opts op;
  if (read_opts(opts, &op) != ATTN_OK) return 0;
  const bool rope = op.rope_theta > 0.f;
  return bwd_workspace(B, H_q, H_kv, N_q, N_kv, D, rope, rope && !op.rope_rotated_keys).total;
}

attn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o, const void *dout,
                       const float *lse, void *dq, void *dk, void *dv, attn_dtype_t dtype, int B, int H_q, int H_kv,
                       int N_q, int N_kv, int D, const int64_t q_str[4], const int64_t k_str[4],
                       const int64_t v_str[4], const int64_t o_str[4], const int64_t do_str[4],
                       const int64_t dq_str[4], const int64_t dk_str[4], const int64_t dv_str[4], int causal,
                       float scale, void *workspace, size_t workspace_bytes, void *stream) {
  return attn_bwd_ex(q, k, v, o, dout, lse, dq, dk, dv, dtype, B, H_q, H_kv, N_q, N_kv, D, q_str, k_str, v_str, o_str,
                     do_str, dq_str, dk_str, dv_str, causal, scale, nullptr, workspace, workspace_bytes, stream);
}

attn_status_t attn_bwd_ex(const void *q, const void *k, const void *v, const void *o, const void *dout,
                          const float *lse, void *dq, void *dk, void *dv, attn_dtype_t dtype, int B, int H_q,
                          int H_kv, int N_q, int N_kv, int D, const int64_t q_str[4], const int64_t k_str[4],
                          const int64_t v_str[4], const int64_t o_str[4], const int64_t do_str[4],
                          const int64_t dq_str[4], const int64_t dk_str[4], const int64_t dv_str[4], int causal,
                          float scale, const attn_options_t *opts, void *workspace, size_t workspace_bytes,
                          void *stream) {
  if (!q || !k || !v || !o || !dout || !lse || !dq || !dk || !dv || !q_str || !k_str || !v_str || !o_str ||
      !do_str || !dq_str || !dk_str || !dv_str)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H_q < 1 || H_kv < 1 || N_q < 1 || N_kv < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (H_q % H_kv != 0 || (causal != 0 && causal != 1)) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f) || B > 65535 || H_q > 65535) return ATTN_ERR_INVALID_ARG;
  // The tiled kernels' 1-D grids: H_q * B query tiles and H_kv * B key tiles.
  if (static_cast<int64_t>(H_q) * B * ((N_q + 127) / 128) > 0x7fffffff ||
      static_cast<int64_t>(H_kv) * B * ((N_kv + 127) / 128) > 0x7fffffff)
    return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(dout) || !aligned16(dq) ||
      !aligned16(dk) || !aligned16(dv) || (reinterpret_cast<uintptr_t>(lse) & 3))
    return ATTN_ERR_ALIGNMENT;
  const int64_t qsz[4] = {B, H_q, N_q, D}, kvsz[4] = {B, H_kv, N_kv, D};
  attn_status_t st;
  if ((st = check_strides(q_str, qsz)) || (st = check_strides(k_str, kvsz)) || (st = check_strides(v_str, kvsz)) ||
      (st = check_strides(o_str, qsz)) || (st = check_strides(do_str, qsz)) || (st = check_strides(dq_str, qsz)) ||
      (st = check_strides(dk_str, kvsz)) || (st = check_strides(dv_str, kvsz)))
    return st;
  Opts op;
  if ((st = read_opts(opts, &op)) != ATTN_OK) return st;
  const bool rope = op.rope_theta > 0.f, rotate_k = rope && !op.rope_rotated_keys;
  const BwdWorkspace ws = bwd_workspace(B, H_q, H_kv, N_q, N_kv, D, rope, rotate_k);
  if (workspace == nullptr || workspace_bytes < ws.total) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 15) != 0) return ATTN_ERR_ALIGNMENT;
  const DeviceState *dev = nullptr;
  if ((st = device_state(&dev)) != ATTN_OK) return st;
  const bool bf16 = dtype == ATTN_BF16;
  BwdMaps m;
  BwdParams p{};
  p.window_left = op.wl;
  p.window_right = op.wr;
  p.alibi_slopes = op.slopes;
  p.kv_ranges = op.kv_ranges;
  const bool masked = op.wl >= 0 || (causal == 0 && op.wr >= 0) || op.slopes != nullptr || op.kv_ranges != nullptr;
  // Rotary embeddings: the kernels run on Q' = R Q and K' = R K, rotated into
  // the workspace first; dQ and dK are turned back by R^T in place at the end.
  const void *q_in = q, *k_in = k;
  const int64_t *q_in_str = q_str, *k_in_str = k_str;
  const int64_t qr_str[4] = {static_cast<int64_t>(H_q) * N_q * D, static_cast<int64_t>(N_q) * D, D, 1};
  const int64_t kr_str[4] = {static_cast<int64_t>(H_kv) * N_kv * D, static_cast<int64_t>(N_kv) * D, D, 1};
  RopeRowsParams rp{};
  if (rope) {
    char *base = static_cast<char *>(workspace);
    rp.B = B;
    fill_rope_steps(op.rope_theta, D, rp.rope_f);
    rp.job[0] = RopeRowsJob{q, base + ws.q_off, q_str[0], q_str[1], q_str[2], qr_str[0], qr_str[1], qr_str[2],
                            H_q, N_q};
    q_in = base + ws.q_off;
    q_in_str = qr_str;
    if (rotate_k) {
      rp.job[1] = RopeRowsJob{k, base + ws.k_off, k_str[0], k_str[1], k_str[2], kr_str[0], kr_str[1], kr_str[2],
                              H_kv, N_kv};
      k_in = base + ws.k_off;
      k_in_str = kr_str;
    }
  }
  if ((st = make_map(&m.q, q_in, bf16, qsz, q_in_str, 128, &p.slots_q)) ||
      (st = make_map(&m.dout, dout, bf16, qsz, do_str, 128, &p.slots_do)) ||
      (st = make_map(&m.k, k_in, bf16, kvsz, k_in_str, 128, &p.slots_k)) ||
      (st = make_map(&m.v, v, bf16, kvsz, v_str, 128, &p.slots_v)))
    return st;
  p.o = o;
  p.dout = dout;
  p.lse = lse;
  p.dvec = static_cast<float *>(workspace);
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  p.err = dev->err;
  p.o_sb = o_str[0];
  p.o_sh = o_str[1];
  p.o_sn = o_str[2];
  p.do_sb = do_str[0];
  p.do_sh = do_str[1];
  p.do_sn = do_str[2];
  p.dq_sb = dq_str[0];
  p.dq_sh = dq_str[1];
  p.dq_sn = dq_str[2];
  p.dk_sb = dk_str[0];
  p.dk_sh = dk_str[1];
  p.dk_sn = dk_str[2];
  p.dv_sb = dv_str[0];
  p.dv_sh = dv_str[1];
  p.dv_sn = dv_str[2];
  p.Nq = N_q;
  p.Nkv = N_kv;
  p.Hq = H_q;
  p.group = H_q / H_kv;
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.B = B;
  p.Hkv = H_kv;
  bwd_chunks(&p, D, causal != 0);
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaSuccess;
  if (rope) {
    rp.sin_sign = 1.f;
    e = launch_rope_rows(D, bf16, op.rope_interleaved != 0, rp, rotate_k ? 2 : 1, s);
    if (e != cudaSuccess) return ATTN_ERR_CUDA;
  }
  e = launch_bwd(D, causal != 0, bf16, masked, m, p, B, H_kv, s, dev->side);
  if (e != cudaSuccess) return ATTN_ERR_CUDA;
  if (rope) {
    // dQ = R^T dQ', dK = R^T dK' (dK' itself when the keys came rotated).
    rp.sin_sign = -1.f;
    rp.job[0] = RopeRowsJob{dq, dq, dq_str[0], dq_str[1], dq_str[2], dq_str[0], dq_str[1], dq_str[2], H_q, N_q};
    rp.job[1] = RopeRowsJob{dk, dk, dk_str[0], dk_str[1], dk_str[2], dk_str[0], dk_str[1], dk_str[2], H_kv, N_kv};
    e = launch_rope_rows(D, bf16, op.rope_interleaved != 0, rp, rotate_k ? 2 : 1, s);
  }
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

size_t attn_decode_workspace_size(int B, int H_q, int H_kv, int D) {
  if (B < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || (D != 64 && D != 128)) return 0;
  const DeviceState *dev = nullptr;
  if (device_state(&dev) != ATTN_OK) return 0;
  return decode_ws_bytes(B, H_q, D, decode_max_splits(B, H_q, H_kv, dev->sm_count));
}

int attn_decode_splits(int B, int H_q, int H_kv, int cache_len, int D) {
  if (B < 1 || H_q < 1 || H_kv < 1 || H_q % H_kv != 0 || cache_len < 1 || (D != 64 && D != 128)) return 0;
  const DeviceState *dev = nullptr;
  if (device_state(&dev) != ATTN_OK) return 0;
  int nsplit = 1, chunk = cache_len;
  decode_plan(B, H_q, H_kv, cache_len, D, dev->sm_count, &nsplit, &chunk);
  return nsplit;
}

attn_status_t attn_fwd_decode(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                              attn_dtype_t dtype, int B, int H_q, int H_kv, int cache_len, int D,
                              const int64_t q_str[4], const int64_t kc_str[4], const int64_t vc_str[4],
                              const int64_t o_str[4], float scale, void *workspace, size_t workspace_bytes,
                              void *stream) {
  return attn_fwd_decode_ex(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D, q_str, kc_str, vc_str,
                            o_str, scale, workspace, workspace_bytes, nullptr, stream);
}

attn_status_t attn_fwd_decode_ex(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                                 attn_dtype_t dtype, int B, int H_q, int H_kv, int cache_len, int D,
                                 const int64_t q_str[4], const int64_t kc_str[4], const int64_t vc_str[4],
                                 const int64_t o_str[4], float scale, void *workspace, size_t workspace_bytes,
                                 const attn_options_t *opts, void *stream) {
  attn_status_t st = decode_check_args(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D, q_str, kc_str,
                                       vc_str, o_str, scale);
  if (st != ATTN_OK) return st;
  const int64_t csz[4] = {B, H_kv, cache_len, D};
  Opts op;
  if ((st = read_opts(opts, &op)) != ATTN_OK) return st;
  if (op.kv_ranges != nullptr) return ATTN_ERR_UNSUPPORTED;  // key ranges are a prefill mask
  const int wl = op.wl;
  const float *slopes = op.slopes;
  const DeviceState *dev = nullptr;
  if ((st = device_state(&dev)) != ATTN_OK) return st;

  const int group = H_q / H_kv;
  const int gh = decode_heads_per_cta(group);
  const int nhc = (group + gh - 1) / gh;
  int nsplit = 1, chunk = cache_len;
  decode_plan(B, H_q, H_kv, decode_span(cache_len, wl), D, dev->sm_count, &nsplit, &chunk, op.num_splits);
  if (nsplit > 1) {
    const size_t need = decode_ws_bytes(B, H_q, D, nsplit);
    if (workspace == nullptr || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15) != 0) return ATTN_ERR_ALIGNMENT;
  }
  DecodeParams p{};
  p.q = q;
  p.kc = k_cache;
  p.vc = v_cache;
  p.o = o;
  p.lse = lse;
  p.ws_o = static_cast<float *>(workspace);
  p.ws_lse = nsplit > 1 ? static_cast<float *>(workspace) + static_cast<size_t>(B) * H_q * nsplit * D : nullptr;
  p.err = dev->err;
  p.q_sb = q_str[0];
  p.q_sh = q_str[1];
  p.kc_sb = kc_str[0];
  p.kc_sh = kc_str[1];
  p.kc_sn = kc_str[2];
  p.vc_sb = vc_str[0];
  p.vc_sh = vc_str[1];
  p.vc_sn = vc_str[2];
  p.o_sb = o_str[0];
  p.o_sh = o_str[1];
  p.Hq = H_q;
  p.group = group;
  p.nhc = nhc;
  p.cache_len = cache_len;
  p.chunk = chunk;
  p.nsplit = nsplit;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.window_left = wl;
  p.alibi_slopes = slopes;
  if (op.rope_theta > 0.f) {
    p.rope = op.rope_interleaved ? 2 : 1;
    fill_rope_steps(op.rope_theta, D, p.rope_f);
  }
  if (static_cast<int64_t>(H_kv) * nhc > 65535) return ATTN_ERR_INVALID_ARG;
  // Tensor maps over the valid rows only: rows >= cache_len read as zeros.
  CUtensorMap tk, tv;
  const bool bf16 = dtype == ATTN_BF16;
  if ((st = make_map(&tk, k_cache, bf16, csz, kc_str, kDecodeStageTokens, &p.slots_k)) ||
      (st = make_map(&tv, v_cache, bf16, csz, vc_str, kDecodeStageTokens, &p.slots_v)))
    return st;
  cudaError_t e = launch_decode(D, bf16, false, gh, tk, tv, p, B, H_kv, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t kv_cache_write(void *k_cache, void *v_cache, const void *k_new, const void *v_new, attn_dtype_t dtype,
                             int B, int H_kv, int n_new, int D, int pos, int max_len, const int64_t kc_str[4],
                             const int64_t vc_str[4], const int64_t kn_str[4], const int64_t vn_str[4],
                             void *stream) {
  return kv_cache_write_ex(k_cache, v_cache, k_new, v_new, dtype, B, H_kv, n_new, D, pos, max_len, kc_str, vc_str,
                           kn_str, vn_str, nullptr, stream);
}

attn_status_t kv_cache_write_ex(void *k_cache, void *v_cache, const void *k_new, const void *v_new,
                                attn_dtype_t dtype, int B, int H_kv, int n_new, int D, int pos, int max_len,
                                const int64_t kc_str[4], const int64_t vc_str[4], const int64_t kn_str[4],
                                const int64_t vn_str[4], const attn_options_t *opts, void *stream) {
  if (!k_cache || !v_cache || !k_new || !v_new || !kc_str || !vc_str || !kn_str || !vn_str)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H_kv < 1 || n_new < 1 || D < 1 || max_len < 1 || pos < 0) return ATTN_ERR_INVALID_ARG;
  if (static_cast<int64_t>(pos) + n_new > max_len) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(k_cache) || !aligned16(v_cache) || !aligned16(k_new) || !aligned16(v_new)) return ATTN_ERR_ALIGNMENT;
  const int64_t csz[4] = {B, H_kv, max_len, D}, nsz[4] = {B, H_kv, n_new, D};
  attn_status_t st;
  if ((st = check_strides(kc_str, csz)) || (st = check_strides(vc_str, csz)) || (st = check_strides(kn_str, nsz)) ||
      (st = check_strides(vn_str, nsz)))
    return st;
  Opts op;
  if ((st = read_opts(opts, &op)) != ATTN_OK) return st;
  const DeviceState *dev = nullptr;
  if ((st = device_state(&dev)) != ATTN_OK) return st;
  KvWriteParams p{};
  p.kc = k_cache;
  p.vc = v_cache;
  p.kn = k_new;
  p.vn = v_new;
  p.kc_sb = kc_str[0];
  p.kc_sh = kc_str[1];
  p.kc_sn = kc_str[2];
  p.vc_sb = vc_str[0];
  p.vc_sh = vc_str[1];
  p.vc_sn = vc_str[2];
  p.kn_sb = kn_str[0];
  p.kn_sh = kn_str[1];
  p.kn_sn = kn_str[2];
  p.vn_sb = vn_str[0];
  p.vn_sh = vn_str[1];
  p.vn_sn = vn_str[2];
  p.Hkv = H_kv;
  p.n_new = n_new;
  p.pos = pos;
  p.D = D;
  p.total_units = static_cast<int64_t>(B) * H_kv * n_new * (D / 8);
  p.err = dev->err;
  p.is_bf16 = dtype == ATTN_BF16;
  if (op.rope_theta > 0.f) {
    p.rope = op.rope_interleaved ? 2 : 1;
    fill_rope_steps(op.rope_theta, D, p.rope_f);
  }
  cudaError_t e = launch_kv_cache_write(p, false, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

// Page geometry shared by the paged entry points.
static attn_status_t check_pages(int num_pages, int page_size, const int32_t *block_table, int max_pages,
                                 int64_t bt_stride) {
  if (num_pages < 1 || max_pages < 1 || block_table == nullptr || bt_stride < max_pages) return ATTN_ERR_INVALID_ARG;
  if (!(page_size == 16 || page_size == 32 || (page_size >= 64 && page_size % 64 == 0))) return ATTN_ERR_UNSUPPORTED;
  if ((reinterpret_cast<uintptr_t>(block_table) & 3) != 0) return ATTN_ERR_ALIGNMENT;
  if (static_cast<int64_t>(max_pages) * page_size > INT_MAX) return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

attn_status_t attn_fwd_decode_paged(const void *q, const void *k_pages, const void *v_pages, void *o, float *lse,
                                    attn_dtype_t dtype, int B, int H_q, int H_kv, int D, int num_pages,
                                    int page_size, const int32_t *block_table, int max_pages, int64_t bt_stride,
                                    const int32_t *cache_lens, int max_cache_len, const int64_t q_str[4],
                                    const int64_t kp_str[4], const int64_t vp_str[4], const int64_t o_str[4],
                                    float scale, void *workspace, size_t workspace_bytes, void *stream) {
  return attn_fwd_decode_paged_ex(q, k_pages, v_pages, o, lse, dtype, B, H_q, H_kv, D, num_pages, page_size,
                                  block_table, max_pages, bt_stride, cache_lens, max_cache_len, q_str, kp_str, vp_str,
                                  o_str, scale, workspace, workspace_bytes, nullptr, stream);
}

attn_status_t attn_fwd_decode_paged_ex(const void *q, const void *k_pages, const void *v_pages, void *o, float *lse,
                                       attn_dtype_t dtype, int B, int H_q, int H_kv, int D, int num_pages,
                                       int page_size, const int32_t *block_table, int max_pages, int64_t bt_stride,
                                       const int32_t *cache_lens, int max_cache_len, const int64_t q_str[4],
                                       const int64_t kp_str[4], const int64_t vp_str[4], const int64_t o_str[4],
                                       float scale, void *workspace, size_t workspace_bytes,
                                       const attn_options_t *opts, void *stream) {
  if (!q || !k_pages || !v_pages || !o || !cache_lens || !q_str || !kp_str || !vp_str || !o_str)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H_q < 1 || H_kv < 1 || D < 1 || H_q % H_kv != 0 || max_cache_len < 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f) || B > 65535) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  attn_status_t st;
  if ((st = check_pages(num_pages, page_size, block_table, max_pages, bt_stride)) != ATTN_OK) return st;
  if (static_cast<int64_t>(max_cache_len) > static_cast<int64_t>(max_pages) * page_size) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_pages) || !aligned16(v_pages) || !aligned16(o) ||
      (lse && (reinterpret_cast<uintptr_t>(lse) & 3)) || (reinterpret_cast<uintptr_t>(cache_lens) & 3))
    return ATTN_ERR_ALIGNMENT;
  const int64_t qsz[4] = {B, H_q, 1, D}, psz[4] = {num_pages, H_kv, page_size, D};
  if ((st = check_strides(q_str, qsz)) || (st = check_strides(kp_str, psz)) || (st = check_strides(vp_str, psz)) ||
      (st = check_strides(o_str, qsz)))
    return st;
  Opts op;
  if ((st = read_opts(opts, &op)) != ATTN_OK) return st;
  if (op.kv_ranges != nullptr) return ATTN_ERR_UNSUPPORTED;  // key ranges are a prefill mask
  const int wl = op.wl;
  const float *slopes = op.slopes;
  const DeviceState *dev = nullptr;
  if ((st = device_state(&dev)) != ATTN_OK) return st;

  const int group = H_q / H_kv;
  const int gh = decode_heads_per_cta(group);
  const int nhc = (group + gh - 1) / gh;
  int nsplit = 1, chunk = max_cache_len;
  decode_plan(B, H_q, H_kv, decode_span(max_cache_len, wl), D, dev->sm_count, &nsplit, &chunk, op.num_splits);
  if (nsplit > 1) {
    const size_t need = decode_ws_bytes(B, H_q, D, nsplit);
    if (workspace == nullptr || workspace_bytes < need) return ATTN_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 15) != 0) return ATTN_ERR_ALIGNMENT;
  }
  if (static_cast<int64_t>(H_kv) * nhc > 65535) return ATTN_ERR_INVALID_ARG;
  DecodeParams p{};
  p.q = q;
  p.kc = k_pages;
  p.vc = v_pages;
  p.o = o;
  p.lse = lse;
  p.ws_o = static_cast<float *>(workspace);
  p.ws_lse = nsplit > 1 ? static_cast<float *>(workspace) + static_cast<size_t>(B) * H_q * nsplit * D : nullptr;
  p.err = dev->err;
  p.q_sb = q_str[0];
  p.q_sh = q_str[1];
  p.o_sb = o_str[0];
  p.o_sh = o_str[1];
  p.Hq = H_q;
  p.group = group;
  p.nhc = nhc;
  p.cache_len = max_cache_len;
  p.chunk = chunk;
  p.nsplit = nsplit;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.block_table = block_table;
  p.cache_lens = cache_lens;
  p.bt_stride = bt_stride;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.window_left = wl;
  p.alibi_slopes = slopes;
  if (op.rope_theta > 0.f) {
    p.rope = op.rope_interleaved ? 2 : 1;
    fill_rope_steps(op.rope_theta, D, p.rope_f);
  }
  // Tensor maps over the page pool: (d, row in page, kv head, page).
  CUtensorMap tk, tv;
  const bool bf16 = dtype == ATTN_BF16;
  const int rows = page_size < kDecodeStageTokens ? page_size : kDecodeStageTokens;
  if ((st = make_map(&tk, k_pages, bf16, psz, kp_str, rows, &p.slots_k)) ||
      (st = make_map(&tv, v_pages, bf16, psz, vp_str, rows, &p.slots_v)))
    return st;
  cudaError_t e = launch_decode(D, bf16, true, gh, tk, tv, p, B, H_kv, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t kv_cache_write_paged(void *k_pages, void *v_pages, const void *k_new, const void *v_new,
                                   attn_dtype_t dtype, int B, int H_kv, int n_new, int D, int num_pages,
                                   int page_size, const int32_t *block_table, int max_pages, int64_t bt_stride,
                                   const int32_t *positions, const int64_t kp_str[4], const int64_t vp_str[4],
                                   const int64_t kn_str[4], const int64_t vn_str[4], void *stream) {
  return kv_cache_write_paged_ex(k_pages, v_pages, k_new, v_new, dtype, B, H_kv, n_new, D, num_pages, page_size,
                                 block_table, max_pages, bt_stride, positions, kp_str, vp_str, kn_str, vn_str,
                                 nullptr, stream);
}

attn_status_t kv_cache_write_paged_ex(void *k_pages, void *v_pages, const void *k_new, const void *v_new,
                                      attn_dtype_t dtype, int B, int H_kv, int n_new, int D, int num_pages,
                                      int page_size, const int32_t *block_table, int max_pages, int64_t bt_stride,
                                      const int32_t *positions, const int64_t kp_str[4], const int64_t vp_str[4],
                                      const int64_t kn_str[4], const int64_t vn_str[4], const attn_options_t *opts,
                                      void *stream) {
  if (!k_pages || !v_pages || !k_new || !v_new || !positions || !kp_str || !vp_str || !kn_str || !vn_str)
    return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H_kv < 1 || n_new < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  attn_status_t st;
  if ((st = check_pages(num_pages, page_size, block_table, max_pages, bt_stride)) != ATTN_OK) return st;
  if (!aligned16(k_pages) || !aligned16(v_pages) || !aligned16(k_new) || !aligned16(v_new) ||
      (reinterpret_cast<uintptr_t>(positions) & 3))
    return ATTN_ERR_ALIGNMENT;
  const int64_t psz[4] = {num_pages, H_kv, page_size, D}, nsz[4] = {B, H_kv, n_new, D};
  if ((st = check_strides(kp_str, psz)) || (st = check_strides(vp_str, psz)) || (st = check_strides(kn_str, nsz)) ||
      (st = check_strides(vn_str, nsz)))
    return st;
  Opts op;
  if ((st = read_opts(opts, &op)) != ATTN_OK) return st;
  const DeviceState *dev = nullptr;
  if ((st = device_state(&dev)) != ATTN_OK) return st;
  KvWriteParams p{};
  p.kc = k_pages;
  p.vc = v_pages;
  p.kn = k_new;
  p.vn = v_new;
  p.kc_sb = kp_str[0];
  p.kc_sh = kp_str[1];
  p.kc_sn = kp_str[2];
  p.vc_sb = vp_str[0];
  p.vc_sh = vp_str[1];
  p.vc_sn = vp_str[2];
  p.kn_sb = kn_str[0];
  p.kn_sh = kn_str[1];
  p.kn_sn = kn_str[2];
  p.vn_sb = vn_str[0];
  p.vn_sh = vn_str[1];
  p.vn_sn = vn_str[2];
  p.Hkv = H_kv;
  p.n_new = n_new;
  p.D = D;
  p.total_units = static_cast<int64_t>(B) * H_kv * n_new * (D / 8);
  p.err = dev->err;
  p.block_table = block_table;
  p.positions = positions;
  p.bt_stride = bt_stride;
  p.page_size = page_size;
  p.max_pages = max_pages;
  p.num_pages = num_pages;
  p.is_bf16 = dtype == ATTN_BF16;
  if (op.rope_theta > 0.f) {
    p.rope = op.rope_interleaved ? 2 : 1;
    fill_rope_steps(op.rope_theta, D, p.rope_f);
  }
  cudaError_t e = launch_kv_cache_write(p, true, static_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_selftest_wait_timeout(void *stream) {
  const DeviceState *dev = nullptr;
  attn_status_t st = device_state(&dev);
  if (st != ATTN_OK) return st;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(dev->err);
  return cudaGetLastError() == cudaSuccess ? ATTN_OK : ATTN_ERR_CUDA;
}

attn_status_t attn_get_device_error(void *stream) {
  const DeviceState *dev = nullptr;
  attn_status_t st = device_state(&dev);
  if (st != ATTN_OK) return st;
  const cudaStream_t s = static_cast<cudaStream_t>(stream);
  // One host thread at a time uses the per-device "taken" word.
  static std::mutex take_mutex;
  std::lock_guard<std::mutex> lock(take_mutex);
  if (cudaStreamSynchronize(s) != cudaSuccess) return ATTN_ERR_CUDA;
  // Read and clear in one atomic exchange on the device.
  take_error_kernel<<<1, 1, 0, s>>>(dev->err, dev->taken);
  if (cudaGetLastError() != cudaSuccess) return ATTN_ERR_CUDA;
  unsigned word = 0;
  if (cudaMemcpyAsync(&word, dev->taken, sizeof(word), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (word == 0) return ATTN_OK;
  return (word & kErrWaitTimeout) ? ATTN_ERR_DEVICE_TIMEOUT : ATTN_ERR_DEVICE_INDEX;
}

const char *attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ATTN_OK";
    case ATTN_ERR_INVALID_ARG: return "ATTN_ERR_INVALID_ARG";
    case ATTN_ERR_UNSUPPORTED: return "ATTN_ERR_UNSUPPORTED";
    case ATTN_ERR_ALIGNMENT: return "ATTN_ERR_ALIGNMENT";
    case ATTN_ERR_WORKSPACE: return "ATTN_ERR_WORKSPACE";
    case ATTN_ERR_CUDA: return "ATTN_ERR_CUDA";
    case ATTN_ERR_DEVICE_TIMEOUT: return "ATTN_ERR_DEVICE_TIMEOUT";
    case ATTN_ERR_DEVICE_INDEX: return "ATTN_ERR_DEVICE_INDEX";
  }
  return "ATTN_ERR_UNKNOWN";
}

int attn_version(void) { return 200; }

}  // extern "C"

// ---------------------------------------------------------------------------
// attn_fwd_prefill_host: prefill from and to host buffers, copies pipelined
// against the compute in chunks of (batch element, block of kv heads).
namespace attn {
namespace {

struct CopyStreams {
  bool ready = false;
  cudaStream_t in = nullptr, out = nullptr;
};
std::mutex g_copy_mutex;
CopyStreams g_copy[kMaxDevices];

// Two non-blocking streams per device, created on first use and kept for the
// life of the process: host-to-device copies and device-to-host copies.
attn_status_t copy_streams(cudaStream_t *in, cudaStream_t *out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_copy_mutex);
  CopyStreams &c = g_copy[dev];
  if (!c.ready) {
    if (cudaStreamCreateWithFlags(&c.in, cudaStreamNonBlocking) != cudaSuccess) return ATTN_ERR_CUDA;
    if (cudaStreamCreateWithFlags(&c.out, cudaStreamNonBlocking) != cudaSuccess) return ATTN_ERR_CUDA;
    c.ready = true;
  }
  *in = c.in;
  *out = c.out;
  return ATTN_OK;
}

size_t round256(size_t x) { return (x + 255) & ~size_t(255); }

// Device staging: Q, O (B,H_q,N_q,D), K, V (B,H_kv,N_kv,D), LSE (B,H_q,N_q).
struct HostLayout {
  size_t q_bytes, kv_bytes, lse_bytes;
  size_t off_q, off_k, off_v, off_o, off_lse, total;
};
HostLayout host_layout(int B, int H_q, int H_kv, int N_q, int N_kv, int D) {
  HostLayout L{};
  L.q_bytes = static_cast<size_t>(B) * H_q * N_q * D * 2;
  L.kv_bytes = static_cast<size_t>(B) * H_kv * N_kv * D * 2;
  L.lse_bytes = static_cast<size_t>(B) * H_q * N_q * 4;
  L.off_q = 0;
  L.off_k = L.off_q + round256(L.q_bytes);
  L.off_v = L.off_k + round256(L.kv_bytes);
  L.off_o = L.off_v + round256(L.kv_bytes);
  L.off_lse = L.off_o + round256(L.q_bytes);
  L.total = L.off_lse + round256(L.lse_bytes);
  return L;
}

bool host_sizes_ok(int B, int H_q, int H_kv, int N_q, int N_kv, int D) {
  return B >= 1 && H_q >= 1 && H_kv >= 1 && N_q >= 1 && N_kv >= 1 && D >= 1 && H_q % H_kv == 0 && B <= 65535 &&
         H_q <= 65535;
}

}  // namespace
}  // namespace attn

extern "C" {

size_t attn_fwd_prefill_host_workspace_size(attn_dtype_t dtype, int B, int H_q, int H_kv, int N_q, int N_kv, int D) {
  if (!valid_dtype(dtype) || (D != 64 && D != 128) || !host_sizes_ok(B, H_q, H_kv, N_q, N_kv, D)) return 0;
  return host_layout(B, H_q, H_kv, N_q, N_kv, D).total;
}

attn_status_t attn_fwd_prefill_host(const void *q, const void *k, const void *v, void *o, float *lse,
                                    attn_dtype_t dtype, int B, int H_q, int H_kv, int N_q, int N_kv, int D,
                                    int causal, float scale, const attn_options_t *opts, void *workspace,
                                    size_t workspace_bytes, void *stream) {
  if (!q || !k || !v || !o || !host_sizes_ok(B, H_q, H_kv, N_q, N_kv, D) || (causal != 0 && causal != 1))
    return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (!valid_dtype(dtype) || (D != 64 && D != 128)) return ATTN_ERR_UNSUPPORTED;
  attn_status_t st;
  Opts op;
  if ((st = read_opts(opts, &op, true)) != ATTN_OK) return st;
  const int wl = op.wl, wr = op.wr;
  const float *slopes = op.slopes;
  const HostLayout L = host_layout(B, H_q, H_kv, N_q, N_kv, D);
  if (workspace == nullptr || workspace_bytes < L.total) return ATTN_ERR_WORKSPACE;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255) != 0) return ATTN_ERR_ALIGNMENT;
  const DeviceState *dev = nullptr;
  if ((st = device_state(&dev)) != ATTN_OK) return st;
  // The chunks run attn_fwd_prefill_ex; a kernel choice it would refuse is
  // refused here, before anything is enqueued.
  const bool masked = wl >= 0 || (causal == 0 && wr >= 0) || slopes != nullptr || op.kv_ranges != nullptr;
  if (op.prefill_kernel == 2 && (D != 128 || masked || op.rope_theta > 0.f || dev->pair_clusters <= 0))
    return ATTN_ERR_UNSUPPORTED;
  cudaStream_t s_in, s_out;
  if ((st = copy_streams(&s_in, &s_out)) != ATTN_OK) return st;
  const cudaStream_t s_comp = static_cast<cudaStream_t>(stream);

  // Chunk = (batch element, block of kv heads) with at least ~2 units per SM,
  // so that each chunk's launch still fills the GPU.
  const int group = H_q / H_kv;
  const int64_t pairs = (N_q + 2 * kPrefillBM - 1) / (2 * kPrefillBM);
  const int64_t want = 2 * static_cast<int64_t>(dev->sm_count);
  const int64_t per_kvh = static_cast<int64_t>(group) * pairs;
  const int kvh = static_cast<int>(std::min<int64_t>(H_kv, std::max<int64_t>(1, (want + per_kvh - 1) / per_kvh)));
  // The checks attn_fwd_prefill_ex applies to a chunk's shapes, made here for
  // the largest chunk before anything is enqueued: the unit count of the
  // persistent schedule and the tensor-map stride limit.
  if (static_cast<int64_t>(kvh) * per_kvh + dev->sm_count > 0x7fffffff) return ATTN_ERR_INVALID_ARG;
  if (static_cast<uint64_t>(kvh) * group * N_q * D * 2 >= (1ull << 40) ||
      static_cast<uint64_t>(kvh) * N_kv * D * 2 >= (1ull << 40))
    return ATTN_ERR_ALIGNMENT;

  char *ws = static_cast<char *>(workspace);
  char *dq = ws + L.off_q, *dk = ws + L.off_k, *dv = ws + L.off_v, *dout = ws + L.off_o;
  float *dl = reinterpret_cast<float *>(ws + L.off_lse);
  const size_t qrow = static_cast<size_t>(N_q) * D * 2, kvrow = static_cast<size_t>(N_kv) * D * 2;  // one head

  cudaEvent_t ev_start;
  if (cudaEventCreateWithFlags(&ev_start, cudaEventDisableTiming) != cudaSuccess) return ATTN_ERR_CUDA;
  // Copies into the staging buffers wait for earlier work on the caller's stream.
  bool fine = cudaEventRecord(ev_start, s_comp) == cudaSuccess && cudaStreamWaitEvent(s_in, ev_start, 0) == cudaSuccess;
  cudaEventDestroy(ev_start);
  for (int b = 0; fine && b < B; ++b) {
    for (int h0 = 0; fine && h0 < H_kv; h0 += kvh) {
      const int nh = std::min(kvh, H_kv - h0), qh0 = h0 * group, nqh = nh * group;
      const size_t qo = (static_cast<size_t>(b) * H_q + qh0) * qrow, qn = nqh * qrow;
      const size_t ko = (static_cast<size_t>(b) * H_kv + h0) * kvrow, kn = nh * kvrow;
      const size_t lo = (static_cast<size_t>(b) * H_q + qh0) * N_q * 4, ln = static_cast<size_t>(nqh) * N_q * 4;
      cudaEvent_t ev_in, ev_done;
      if (cudaEventCreateWithFlags(&ev_in, cudaEventDisableTiming) != cudaSuccess) {
        fine = false;
        break;
      }
      if (cudaEventCreateWithFlags(&ev_done, cudaEventDisableTiming) != cudaSuccess) {
        cudaEventDestroy(ev_in);
        fine = false;
        break;
      }
      fine = cudaMemcpyAsync(dq + qo, static_cast<const char *>(q) + qo, qn, cudaMemcpyHostToDevice, s_in) ==
                 cudaSuccess &&
             cudaMemcpyAsync(dk + ko, static_cast<const char *>(k) + ko, kn, cudaMemcpyHostToDevice, s_in) ==
                 cudaSuccess &&
             cudaMemcpyAsync(dv + ko, static_cast<const char *>(v) + ko, kn, cudaMemcpyHostToDevice, s_in) ==
                 cudaSuccess &&
             cudaEventRecord(ev_in, s_in) == cudaSuccess && cudaStreamWaitEvent(s_comp, ev_in, 0) == cudaSuccess;
      if (fine) {
        // The chunk is a contiguous (1, nqh, N_q, D) / (1, nh, N_kv, D) problem.
        const int64_t sq[4] = {static_cast<int64_t>(nqh) * N_q * D, static_cast<int64_t>(N_q) * D, D, 1};
        const int64_t sk[4] = {static_cast<int64_t>(nh) * N_kv * D, static_cast<int64_t>(N_kv) * D, D, 1};
        attn_options_t oc{wl, wr, slopes ? slopes + qh0 : nullptr, op.rope_theta, op.rope_interleaved, 0,
                          op.rope_rotated_keys,
                          op.kv_ranges ? op.kv_ranges + static_cast<size_t>(b) * N_q * 2 : nullptr,
                          op.prefill_kernel};
        const attn_status_t cs = attn_fwd_prefill_ex(dq + qo, dk + ko, dv + ko, dout + qo,
                                                     lse ? reinterpret_cast<float *>(reinterpret_cast<char *>(dl) + lo)
                                                         : nullptr,
                                                     dtype, 1, nqh, nh, N_q, N_kv, D, sq, sk, sk, sq, causal, scale,
                                                     &oc, stream);
        if (cs != ATTN_OK) {
          // Not expected after the checks above; the copies already enqueued on
          // the library's streams are joined to the caller's stream first.
          cudaEventDestroy(ev_in);
          cudaEventDestroy(ev_done);
          cudaEvent_t ev_j;
          if (cudaEventCreateWithFlags(&ev_j, cudaEventDisableTiming) == cudaSuccess) {
            cudaEventRecord(ev_j, s_in);
            cudaStreamWaitEvent(s_comp, ev_j, 0);
            cudaEventRecord(ev_j, s_out);
            cudaStreamWaitEvent(s_comp, ev_j, 0);
            cudaEventDestroy(ev_j);
          }
          return cs;
        }
        fine = cudaEventRecord(ev_done, s_comp) == cudaSuccess && cudaStreamWaitEvent(s_out, ev_done, 0) == cudaSuccess &&
               cudaMemcpyAsync(static_cast<char *>(o) + qo, dout + qo, qn, cudaMemcpyDeviceToHost, s_out) ==
                   cudaSuccess &&
               (!lse || cudaMemcpyAsync(reinterpret_cast<char *>(lse) + lo, reinterpret_cast<char *>(dl) + lo, ln,
                                        cudaMemcpyDeviceToHost, s_out) == cudaSuccess);
      }
      cudaEventDestroy(ev_in);
      cudaEventDestroy(ev_done);
    }
  }
  // The caller's stream waits for the last device-to-host copy.
  cudaEvent_t ev_end;
  if (cudaEventCreateWithFlags(&ev_end, cudaEventDisableTiming) != cudaSuccess) return ATTN_ERR_CUDA;
  const bool joined = cudaEventRecord(ev_end, s_out) == cudaSuccess && cudaStreamWaitEvent(s_comp, ev_end, 0) == cudaSuccess;
  cudaEventDestroy(ev_end);
  return (fine && joined) ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// attn_fwd_decode_noalloc: decode whose split scratch lives in a fixed array
// compiled into the library instead of a caller-provided buffer.
namespace attn {
namespace {

// Scratch for the split partials of attn_fwd_decode_noalloc.  It lives in the
// library image, so every device that loads the library holds these bytes
// until the process exits, and every call on a device shares them.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mutex;
void *g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device.  The name
// g_noalloc_scratch means nothing to the device in host code, so the address
// is looked up once per device, with that device current.
attn_status_t noalloc_scratch(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_noalloc_mutex);
  if (g_noalloc_ptr[dev] == nullptr) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) return ATTN_ERR_CUDA;
    g_noalloc_ptr[dev] = ptr;
  }
  *out = g_noalloc_ptr[dev];
  return ATTN_OK;
}

}  // namespace
}  // namespace attn

extern "C" {

attn_status_t attn_fwd_decode_noalloc(const void *q, const void *k_cache, const void *v_cache, void *o, float *lse,
                                      attn_dtype_t dtype, int B, int H_q, int H_kv, int cache_len, int D,
                                      const int64_t q_str[4], const int64_t kc_str[4], const int64_t vc_str[4],
                                      const int64_t o_str[4], float scale, void *stream) {
  // The same argument checks, in the same order, as attn_fwd_decode; then the
  // scratch this call would need must fit the fixed array.
  attn_status_t st = decode_check_args(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D, q_str, kc_str,
                                       vc_str, o_str, scale);
  if (st != ATTN_OK) return st;
  const DeviceState *dev = nullptr;
  if ((st = device_state(&dev)) != ATTN_OK) return st;
  int nsplit = 1, chunk = cache_len;
  decode_plan(B, H_q, H_kv, cache_len, D, dev->sm_count, &nsplit, &chunk);
  if (decode_ws_bytes(B, H_q, D, nsplit) > kNoAllocScratchBytes) return ATTN_ERR_WORKSPACE;
  void *scratch = nullptr;
  if ((st = noalloc_scratch(&scratch)) != ATTN_OK) return st;
  // Nothing in the scratch has to start at zero: each partial the merge kernel
  // reads is written earlier in the same call.
  return attn_fwd_decode(q, k_cache, v_cache, o, lse, dtype, B, H_q, H_kv, cache_len, D, q_str, kc_str, vc_str,
                         o_str, scale, scratch, kNoAllocScratchBytes, stream);
}

}  // extern "C"
