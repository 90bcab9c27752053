// decode.cu -- split-KV decode attention and the KV-cache write, sm_103a.
//
// Decode ("Triton-FlashAttention", Phase 2): one new query token per
// (batch, q-head) attends to the first cache_len rows of a preallocated cache.
// The work is HBM-bound (every cached K/V byte is read once per step), so
// this path stays on the CUDA cores and is built for streaming:
//
//   decode_split: one CTA per (split, kv-head [x head chunk], batch).  The
//     CTA reads its share of the cache ONCE for all H_q/H_kv query heads of
//     the group.  Each row of K or V is read by D/8 lanes with 128-bit
//     non-caching loads (a warp covers 256/D consecutive tokens per load,
//     fully coalesced), next-step rows are prefetched while the current
//     step is reduced, dot products are finished with xor warp shuffles
//     across the lanes of a row, and every group of lanes keeps its own
//     online-softmax state (running max, running sum, unnormalised output
//     slice), in base-2 units.  The groups of a CTA are merged through shared
//     memory at the end.
//   decode_merge: when the cache is split over several CTAs, combines the
//     partials of every (b, q-head): lse = ln sum_s e^{lse_s},
//     O = sum_s e^{lse_s - lse} O_s.
//
// kv_cache_write: copies new tokens into cache rows [pos, pos + n) with one
// 16-byte piece per thread.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attn {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kU = 4;  // tokens per lane group per step
constexpr float kLn2 = 0.693147180559945309f;

__device__ __forceinline__ uint4 ld_stream(const void *p) {
  uint4 v;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

template <bool BF16>
__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if constexpr (BF16) {
      __nv_bfloat162 h = *reinterpret_cast<const __nv_bfloat162 *>(&w[i]);
      float2 t = __bfloat1622float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    } else {
      __half2 h = *reinterpret_cast<const __half2 *>(&w[i]);
      float2 t = __half22float2(h);
      f[2 * i] = t.x;
      f[2 * i + 1] = t.y;
    }
  }
}

template <bool BF16>
__device__ __forceinline__ void store_out(void *base, int64_t idx, float x) {
  if constexpr (BF16)
    reinterpret_cast<__nv_bfloat16 *>(base)[idx] = __float2bfloat16_rn(x);
  else
    reinterpret_cast<__half *>(base)[idx] = __float2half_rn(x);
}

template <int D, int GH, bool BF16>
__global__ void __launch_bounds__(kThreads) decode_split_kernel(const DecodeParams p) {
  constexpr int LPT = D / 8;       // lanes per token row (16 bytes each)
  constexpr int GPW = 32 / LPT;    // lane groups per warp
  constexpr int NG = kWarps * GPW; // lane groups per CTA
  constexpr int U = (GH >= 8) ? 2 : kU;  // tokens per lane group per step
  constexpr int STEP = NG * U;     // tokens per CTA step
  __shared__ float sm_m[NG][GH];
  __shared__ float sm_l[NG][GH];
  __shared__ float sm_acc[NG][GH][D];

  if (load_volatile(p.err) != 0) return;

  const int split = blockIdx.x;
  const int hk = blockIdx.y / p.nhc, hc = blockIdx.y % p.nhc;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int gi = warp * GPW + lane / LPT;
  const int d0 = (lane % LPT) * 8;
  const int h_first = hk * p.group + hc * GH;  // first q head of this CTA
  const int nh = min(GH, p.group - hc * GH);   // q heads actually handled

  // Query slices, pre-multiplied by scale * log2(e).
  float qf[GH][8];
#pragma unroll
  for (int i = 0; i < GH; ++i) {
    if (i < nh) {
      const char *qp = reinterpret_cast<const char *>(p.q) +
                       2 * (static_cast<int64_t>(b) * p.q_sb + static_cast<int64_t>(h_first + i) * p.q_sh + d0);
      float f[8];
      unpack8<BF16>(*reinterpret_cast<const uint4 *>(qp), f);
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[i][e] = f[e] * p.scale_log2;
    } else {
#pragma unroll
      for (int e = 0; e < 8; ++e) qf[i][e] = 0.f;
    }
  }

  float m[GH], l[GH], acc[GH][8];
#pragma unroll
  for (int i = 0; i < GH; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc[i][e] = 0.f;
  }

  const int t_begin = split * p.chunk;
  const int t_end = min(t_begin + p.chunk, p.cache_len);
  const char *kbase = reinterpret_cast<const char *>(p.kc) +
                      2 * (static_cast<int64_t>(b) * p.kc_sb + static_cast<int64_t>(hk) * p.kc_sh + d0);
  const char *vbase = reinterpret_cast<const char *>(p.vc) +
                      2 * (static_cast<int64_t>(b) * p.vc_sb + static_cast<int64_t>(hk) * p.vc_sh + d0);
  const int64_t kstep = 2 * p.kc_sn, vstep = 2 * p.vc_sn;

  // Raw 16-byte pieces of the current step; the next step's are loaded while
  // this one is reduced.
  uint4 kr[U], vr[U];
  auto load_step = [&](int base, uint4 (&kk)[U], uint4 (&vv)[U]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int t = base + u * NG + gi;
      if (t < t_end) {
        kk[u] = ld_stream(kbase + t * kstep);
        vv[u] = ld_stream(vbase + t * vstep);
      } else {
        kk[u] = make_uint4(0, 0, 0, 0);
        vv[u] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  load_step(t_begin, kr, vr);
  for (int base = t_begin; base < t_end; base += STEP) {
    uint4 kn[U], vn[U];
    const bool more = base + STEP < t_end;
    if (more) load_step(base + STEP, kn, vn);

    float s[U][GH];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float kf[8];
      unpack8<BF16>(kr[u], kf);
#pragma unroll
      for (int i = 0; i < GH; ++i) {
        float a = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) a = fmaf(qf[i][e], kf[e], a);
        s[u][i] = a;
      }
    }
#pragma unroll
    for (int off = LPT / 2; off >= 1; off >>= 1)
#pragma unroll
      for (int u = 0; u < U; ++u)
#pragma unroll
        for (int i = 0; i < GH; ++i) s[u][i] += __shfl_xor_sync(0xffffffffu, s[u][i], off);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (base + u * NG + gi >= t_end) {
#pragma unroll
        for (int i = 0; i < GH; ++i) s[u][i] = -INFINITY;
      }
    }
    float pw[U][GH];
#pragma unroll
    for (int i = 0; i < GH; ++i) {
      float mx = s[0][i];
#pragma unroll
      for (int u = 1; u < U; ++u) mx = fmaxf(mx, s[u][i]);
      const float m_new = fmaxf(m[i], mx);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
      const float alpha = fast_exp2(m[i] - m_use);
      l[i] *= alpha;
#pragma unroll
      for (int e = 0; e < 8; ++e) acc[i][e] *= alpha;
#pragma unroll
      for (int u = 0; u < U; ++u) {
        pw[u][i] = fast_exp2(s[u][i] - m_use);
        l[i] += pw[u][i];
      }
      m[i] = m_new;
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float vf[8];
      unpack8<BF16>(vr[u], vf);
#pragma unroll
      for (int i = 0; i < GH; ++i)
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[i][e] = fmaf(pw[u][i], vf[e], acc[i][e]);
    }
    if (more) {
#pragma unroll
      for (int u = 0; u < U; ++u) {
        kr[u] = kn[u];
        vr[u] = vn[u];
      }
    }
  }

  // Merge the lane groups of this CTA.
  if ((lane % LPT) == 0) {
#pragma unroll
    for (int i = 0; i < GH; ++i) {
      sm_m[gi][i] = m[i];
      sm_l[gi][i] = l[i];
    }
  }
#pragma unroll
  for (int i = 0; i < GH; ++i)
#pragma unroll
    for (int e = 0; e < 8; ++e) sm_acc[gi][i][d0 + e] = acc[i][e];
  __syncthreads();

  for (int idx = threadIdx.x; idx < nh * D; idx += kThreads) {
    const int i = idx / D, d = idx % D;
    float M = -INFINITY;
#pragma unroll
    for (int g = 0; g < NG; ++g) M = fmaxf(M, sm_m[g][i]);
    const float M_use = (M == -INFINITY) ? 0.f : M;
    float L = 0.f, A = 0.f;
#pragma unroll
    for (int g = 0; g < NG; ++g) {
      const float w = fast_exp2(sm_m[g][i] - M_use);
      L = fmaf(sm_l[g][i], w, L);
      A = fmaf(sm_acc[g][i][d], w, A);
    }
    const int hq = h_first + i;
    const float o = (L > 0.f) ? A / L : 0.f;
    const float lse = (L > 0.f) ? (M + __log2f(L)) * kLn2 : -INFINITY;
    if (p.nsplit == 1) {
      store_out<BF16>(p.o, static_cast<int64_t>(b) * p.o_sb + static_cast<int64_t>(hq) * p.o_sh + d, o);
      if (d == 0 && p.lse != nullptr) p.lse[static_cast<int64_t>(b) * p.Hq + hq] = lse;
    } else {
      const int64_t row = (static_cast<int64_t>(b) * p.Hq + hq) * p.nsplit + split;
      p.ws_o[row * D + d] = o;
      if (d == 0) p.ws_lse[row] = lse;
    }
  }
}

template <int D, bool BF16>
__global__ void __launch_bounds__(D) decode_merge_kernel(const DecodeParams p) {
  const int bh = blockIdx.x;
  const int b = bh / p.Hq, hq = bh % p.Hq;
  const int d = threadIdx.x;
  const float *ls = p.ws_lse + static_cast<int64_t>(bh) * p.nsplit;
  const float *os = p.ws_o + static_cast<int64_t>(bh) * p.nsplit * D;
  float M = -INFINITY;
  for (int s = 0; s < p.nsplit; ++s) M = fmaxf(M, ls[s]);
  float W = 0.f, A = 0.f;
  if (M != -INFINITY) {
    for (int s = 0; s < p.nsplit; ++s) {
      const float w = expf(ls[s] - M);
      W += w;
      A = fmaf(w, os[static_cast<int64_t>(s) * D + d], A);
    }
  }
  store_out<BF16>(p.o, static_cast<int64_t>(b) * p.o_sb + static_cast<int64_t>(hq) * p.o_sh + d,
                  W > 0.f ? A / W : 0.f);
  if (d == 0 && p.lse != nullptr) p.lse[bh] = W > 0.f ? M + logf(W) : -INFINITY;
}

__global__ void __launch_bounds__(256) kv_cache_write_kernel(const KvWriteParams p) {
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

template <int D, int GH, bool BF16>
cudaError_t launch_split(const DecodeParams &p, int B, int Hkv, cudaStream_t stream) {
  dim3 grid(p.nsplit, Hkv * p.nhc, B);
  decode_split_kernel<D, GH, BF16><<<grid, kThreads, 0, stream>>>(p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || p.nsplit == 1) return e;
  decode_merge_kernel<D, BF16><<<B * p.Hq, D, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

int decode_heads_per_cta(int group) {
  if (group <= 1) return 1;
  if (group <= 2) return 2;
  if (group <= 4) return 4;
  return 8;
}

int decode_tokens_per_step(int D) { return kWarps * (32 / (D / 8)) * kU; }  // a multiple of every U

cudaError_t launch_decode(int D, bool bf16, int gh, const DecodeParams &p, int B, int Hkv, cudaStream_t stream) {
#define ATTN_DECODE_CASE(DD, GG, BB) \
  if (D == DD && gh == GG && bf16 == BB) return launch_split<DD, GG, BB>(p, B, Hkv, stream);
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

cudaError_t launch_kv_cache_write(const KvWriteParams &p, cudaStream_t stream) {
  const int64_t work = 2 * p.total_units;
  int64_t blocks = (work + 255) / 256;
  if (blocks > 65535 * 8) blocks = 65535 * 8;
  kv_cache_write_kernel<<<static_cast<unsigned>(blocks), 256, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace attn
