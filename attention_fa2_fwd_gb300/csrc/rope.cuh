// rope.cuh -- rotary position embeddings (RoPE) on chip, shared by the
// prefill kernel, the decode kernel and the KV-cache write.
//
// Pair c of a query or key row at position p turns by p * theta^(-2c/D)
// radians (x_a' = x_a cos - x_b sin, x_b' = x_b cos + x_a sin).  The host
// gives each pair's angle per unit position as a 64-bit fixed-point fraction
// of a full turn, f_c = frac(theta^(-2c/D) / 2 pi) * 2^64, so the angle at p
// is (p * f_c mod 2^64) / 2^64 turns: the wrap-around of the 64-bit product
// is the reduction modulo one turn, exact for any position.  Its top 32 bits,
// read as a signed fraction of a half turn, go to sincospif.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <cstdint>

#include "ptx.cuh"

namespace attn {

// sin and cos of the angle of a pair with turn step f at integer position pos.
__device__ __forceinline__ void rope_sincos(uint32_t pos, uint64_t f, float *s, float *c) {
  const uint64_t t = static_cast<uint64_t>(pos) * f;   // turns, modulo 1, as a 64-bit fraction
  const int32_t hi = static_cast<int32_t>(t >> 32);    // signed: [-1/2, 1/2) turn in units of 2^-32
  sincospif(static_cast<float>(hi) * 4.656612873077393e-10f, s, c);  // x 2^-31: sin/cos(pi x) = sin/cos(2 pi t)
}

// Two 16-bit values of a 32-bit word as floats (element order kept), and back.
template <bool BF16>
__device__ __forceinline__ float2 rope_unpack(uint32_t w) {
  if constexpr (BF16) {
    return make_float2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
  } else {
    return __half22float2(*reinterpret_cast<const __half2 *>(&w));
  }
}
template <bool BF16>
__device__ __forceinline__ uint32_t rope_pack(float a, float b) {
  if constexpr (BF16) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  } else {
    __half2 v = __floats2half2_rn(a, b);
    return *reinterpret_cast<uint32_t *>(&v);
  }
}

// Rotates the 8 pairs of one group held in two 16-byte chunks, in scalar
// fp32 (one multiply and one fused multiply-add per coordinate; negations fold
// into the FMA).  Rotate-half layout: word k of chunk A holds x_a of pairs
// 2k, 2k+1 and word k of chunk B their x_b.  Interleaved layout: word k of A
// holds pair k (x_a, x_b) and word k of B pair 4 + k.  cs[i], sn[i]: cos and
// sin of pair i of the group.
template <bool BF16, bool INTERLEAVED>
__device__ __forceinline__ void rope_rotate_group(uint4 &A, uint4 &B, const float (&cs)[8], const float (&sn)[8]) {
  uint32_t *a = reinterpret_cast<uint32_t *>(&A);
  uint32_t *b = reinterpret_cast<uint32_t *>(&B);
  if constexpr (!INTERLEAVED) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 xa = rope_unpack<BF16>(a[k]), xb = rope_unpack<BF16>(b[k]);
      const float c0 = cs[2 * k], s0 = sn[2 * k], c1 = cs[2 * k + 1], s1 = sn[2 * k + 1];
      a[k] = rope_pack<BF16>(fmaf(xa.x, c0, -xb.x * s0), fmaf(xa.y, c1, -xb.y * s1));
      b[k] = rope_pack<BF16>(fmaf(xb.x, c0, xa.x * s0), fmaf(xb.y, c1, xa.y * s1));
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t *w = h == 0 ? a : b;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = 4 * h + k;
        const float2 x = rope_unpack<BF16>(w[k]);
        w[k] = rope_pack<BF16>(fmaf(x.x, cs[i], -x.y * sn[i]), fmaf(x.y, cs[i], x.x * sn[i]));
      }
    }
  }
}

// Chunk indices (16-byte units of a row) of group g: rotate-half pairs
// (c, c + D/2) -> chunks g and g + D/16; interleaved pairs (2c, 2c+1) -> 2g, 2g+1.
template <int D, bool INTERLEAVED>
__device__ __forceinline__ void rope_group_chunks(int g, int *ca, int *cb) {
  if constexpr (INTERLEAVED) {
    *ca = 2 * g;
    *cb = 2 * g + 1;
  } else {
    *ca = g;
    *cb = g + D / 16;
  }
}

// (cos, sin) of 8 pairs along consecutive positions: each step turns them by
// the angle of one position (cos(a + t) = cos a cos t - sin a sin t, sin(a + t)
// = sin a cos t + cos a sin t), a rotation, so the errors stay near one
// rounding per step (a thread walks at most 16 rows).  (A three-term
// recurrence, one FMA per value, was tried: its errors grow quadratically with
// the steps and visibly moved 16-bit roundings.)
struct RopeWalk {
  float cs[8], sn[8];  // at the current position
  __device__ __forceinline__ void start(const float (&cs0)[8], const float (&sn0)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      cs[i] = cs0[i];
      sn[i] = sn0[i];
    }
  }
  // c1, s1: cos and sin of one position's angle.
  __device__ __forceinline__ void step(const float (&c1)[8], const float (&s1)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float nc = fmaf(cs[i], c1[i], -sn[i] * s1[i]), ns = fmaf(sn[i], c1[i], cs[i] * s1[i]);
      cs[i] = nc;
      sn[i] = ns;
    }
  }
};

}  // namespace attn
