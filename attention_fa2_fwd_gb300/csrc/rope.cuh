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

// Rotates the 8 pairs of one group held in two 16-byte chunks.  Rotate-half
// layout: word k of chunk A holds x_a of pairs 2k, 2k+1 and word k of chunk B
// their x_b.  Interleaved layout: word k of A holds pair k (x_a, x_b) and word
// k of B pair 4 + k.  cs[i], sn[i]: cos and sin of pair i of the group.
template <bool BF16, bool INTERLEAVED>
__device__ __forceinline__ void rope_rotate_group(uint4 &A, uint4 &B, const float (&cs)[8], const float (&sn)[8]) {
  uint32_t *a = reinterpret_cast<uint32_t *>(&A);
  uint32_t *b = reinterpret_cast<uint32_t *>(&B);
  if constexpr (!INTERLEAVED) {
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 xa = rope_unpack<BF16>(a[k]), xb = rope_unpack<BF16>(b[k]);
      const uint64_t c2 = pack_f2(cs[2 * k], cs[2 * k + 1]), s2 = pack_f2(sn[2 * k], sn[2 * k + 1]);
      const uint64_t ns2 = pack_f2(-sn[2 * k], -sn[2 * k + 1]);
      const uint64_t va = pack_f2(xa.x, xa.y), vb = pack_f2(xb.x, xb.y);
      const float2 ya = unpack_f2(ffma_f2(va, c2, fmul_f2(vb, ns2)));  // x_a c - x_b s
      const float2 yb = unpack_f2(ffma_f2(vb, c2, fmul_f2(va, s2)));   // x_b c + x_a s
      a[k] = rope_pack<BF16>(ya.x, ya.y);
      b[k] = rope_pack<BF16>(yb.x, yb.y);
    }
  } else {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      uint32_t *w = h == 0 ? a : b;
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int i = 4 * h + k;
        const float2 x = rope_unpack<BF16>(w[k]);
        // (x_a', x_b') = (x_a, x_b) c + (x_b, x_a) (-s, s)
        const float2 y = unpack_f2(
            ffma_f2(pack_f2(x.x, x.y), pack_f2(cs[i], cs[i]), fmul_f2(pack_f2(x.y, x.x), pack_f2(-sn[i], sn[i]))));
        w[k] = rope_pack<BF16>(y.x, y.y);
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

// Advances (cs, sn) of 8 pairs by one position: angle + step.
__device__ __forceinline__ void rope_step(float (&cs)[8], float (&sn)[8], const float (&c1)[8], const float (&s1)[8]) {
#pragma unroll
  for (int i = 0; i < 8; i += 2) {
    const uint64_t c = pack_f2(cs[i], cs[i + 1]), s = pack_f2(sn[i], sn[i + 1]);
    const uint64_t cc1 = pack_f2(c1[i], c1[i + 1]), ss1 = pack_f2(s1[i], s1[i + 1]);
    const uint64_t nss1 = pack_f2(-s1[i], -s1[i + 1]);
    const float2 cn = unpack_f2(ffma_f2(c, cc1, fmul_f2(s, nss1)));  // cos(a + d) = cos a cos d - sin a sin d
    const float2 sv = unpack_f2(ffma_f2(s, cc1, fmul_f2(c, ss1)));   // sin(a + d) = sin a cos d + cos a sin d
    cs[i] = cn.x;
    cs[i + 1] = cn.y;
    sn[i] = sv.x;
    sn[i + 1] = sv.y;
  }
}

}  // namespace attn
