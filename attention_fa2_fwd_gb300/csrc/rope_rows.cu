// rope_rows.cu -- rotary position embeddings applied to whole rows of (B, H,
// N, D) tensors in HBM, forwards or backwards.
//
// The backward of rotary attention ("Triton-FlashAttention", RoPE among the
// fused extensions) runs the plain backward on the rotated queries and keys
// Q' = R Q, K' = R K, and turns the resulting dQ', dK' back with R^T: R rotates
// pair c of the row at position n by n * theta^(-2c/D), so R^T is the rotation
// by the opposite angle (same cosine, negated sine).
//
// One thread owns one group of 8 pairs (two 16-byte chunks, the layout of
// rope_rotate_group) at one position n, computes the 8 (cos, sin) exactly from
// the fixed-point turn steps, and applies them to that chunk pair in up to
// kRowsPerThread consecutive (b, h) rows.  A warp covers 32 / (D / 16)
// consecutive positions of one (b, h), so each of its loads and stores covers
// whole rows: fully coalesced, HBM-bound (read and write each element once).
#include "attn_internal.h"
#include "rope.cuh"

namespace attn {

namespace {

constexpr int kRopeRowsThreads = 256;
constexpr int kRowsPerThread = 8;

template <bool BF16, bool INTERLEAVED, int D>
__global__ void __launch_bounds__(kRopeRowsThreads) rope_rows_kernel(const __grid_constant__ RopeRowsParams p) {
  const RopeRowsJob &job = p.job[blockIdx.y];
  constexpr int G = D / 16;  // groups of 8 pairs per row
  const int64_t pos_blocks = (static_cast<int64_t>(job.N) * G + kRopeRowsThreads - 1) / kRopeRowsThreads;
  const int64_t bh_total = static_cast<int64_t>(p.B) * job.H;
  const int64_t bh_blocks = (bh_total + kRowsPerThread - 1) / kRowsPerThread;
  if (static_cast<int64_t>(blockIdx.x) >= pos_blocks * bh_blocks) return;
  const int64_t t = (blockIdx.x % pos_blocks) * kRopeRowsThreads + threadIdx.x;
  if (t >= static_cast<int64_t>(job.N) * G) return;
  const int n = static_cast<int>(t / G), g = static_cast<int>(t % G);
  const int64_t bh0 = (blockIdx.x / pos_blocks) * kRowsPerThread;

  float cs[8], sn[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    rope_sincos(static_cast<uint32_t>(n), p.rope_f[8 * g + i], &sn[i], &cs[i]);
    sn[i] *= p.sin_sign;
  }
  int ca, cb;
  rope_group_chunks<D, INTERLEAVED>(g, &ca, &cb);

  uint4 A[kRowsPerThread], Bv[kRowsPerThread];
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
    const int64_t bh = bh0 + r;
    if (bh < bh_total) {
      const int64_t b = bh / job.H, h = bh - b * job.H;
      const uint4 *row = reinterpret_cast<const uint4 *>(static_cast<const uint16_t *>(job.src) + b * job.s_sb +
                                                         h * job.s_sh + n * job.s_sn);
      A[r] = row[ca];
      Bv[r] = row[cb];
    }
  }
#pragma unroll
  for (int r = 0; r < kRowsPerThread; ++r) {
    const int64_t bh = bh0 + r;
    if (bh < bh_total) {
      const int64_t b = bh / job.H, h = bh - b * job.H;
      rope_rotate_group<BF16, INTERLEAVED>(A[r], Bv[r], cs, sn);
      uint4 *row = reinterpret_cast<uint4 *>(static_cast<uint16_t *>(job.dst) + b * job.d_sb + h * job.d_sh +
                                             n * job.d_sn);
      row[ca] = A[r];
      row[cb] = Bv[r];
    }
  }
}

template <bool BF16, bool INTERLEAVED, int D>
cudaError_t launch_one(const RopeRowsParams &p, int n_jobs, cudaStream_t stream) {
  constexpr int G = D / 16;
  int64_t blocks = 0;
  for (int j = 0; j < n_jobs; ++j) {
    const int64_t pos_blocks = (static_cast<int64_t>(p.job[j].N) * G + kRopeRowsThreads - 1) / kRopeRowsThreads;
    const int64_t bh_blocks = (static_cast<int64_t>(p.B) * p.job[j].H + kRowsPerThread - 1) / kRowsPerThread;
    blocks = pos_blocks * bh_blocks > blocks ? pos_blocks * bh_blocks : blocks;
  }
  if (blocks < 1 || blocks > 0x7fffffff) return cudaErrorInvalidValue;
  rope_rows_kernel<BF16, INTERLEAVED, D>
      <<<dim3(static_cast<unsigned>(blocks), n_jobs), kRopeRowsThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_rope_rows(int D, bool bf16, bool interleaved, const RopeRowsParams &p, int n_jobs,
                             cudaStream_t stream) {
  if (n_jobs < 1 || n_jobs > 2) return cudaErrorInvalidValue;
  if (D == 128) {
    if (bf16) return interleaved ? launch_one<true, true, 128>(p, n_jobs, stream) : launch_one<true, false, 128>(p, n_jobs, stream);
    return interleaved ? launch_one<false, true, 128>(p, n_jobs, stream) : launch_one<false, false, 128>(p, n_jobs, stream);
  }
  if (D == 64) {
    if (bf16) return interleaved ? launch_one<true, true, 64>(p, n_jobs, stream) : launch_one<true, false, 64>(p, n_jobs, stream);
    return interleaved ? launch_one<false, true, 64>(p, n_jobs, stream) : launch_one<false, false, 64>(p, n_jobs, stream);
  }
  return cudaErrorInvalidValue;
}

}  // namespace attn
