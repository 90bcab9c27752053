// bwd_masked.cu -- the backward kernels with sliding windows, ALiBi and
// per-row key ranges (the MASKED build of bwd_kernel.cuh).
#include "bwd_kernel.cuh"

namespace attn {

cudaError_t launch_bwd_masked(int D, bool causal, bool bf16, const BwdMaps &m, const BwdParams &p, int B, int Hkv,
                              cudaStream_t stream, cudaStream_t side) {
  return launch_bwd_variant<true>(D, causal, bf16, m, p, B, Hkv, stream, side);
}

}  // namespace attn
