// bwd.cu -- the backward kernels without windows, ALiBi or key ranges (plain
// causal or full attention), and the entry that routes the masked backward to
// bwd_masked.cu.  The kernels are in bwd_kernel.cuh.
#include "bwd_kernel.cuh"

namespace attn {

cudaError_t launch_bwd(int D, bool causal, bool bf16, bool masked, const BwdMaps &m, const BwdParams &p, int B,
                       int Hkv, cudaStream_t stream, cudaStream_t side) {
  if (masked) return launch_bwd_masked(D, causal, bf16, m, p, B, Hkv, stream, side);
  return launch_bwd_variant<false>(D, causal, bf16, m, p, B, Hkv, stream, side);
}

}  // namespace attn
