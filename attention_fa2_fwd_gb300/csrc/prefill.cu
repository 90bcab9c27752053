// prefill.cu -- the prefill kernel without sliding windows or ALiBi (plain
// causal or full attention), and the entry that routes masked calls to
// prefill_masked.cu.  The kernel itself is in prefill_kernel.cuh.
#include "prefill_kernel.cuh"

namespace attn {

cudaError_t launch_prefill(int D, bool causal, bool bf16, bool varlen, bool masked, const CUtensorMap &tq,
                           const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p, int B,
                           cudaStream_t stream) {
  if (masked) return launch_prefill_masked(D, causal, bf16, varlen, tq, tk, tv, p, B, stream);
  return launch_prefill_variant<false>(D, causal, bf16, varlen, tq, tk, tv, p, B, stream);
}

}  // namespace attn
