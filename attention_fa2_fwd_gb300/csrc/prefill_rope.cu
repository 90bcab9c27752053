// prefill_rope.cu -- the prefill kernel with rotary position embeddings on the
// Q and K tiles (kernel in prefill_kernel.cuh, instantiated here with ROPE).
#include "prefill_kernel.cuh"

namespace attn {

cudaError_t launch_prefill_rope(int D, bool causal, bool bf16, bool varlen, const CUtensorMap &tq,
                                const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p, int B,
                                cudaStream_t stream) {
  return launch_prefill_variant<false, true>(D, causal, bf16, varlen, tq, tk, tv, p, B, stream);
}

}  // namespace attn
