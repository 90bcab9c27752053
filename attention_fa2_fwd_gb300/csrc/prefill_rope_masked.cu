// prefill_rope_masked.cu -- the prefill kernel with rotary position embeddings
// together with sliding windows or ALiBi biases (kernel in prefill_kernel.cuh,
// instantiated here with MASKED and ROPE).
#include "prefill_kernel.cuh"

namespace attn {

cudaError_t launch_prefill_rope_masked(int D, bool causal, bool bf16, bool varlen, const CUtensorMap &tq,
                                       const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p, int B,
                                       cudaStream_t stream) {
  return launch_prefill_variant<true, true>(D, causal, bf16, varlen, tq, tk, tv, p, B, stream);
}

}  // namespace attn
