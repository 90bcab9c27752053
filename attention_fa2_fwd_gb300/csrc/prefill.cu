// prefill.cu -- the prefill kernel without sliding windows, ALiBi or rotary
// embeddings (plain causal or full attention), and the entry that routes the
// other variants to their own translation units (prefill_masked.cu,
// prefill_rope.cu, prefill_rope_masked.cu).  The kernel itself is in
// prefill_kernel.cuh.
#include "prefill_kernel.cuh"

namespace attn {

cudaError_t launch_prefill(int D, bool causal, bool bf16, bool varlen, bool masked, bool rope, const CUtensorMap &tq,
                           const CUtensorMap &tk, const CUtensorMap &tv, const PrefillParams &p, int B,
                           cudaStream_t stream) {
  if (rope) {
    return masked ? launch_prefill_rope_masked(D, causal, bf16, varlen, tq, tk, tv, p, B, stream)
                  : launch_prefill_rope(D, causal, bf16, varlen, tq, tk, tv, p, B, stream);
  }
  if (masked) return launch_prefill_masked(D, causal, bf16, varlen, tq, tk, tv, p, B, stream);
  return launch_prefill_variant<false, false>(D, causal, bf16, varlen, tq, tk, tv, p, B, stream);
}

}  // namespace attn
