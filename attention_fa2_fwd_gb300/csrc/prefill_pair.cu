// prefill_pair.cu -- the CTA-pair prefill kernel (head dimension 128, plain
// causal or full attention); the kernel is in prefill_pair_kernel.cuh.
#include "prefill_pair_kernel.cuh"

namespace attn {

cudaError_t launch_prefill_pair(bool causal, bool bf16, const CUtensorMap &tq, const CUtensorMap &tk_half,
                                const CUtensorMap &tv, const PrefillParams &p, cudaStream_t stream) {
  if (causal) {
    return bf16 ? pair_launch_one<true, true>(tq, tk_half, tv, p, stream)
                : pair_launch_one<true, false>(tq, tk_half, tv, p, stream);
  }
  return bf16 ? pair_launch_one<false, true>(tq, tk_half, tv, p, stream)
              : pair_launch_one<false, false>(tq, tk_half, tv, p, stream);
}

int prefill_pair_max_clusters() {
  // Every build has the same shared memory and threads, so one answers for all.
  return pair_clusters_one<true, true>();
}

}  // namespace attn
