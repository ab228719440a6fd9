// Kernel instance: attention forward, bf16_d128, CTA-pair variant (cta_group::2 MMAs
// over 256-row slots; see fa_fwd_kernel.cuh).
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_pair_bf16_d128(const CUtensorMap& q, const CUtensorMap& k,
                                      const CUtensorMap& v, const CUtensorMap& o,
                                      const FwdParams& p, int grid, cudaStream_t s) {
    return launch_fwd<128, false, true>(q, k, v, o, p, grid, s, false);
}
cudaError_t max_resident_pairs_bf16_d128(int* pairs) { return max_resident_pairs<128, false>(pairs); }
}  // namespace fa
