// Kernel instance: attention forward, bf16_d128 (see fa_fwd_kernel.cuh).
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_bf16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o,
                          const FwdParams& p, int grid, cudaStream_t s, bool after_append,
                          bool cache, bool var, bool steady) {
    if (cache) return launch_fwd<128, false, false, true, true>(q, k, v, o, p, grid, s, after_append);
    if (var)
        return steady ? launch_fwd<128, false, false, false, true, true>(q, k, v, o, p, grid, s, after_append)
                      : launch_fwd<128, false, false, false, true>(q, k, v, o, p, grid, s, after_append);
    return steady ? launch_fwd<128, false, false, false, false, true>(q, k, v, o, p, grid, s, after_append)
                  : launch_fwd<128, false, false, false, false>(q, k, v, o, p, grid, s, after_append);
}
}  // namespace fa
