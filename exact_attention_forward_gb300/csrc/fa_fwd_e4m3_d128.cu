// Kernel instance: attention forward, e4m3_d128 (see fa_fwd_kernel.cuh).
#include "fa_fwd_kernel.cuh"

namespace fa {
cudaError_t launch_fwd_e4m3_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                          const CUtensorMap& o,
                          const FwdParams& p, int grid, cudaStream_t s, bool after_append,
                          bool cache, bool var) {
    if (cache) return launch_fwd<128, true, false, true, true>(q, k, v, o, p, grid, s, after_append);
    return var ? launch_fwd<128, true, false, false, true>(q, k, v, o, p, grid, s, after_append)
               : launch_fwd<128, true, false, false, false>(q, k, v, o, p, grid, s, after_append);
}
}  // namespace fa
