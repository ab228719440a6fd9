// fa_append_kv.cu -- writes new key/value rows into a fixed-capacity cache before
// the attention reads it: the "load the new K/V first" step of the AppendKV branch
// in the producer loop of the page "FlashAttention core algorithm: forward pass"
// (scheduler-loop excerpt).  A pure copy, bound by HBM bandwidth: every byte of
// the new rows is read once and written once.
#include <cstdint>

#include "fa_internal.h"

namespace fa {

// One warp per (tensor, sequence b, new row i): the row holds heads_k * head_dim
// elements, contiguous in both layouts ([B, n_new, Hk, D] -> [B, capacity, Hk, D]),
// copied with 16-byte vectors.  A sequence whose filled length leaves no room
// (len < 0 or len + n_new > capacity) is not written; the device error word records it.
__global__ void __launch_bounds__(256) fa_append_kv_kernel(uint4* __restrict__ k_cache,
                                                           uint4* __restrict__ v_cache,
                                                           const uint4* __restrict__ k_new,
                                                           const uint4* __restrict__ v_new,
                                                           const int32_t* __restrict__ lens,
                                                           int batch, int capacity, int n_new,
                                                           int vecs_per_row, uint32_t* err) {
    // the attention grid behind this one may start its set-up now; it waits for this
    // grid's completion before reading the cache
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const long long warp = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const long long rows = (long long)batch * n_new;
    if (warp >= 2 * rows) return;
    const bool is_v = warp >= rows;
    const long long r = is_v ? warp - rows : warp;
    const int b = (int)(r / n_new);
    const int i = (int)(r % n_new);
    const int len = __ldg(lens + b);
    if (len < 0 || len > capacity - n_new) {
        if (lane == 0 && i == 0 && !is_v) atomicOr(err, kErrBadLength);
        return;
    }
    const uint4* src = (is_v ? v_new : k_new) + r * vecs_per_row;
    uint4* dst = (is_v ? v_cache : k_cache) + ((long long)b * capacity + len + i) * vecs_per_row;
    for (int c = lane; c < vecs_per_row; c += 32) dst[c] = __ldg(src + c);
}

cudaError_t launch_append_kv(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                             const int32_t* cache_seqlens, int batch, int capacity, int n_new,
                             long long row_bytes, uint32_t* err, cudaStream_t s) {
    const long long warps = 2ll * batch * n_new;
    const int threads = 256;
    const long long blocks = (warps * 32 + threads - 1) / threads;
    fa_append_kv_kernel<<<(unsigned)blocks, threads, 0, s>>>(
        static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), static_cast<const uint4*>(k_new),
        static_cast<const uint4*>(v_new), cache_seqlens, batch, capacity, n_new,
        (int)(row_bytes / 16), err);
    return cudaGetLastError();
}

}  // namespace fa
