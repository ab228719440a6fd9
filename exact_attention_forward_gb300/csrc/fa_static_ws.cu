// fa_static_ws.cu -- fa_fwd_static_workspace: the forward pass with its
// split-KV scratch taken from a fixed array that the library owns, for callers
// that cannot allocate device memory themselves.
//
// Who needs it: code embedded in a host program that owns all device memory
// and offers no way to ask for scratch (plugins, for instance), and latency-
// critical loops where a cudaMalloc / cudaFree would synchronise the device.
// Such callers pass inputs and outputs as usual; the partial results of the
// key splits go to `g_fa_static_scratch` below instead of a caller workspace.
//
// Limits and sharing rules:
//  * the array holds kStaticScratchBytes (16 MiB).  Every GPU that loads this
//    library keeps that much device memory reserved until the process exits.
//  * shapes whose split scratch would exceed it are rejected with
//    FA_ERR_WORKSPACE before anything is launched (fa_last_error_detail names
//    both sizes);
//  * all calls on a device share the one array, which keeps whatever the last
//    call left in it.  Nothing in it has to start at zero: every split writes
//    each partial row it owns before the merge kernel reads it.  Calls whose
//    kernels overlap on the GPU (e.g. from two streams at once) race on the
//    array and corrupt each other's results; serialise them.
//  * the first call on a device looks up the array's device address
//    (cudaGetSymbolAddress, with that device current); make that first call
//    before any stream capture.  The address belongs to the device's current
//    context: after a cudaDeviceReset the next call looks it up again (also
//    before any capture).
// No cudaMalloc, cudaFree or allocating library routine is called here.
#include <mutex>

#include "fa.h"
#include "fa_internal.h"

namespace {

constexpr size_t kStaticScratchBytes = 16u << 20;  // 16 MiB
constexpr int kMaxDevices = 64;

// The scratch itself.  In host code this name is only a host-side stand-in for
// the device array: its device address comes from cudaGetSymbolAddress.
static __device__ __align__(256) unsigned char g_fa_static_scratch[kStaticScratchBytes];

std::mutex g_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};
unsigned long long g_scratch_ctx[kMaxDevices] = {0};  // context the address was looked up in

}  // namespace

extern "C" fa_status fa_fwd_static_workspace(
    const void* q, const void* k, const void* v, void* o, float* lse, int batch, int heads,
    int seqlen_q, int seqlen_k, int head_dim, int head_dim_v, float softmax_scale, int causal,
    fa_dtype dtype, const float* q_descale, const float* k_descale, const float* v_descale,
    void* stream) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices)
        return fa::set_error_detail(FA_ERR_CUDA, "no usable current CUDA device");
    void* scratch = nullptr;
    {
        const unsigned long long ctx = fa::current_context_id();
        std::lock_guard<std::mutex> lk(g_mu);
        if (!g_scratch_addr[dev] || ctx == 0 || ctx != g_scratch_ctx[dev]) {
            void* addr = nullptr;
            cudaError_t e = cudaGetSymbolAddress(&addr, g_fa_static_scratch);
            if (e != cudaSuccess || addr == nullptr)
                return fa::set_error_detail(FA_ERR_CUDA,
                                            "device address of the static scratch unavailable");
            g_scratch_addr[dev] = addr;
            g_scratch_ctx[dev] = fa::current_context_id();
        }
        scratch = g_scratch_addr[dev];
    }
    // fa_fwd validates everything, including that the split scratch this shape
    // needs fits in kStaticScratchBytes (FA_ERR_WORKSPACE otherwise).
    return fa_fwd(q, k, v, o, lse, batch, heads, seqlen_q, seqlen_k, nullptr, nullptr, seqlen_q,
                  seqlen_k, head_dim, head_dim_v, softmax_scale, causal, dtype, q_descale,
                  k_descale, v_descale, scratch, kStaticScratchBytes, stream);
}
