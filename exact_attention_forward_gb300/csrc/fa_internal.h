// fa_internal.h -- types shared by the host launcher and the kernel
// translation units (never exported; the public ABI is include/fa.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Everything a forward launch needs besides the three TMA tensor maps.
struct FwdParams {
    void* o;                    // bf16 output (or unused in split mode)
    float* lse;                 // fp32 LSE (or unused in split mode)
    const int32_t* cu_q;        // varlen offsets (device) or nullptr
    const int32_t* cu_k;
    const float* q_descale;     // FP8 only, device scalars or nullptr (= 1)
    const float* k_descale;
    const float* v_descale;
    float* ws_o;                // split mode: normalised partial O [splits, B, H, Sq, Dv] fp32
    float* ws_lse;              // split mode: partial LSE [splits, B, H, Sq] fp32
    uint32_t* err;              // device error word
    int batch, heads;
    int kv_group;               // query heads per K/V head (grouped-query attention; 1 = MHA)
    int seqlen_q, seqlen_k;     // fixed length: the lengths; varlen: max lengths
    int total_q;                // varlen: packed rows of Q (LSE row stride)
    int n_mpairs;               // ceil(seqlen_q / 256): query-row pairs of tiles
    int n_splits;               // key-range splits (1 = none)
    int blocks_per_split;       // key blocks per split
    int n_items;                // n_mpairs * batch * heads * n_splits
    float scale_log2;           // softmax_scale * log2(e)
    int causal, varlen, split;
    uint64_t wait_limit_ns;     // bound of every device-side wait
    uint32_t inject;            // debug fault injection (see fa_debug_set)
};

enum : uint32_t { kErrTimeout = 1u };

// Kernel instances (one translation unit each).
cudaError_t launch_fwd_bf16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const FwdParams& p, int grid, cudaStream_t s);
cudaError_t launch_fwd_bf16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const FwdParams& p, int grid, cudaStream_t s);
cudaError_t launch_fwd_e4m3_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const FwdParams& p, int grid, cudaStream_t s);
cudaError_t launch_combine(const float* ws_o, const float* ws_lse, void* o, float* lse,
                           int batch, int heads, int seqlen_q, int dv, int n_splits,
                           cudaStream_t s);
uint32_t* device_error_word();  // address of the device error word (current device)

}  // namespace fa
