// fa_internal.h -- types shared by the host launcher and the kernel
// translation units (never exported; the public ABI is include/fa.h).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "fa.h"

namespace fa {

// Everything a forward launch needs besides the three TMA tensor maps.
struct FwdParams {
    void* o;                    // bf16 output (or unused in split mode)
    float* lse;                 // fp32 LSE (or unused in split mode)
    const int32_t* cu_q;        // varlen offsets (device) or nullptr
    const int32_t* cu_k;
    const float* q_descale;     // FP8 only, device arrays or nullptr (= 1); the descale of
    const float* k_descale;     //   (batch b, query head h) is at b * descale_sb +
    const float* v_descale;     //   (h / kv_group) * descale_sh (0, 0: one value per tensor)
    long long descale_sb, descale_sh;
    const int32_t* seqused_k;   // fixed length: keys of sequence b = seqused_k[b] + seqused_add
    int seqused_add;            //   (nullptr: seqlen_k); lengths outside [0, seqlen_k] are clamped
                                //   and flagged in the device error word
    void* k_cache;              // key/value cache calls with few new rows: the producers write
    void* v_cache;              //   k_new / v_new ([B, append_rows, Hk, D]) into the caches at
    const void* k_new;          //   the filled length, each the rows inside the key blocks it
    const void* v_new;          //   loads, just before loading them (0 rows: none here)
    int append_rows;
    float* ws_o;                // split mode: normalised partial O [splits, B, H, Sq, Dv] fp32
    float* ws_lse;              // split mode: partial LSE [splits, B, H, Sq] fp32
    uint32_t* err;              // device error word
    uint32_t* sched;            // work counter pair {next item - grid, CTAs done}, zero at launch
    int batch, heads;
    int kv_group;               // query heads per K/V head (grouped-query attention; 1 = MHA)
    int pack;                   // > 1: the kv_group query heads of a K/V head share tiles
                                //   (rows = query row x head); 1: one head per tile
    int pack_shift;             // log2(pack) (pack is a power of two)
    int item_heads;             // heads the items run over: heads, or heads / pack
    int seqlen_q, seqlen_k;     // fixed length: the lengths; varlen: max lengths
    int total_q;                // varlen: packed rows of Q (LSE row stride)
    int n_mpairs;               // ceil(seqlen_q * pack / 256) (packed) row pairs of tiles;
                                //   CTA pairs: ceil(seqlen_q / 512) groups of four tiles
    int n_splits;               // key-range splits (1 = none)
    int blocks_per_split;       // key blocks per split
    int n_items;                // n_mpairs * batch * item_heads * n_splits
    int band_levels;            // static order: the first band_items items run in bands of
    int band_items;             //   band_levels consecutive pair levels per (batch, head), so
    int band_lv;                //   CTAs running at the same time share K/V in L2; band_lv =
                                //   banded levels (band_items / items per level); 0: none
    int half_from;              // static order, one CTA per tile pair: items from this index
                                //   on are single query tiles, two per tile pair (index
                                //   half_from + 2i + t: tile t of pair item half_from + i), so
                                //   a part-filled last round spreads over more CTAs; n_items
                                //   counts them; 0: none
    float scale_log2;           // softmax_scale * log2(e)
    int causal, varlen, split;
    int greedy;                 // items handed out by the device counter (varlen) or a static snake
    int stream;                 // cache launches: balanced plan -- each CTA takes an equal share
                                //   of all items' key blocks (pieces in n_splits partial slots)
    int v_e5m2;                 // FP8: V stored as E5M2 (Q, K and P stay E4M3)
    uint64_t wait_limit_ns;     // bound of every device-side wait
    uint32_t inject;            // debug fault injection (see fa_debug_set)
    uint64_t* trace;            // event log of a build with FA_TRACE (see fa_debug_trace), or null
};

enum : uint32_t { kErrTimeout = 1u, kErrBadLength = 2u };

// Event trace of a build with -DFA_TRACE: kTraceCtas CTAs log up to kTraceCap events per
// role (kTraceRoles roles) as 64-bit words (fa_debug_trace).
constexpr int kTraceCtas = 8;
constexpr int kTraceRoles = 4;
constexpr int kTraceCap = 8192;
constexpr size_t kTraceBytes = (size_t)kTraceCtas * kTraceRoles * kTraceCap * sizeof(uint64_t);

// Kernel instances (one translation unit each).
// q, k, v: TMA load maps; o: TMA store map of the bf16 output (same 4-D view as q);
// after_append: launched right behind the cache-append kernel on the same stream;
// cache: a key/value-cache call (p.seqused_k set): the instance that holds the cache code;
// var: otherwise, a call with packed variable-length batches or debug injection (false: the
// fixed-length instance, which leaves that code out)
cudaError_t launch_fwd_bf16_d64(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                const CUtensorMap& o, const FwdParams& p, int grid, cudaStream_t s,
                                bool after_append, bool cache, bool var);
// steady (bf16 D = 128 only): the instance specialised for long launches (fixed length or varlen)
cudaError_t launch_fwd_bf16_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& o, const FwdParams& p, int grid, cudaStream_t s,
                                bool after_append, bool cache, bool var, bool steady);
cudaError_t launch_fwd_e4m3_d128(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                                 const CUtensorMap& o, const FwdParams& p, int grid, cudaStream_t s,
                                bool after_append, bool cache, bool var);
// CTA-pair variant (bf16, D = 128; no packing, splits or cache lengths): grid = 2 x pairs,
// launched as clusters of two; k is a map with 64-row boxes (half a key block)
cudaError_t launch_fwd_pair_bf16_d128(const CUtensorMap& q, const CUtensorMap& k,
                                      const CUtensorMap& v, const CUtensorMap& o,
                                      const FwdParams& p, int grid, cudaStream_t s);
cudaError_t max_resident_pairs_bf16_d128(int* pairs);
cudaError_t launch_append_kv(void* k_cache, void* v_cache, const void* k_new, const void* v_new,
                             const int32_t* cache_seqlens, int batch, int capacity, int n_new,
                             long long row_bytes, uint32_t* err, cudaStream_t s);
// (cu_q: packed varlen offsets on the device, or nullptr; total_q: packed query rows)
cudaError_t launch_combine(const float* ws_o, const float* ws_lse, void* o, float* lse,
                           int batch, int heads, int seqlen_q, int dv, int n_splits,
                           const int32_t* cu_q, int total_q, cudaStream_t s);
// Records `msg` as this thread's fa_last_error_detail() and returns `status` (for entry
// points outside fa_api.cu).
fa_status set_error_detail(fa_status status, const char* msg);
// Unique id (cuCtxGetId) of the calling thread's current CUDA context, 0 if none.  Device
// addresses of __device__ variables and per-function attributes belong to one context;
// state cached per device is keyed on this so that a new context (after cudaDeviceReset)
// sets it up again.
unsigned long long current_context_id();

}  // namespace fa
