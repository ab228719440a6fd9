/*
 * fa.h -- C ABI of the GB300 (sm_103a) attention forward library.
 *
 * The operation is the exact attention forward pass described by the page
 * "FlashAttention core algorithm: forward pass" (inference.lei6393.com,
 * FlashAttention 02-core-algorithm / 03-forward-pass): for each query row the
 * consumer mainloop accumulates softmax(scale * Q K^T) V block by block over
 * K/V with a running row maximum and row sum, using exp2 with a pre-multiplied
 * softmax_scale_log2 (consumer excerpt, step 1), folds the FP8 q/k descales
 * into that scale (same excerpt, FP8 branch), and the epilogue writes O and
 * the per-row log-sum-exp, or all-zero O and -inf LSE for rows that see no
 * key (epilogue excerpt, store / store_zero).  The algorithm itself is the
 * one of "FlashAttention: Fast and Memory-Efficient Exact Attention with
 * IO-Awareness" (arXiv:2205.14135), which the page "FlashAttention SM120
 * forward reuses the SM80 mainloop" (xuesongtap.github.io) cites as its
 * background (reference [8]).
 *
 * Per query row i of head h in batch b, with visible key set V_i:
 *     O_i   = sum_{j in V_i} softmax_j(scale * q_i . k_j) v_j
 *     LSE_i = ln sum_{j in V_i} exp(scale * q_i . k_j)
 * V_i = all keys, or with causal = 1, {j : j <= i + Sk - Sq} (bottom-right
 * aligned).  V_i empty => O_i = 0 and LSE_i = -inf, never NaN.
 *
 * Conventions for every entry point:
 *  - All tensor pointers are DEVICE pointers owned by the caller, 16-byte
 *    aligned (k and v may be NULL when seqlen_k == 0: no key rows exist).
 *    The library allocates no device memory, never synchronises the stream,
 *    and keeps only host-side caches.
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default).
 *  - Every argument is validated before anything is launched; on a non-OK
 *    status nothing has been written and fa_last_error_detail() says why.
 */
#ifndef FA_GB300_H
#define FA_GB300_H

#include <stddef.h>
#include <stdint.h>

/* Only the entry points below are exported; the library is built with hidden
 * visibility, so two builds loaded into one process never bind to each other's
 * internals. */
#if defined(__GNUC__)
#define FA_API __attribute__((visibility("default")))
#else
#define FA_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FA_OK = 0,
    FA_ERR_INVALID_ARG = 1,     /* NULL/misaligned pointer, negative size, bad scale, ... */
    FA_ERR_UNSUPPORTED = 2,     /* valid but not built: head_dim not in {64,128}, ... */
    FA_ERR_CUDA = 3,            /* a CUDA runtime/driver call failed (launch, tensor map) */
    FA_ERR_WORKSPACE = 4,       /* workspace given but smaller than fa_fwd_workspace_size() */
    FA_ERR_DEVICE_TIMEOUT = 5,  /* a bounded device-side wait gave up (see fa_device_error) */
    FA_ERR_DEVICE_ARG = 6       /* a device-resident length was out of range (fa_device_error) */
} fa_status;

typedef enum {
    FA_DTYPE_BF16 = 0,          /* Q, K, V bfloat16 */
    FA_DTYPE_E4M3 = 1,          /* float8 e4m3 (OCP "fn": no infinities, max 448) */
    FA_DTYPE_E5M2 = 2           /* float8 e5m2 (OCP, max 57344): accepted for V only */
} fa_dtype;

/*
 * fa_fwd -- attention forward pass.
 *
 * Layouts (row-major, contiguous):
 *   fixed length (cu_seqlens_q == cu_seqlens_k == NULL):
 *     q [batch, seqlen_q, heads, head_dim]      k, v [batch, seqlen_k, heads, head_dim]
 *     o [batch, seqlen_q, heads, head_dim_v] bf16
 *     lse [batch, heads, seqlen_q] fp32
 *   packed variable length (both cu_seqlens given; device int32 [batch + 1],
 *   non-decreasing, cu[0] = 0):
 *     q [seqlen_q, heads, head_dim]  where seqlen_q = cu_seqlens_q[batch] (total rows)
 *     k, v [seqlen_k, heads, head_dim] where seqlen_k = cu_seqlens_k[batch]
 *     o [seqlen_q, heads, head_dim_v] bf16,  lse [heads, seqlen_q] fp32
 *     max_seqlen_q / max_seqlen_k bound every sequence's length; a sequence may
 *     have zero query rows or zero keys (its rows then get O = 0, LSE = -inf).
 * batch, heads >= 1 (batch == 0 or seqlen_q == 0: FA_OK, nothing launched).
 * head_dim == head_dim_v in {64, 128}; other values: FA_ERR_UNSUPPORTED.
 * softmax_scale: finite, > 0 (typically 1/sqrt(head_dim)).
 * causal: 0 or 1.
 * dtype FA_DTYPE_E4M3: q/k/v_descale are device fp32 scalars (NULL means 1.0);
 *   scores use softmax_scale * q_descale * k_descale and O is multiplied by
 *   v_descale.  Descale pointers must be NULL for FA_DTYPE_BF16.
 * workspace: optional device scratch for splitting long key ranges over
 *   several CTAs (short-query / long-key shapes).  NULL disables splitting.
 *   If non-NULL it must hold fa_fwd_workspace_size(batch, heads,
 *   max_seqlen_q, max_seqlen_k, head_dim_v, causal) bytes, else
 *   FA_ERR_WORKSPACE.  For varlen the longest lengths decide whether and how
 *   far the key range is split, and the partial results are laid out per
 *   sequence with max_seqlen_q rows each.
 * stream: cudaStream_t.
 */
FA_API fa_status fa_fwd(const void* q, const void* k, const void* v,
                 void* o, float* lse,
                 int batch, int heads, int seqlen_q, int seqlen_k,
                 const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                 int max_seqlen_q, int max_seqlen_k,
                 int head_dim, int head_dim_v, float softmax_scale, int causal,
                 fa_dtype dtype,
                 const float* q_descale, const float* k_descale, const float* v_descale,
                 void* workspace, size_t workspace_bytes,
                 void* stream);

/*
 * fa_fwd_gqa -- fa_fwd with grouped-query / multi-query attention: K and V have
 * heads_k heads (heads_k >= 1 dividing heads; heads_k == heads is fa_fwd) and query
 * head h attends with key/value head h / (heads / heads_k).  Layouts as fa_fwd with
 * heads_k in place of heads for k and v:
 *   fixed length  k, v [batch, seqlen_k, heads_k, head_dim]
 *   varlen        k, v [seqlen_k, heads_k, head_dim]
 * All other arguments, the outputs and the errors are those of fa_fwd (plus
 * FA_ERR_INVALID_ARG when heads_k does not divide heads).  Not on the pages: the
 * same forward pass with the K/V head index shared by a group of query heads.
 */
FA_API fa_status fa_fwd_gqa(const void* q, const void* k, const void* v,
                            void* o, float* lse,
                            int batch, int heads, int heads_k, int seqlen_q, int seqlen_k,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int max_seqlen_q, int max_seqlen_k,
                            int head_dim, int head_dim_v, float softmax_scale, int causal,
                            fa_dtype dtype,
                            const float* q_descale, const float* k_descale,
                            const float* v_descale,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * fa_fwd_fp8 -- FP8 attention with per-(batch, head) descales and an optional
 * E5M2 V.  The page "FlashAttention core algorithm: forward pass" (consumer
 * mainloop excerpt, FP8 branch) multiplies the softmax scale of a work tile by
 * q_descale * k_descale; a work tile belongs to one (batch, head), so here each
 * (batch b, key/value head g) has its own descales:
 *     q/k/v_descale[b * descale_stride_b + g * descale_stride_h]
 * (device fp32; query head h uses g = h / (heads / heads_k); strides in
 * elements, >= 0; strides 0, 0 = one value per tensor as in fa_fwd; a NULL
 * descale means 1).  Scores use softmax_scale * q_descale * k_descale and the
 * output row is multiplied by v_descale.  The arrays must hold every index the
 * strides reach for b < batch, g < heads_k (not checked: device memory).
 * q, k: E4M3.  v_dtype: FA_DTYPE_E4M3 or FA_DTYPE_E5M2 (P is rounded to E4M3
 * either way).  head_dim = head_dim_v = 128.  All else as fa_fwd_gqa, whose
 * layouts, workspace rules and errors apply.
 */
FA_API fa_status fa_fwd_fp8(const void* q, const void* k, const void* v,
                            void* o, float* lse,
                            int batch, int heads, int heads_k, int seqlen_q, int seqlen_k,
                            const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                            int max_seqlen_q, int max_seqlen_k,
                            int head_dim, float softmax_scale, int causal,
                            fa_dtype v_dtype,
                            const float* q_descale, const float* k_descale,
                            const float* v_descale,
                            int64_t descale_stride_b, int64_t descale_stride_h,
                            void* workspace, size_t workspace_bytes,
                            void* stream);

/*
 * fa_fwd_2cta -- the bf16 forward pass of fa_fwd_gqa computed by the CTA-pair
 * kernel: clusters of two CTAs on two SMs run 256-row tcgen05 MMAs
 * (cta_group::2), each CTA loading its own query rows and one half of every K/V
 * block (64 keys of K, 64 head-dim columns of V), so each SM streams half of the
 * K/V bytes through shared memory.  The page "Dissecting the SM_120
 * Microarchitecture" (section 4, feature matrix Fig. 1) lists this 2-SM
 * cooperative MMA among the SM_100-class features; the attention it computes is
 * that of fa_fwd.
 *   q, k, v, o, lse, batch, heads, heads_k, seqlen_q/k, cu_seqlens_q/k,
 *   max_seqlen_q/k, softmax_scale, causal, stream: as fa_fwd_gqa (bf16 only,
 *   head_dim = head_dim_v = 128, no workspace: no key splits).
 * Same outputs, layouts and validation as fa_fwd_gqa.  FA_ERR_UNSUPPORTED for
 * head_dim != 128, or when no cluster of two CTAs fits on the device.  The
 * work items (512 query rows of one batch and head) follow a static order,
 * also for varlen: longest first, for fixed lengths grouped by (batch, head)
 * where that keeps the CTAs' loads balanced.
 */
FA_API fa_status fa_fwd_2cta(const void* q, const void* k, const void* v,
                             void* o, float* lse,
                             int batch, int heads, int heads_k, int seqlen_q, int seqlen_k,
                             const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                             int max_seqlen_q, int max_seqlen_k,
                             int head_dim, float softmax_scale, int causal,
                             void* stream);

/*
 * fa_fwd_kvcache -- append new key/value rows to a key/value cache, then attend
 * over the cache.  The AppendKV branch of the producer loop on the page
 * "FlashAttention core algorithm: forward pass" (scheduler-loop excerpt) loads
 * the new K/V before the attention of the same work tile; here, for up to 4 new
 * rows per sequence, the attention kernel writes them into the cache itself (each
 * work tile the rows inside the key blocks it loads, before loading them); for
 * more, a copy kernel writes them first.  Both run on `stream`.
 *   q        [batch, seqlen_q, heads, head_dim]
 *   k_cache, v_cache [batch, cache_capacity, heads_k, head_dim]   (written)
 *   k_new, v_new     [batch, seqlen_new, heads_k, head_dim] or NULL (seqlen_new 0)
 *   cache_seqlens    device int32 [batch]: rows already filled in each sequence
 *                    (read only: the caller advances it by seqlen_new afterwards)
 *   o [batch, seqlen_q, heads, head_dim] bf16, lse [batch, heads, seqlen_q] fp32
 * Sequence b: rows cache_seqlens[b] .. + seqlen_new - 1 of the caches receive
 * k_new[b] / v_new[b]; then query row i attends over the first
 * L_b = cache_seqlens[b] + seqlen_new cache rows, with causal = 1 bottom-right
 * aligned (key j visible iff j <= i + L_b - seqlen_q).  L_b = 0 gives O = 0 and
 * LSE = -inf.  dtype / v_dtype / descales as fa_fwd (bf16) or fa_fwd_fp8 (FP8;
 * new rows must already be quantised with the cache's descales: bytes are copied).
 * cache_seqlens lives on the device, so it is checked there: a sequence with
 * cache_seqlens[b] < 0 or cache_seqlens[b] + seqlen_new > cache_capacity gets no
 * rows appended, its attention uses the length clamped to [0, capacity], and
 * fa_device_error() afterwards returns FA_ERR_DEVICE_ARG.  workspace: partial
 * results of key splits, sized by fa_fwd_kvcache_workspace_size below; NULL means
 * one CTA per work item.
 */
FA_API fa_status fa_fwd_kvcache(const void* q, void* k_cache, void* v_cache,
                                const void* k_new, const void* v_new,
                                void* o, float* lse,
                                int batch, int heads, int heads_k, int seqlen_q,
                                int cache_capacity, const int32_t* cache_seqlens,
                                int seqlen_new,
                                int head_dim, float softmax_scale, int causal,
                                fa_dtype dtype, fa_dtype v_dtype,
                                const float* q_descale, const float* k_descale,
                                const float* v_descale,
                                int64_t descale_stride_b, int64_t descale_stride_h,
                                void* workspace, size_t workspace_bytes,
                                void* stream);

/*
 * Bytes of workspace that fa_fwd would use to split the key range of a problem
 * of this shape on the current device (0 = it would not split): a fixed-length
 * problem, or a packed varlen batch whose longest sequences have lengths
 * seqlen_q / seqlen_k (max_seqlen_q / max_seqlen_k).  Splitting follows the
 * log-sum-exp merge identity: each split writes a normalised partial O and its
 * LSE, a second kernel merges them.  `causal` is accepted for the split rule;
 * the current rule does not depend on it.
 */
FA_API size_t fa_fwd_workspace_size(int batch, int heads, int seqlen_q, int seqlen_k,
                             int head_dim_v, int causal);

/* Number of key splits fa_fwd would use for that shape with a workspace. */
FA_API int fa_fwd_num_splits(int batch, int heads, int seqlen_q, int seqlen_k, int causal);

/*
 * The same two queries for grouped-query shapes (heads_k K/V heads; fa_fwd_gqa,
 * fa_fwd_fp8, fa_fwd_kvcache with cache_capacity as seqlen_k).  When a whole group of
 * short query blocks fits one 256-row tile pair (heads / heads_k a power of two
 * <= 128 and seqlen_q * heads / heads_k <= 256, fixed length), the query heads of a
 * group share tiles, so fewer work items exist and more key splits may be used; the
 * MHA queries above then under-size the workspace (FA_ERR_WORKSPACE).
 */
FA_API size_t fa_fwd_workspace_size_gqa(int batch, int heads, int heads_k, int seqlen_q,
                                        int seqlen_k, int head_dim_v, int causal);
FA_API int fa_fwd_num_splits_gqa(int batch, int heads, int heads_k, int seqlen_q, int seqlen_k,
                                 int causal);

/*
 * The same two queries for fa_fwd_kvcache.  Cache lengths differ per sequence and are
 * known only on the device.  Where the fixed-length rule would not split and the work
 * items are few (under two waves), long (>= 8 key blocks of capacity) and see all
 * their keys (non-causal, or one query row), with batch <= 64, a cache call is
 * balanced instead: every CTA takes an equal share of the key blocks of all items,
 * computed on the device from cache_seqlens, and each item's pieces (at most 4) are
 * merged by the LSE identity.  These queries return that plan's needs; a smaller
 * workspace gives FA_ERR_WORKSPACE, none gives one CTA per item.
 */
FA_API size_t fa_fwd_kvcache_workspace_size(int batch, int heads, int heads_k, int seqlen_q,
                                            int cache_capacity, int head_dim, int causal);
FA_API int fa_fwd_kvcache_num_splits(int batch, int heads, int heads_k, int seqlen_q,
                                     int cache_capacity, int causal);

/*
 * fa_fwd_static_workspace -- fa_fwd for fixed-length inputs, for callers that
 * cannot allocate device memory: code embedded in a host program that owns
 * all device memory and gives out no scratch (plugins, for instance), or
 * latency-critical loops where cudaMalloc/cudaFree would synchronise the
 * device.  The paper has no counterpart: this is a packaging of the split
 * path above, not a step of the method.
 *
 * Arguments are those of fa_fwd without cu_seqlens and without workspace.
 * When the shape splits its key range, the partial results go to a 16 MiB
 * array that the library holds in device memory (reserved on every GPU that
 * loads the library, until the process exits).  Shapes needing more return
 * FA_ERR_WORKSPACE and launch nothing.  All calls on a device share that
 * array: calls whose kernels overlap on the GPU race and corrupt each other;
 * nothing in it needs to start at zero.  The first call on a device looks up
 * the array's device address, so make it before any stream capture.  This
 * entry point itself allocates nothing.
 */
FA_API fa_status fa_fwd_static_workspace(const void* q, const void* k, const void* v,
                                  void* o, float* lse,
                                  int batch, int heads, int seqlen_q, int seqlen_k,
                                  int head_dim, int head_dim_v, float softmax_scale, int causal,
                                  fa_dtype dtype,
                                  const float* q_descale, const float* k_descale,
                                  const float* v_descale,
                                  void* stream);

/* Static description of a status code. */
FA_API const char* fa_status_string(fa_status status);

/* Thread-local message describing the last non-OK status of this thread. */
FA_API const char* fa_last_error_detail(void);

/*
 * Device-side failure detection.  Every wait inside the kernels is bounded
 * (by wall clock, default 4 s).  A wait that runs out sets a bit in a
 * device-resident error word, the kernel's CTAs abandon their work and exit
 * cleanly (TMEM released), and the context stays usable.
 * fa_device_error synchronises the current device, copies the word to
 * *flags (bit 0: a wait timed out; bit 1: a device-resident cache length was
 * out of range; bits 8..15: the site of the first timeout) and, if clear != 0,
 * resets it.  Returns FA_ERR_DEVICE_TIMEOUT if a timeout bit was set, else
 * FA_ERR_DEVICE_ARG if the length bit was set, FA_OK otherwise (FA_ERR_CUDA on
 * a CUDA failure).
 */
FA_API fa_status fa_device_error(uint32_t* flags, int clear);

/*
 * Debug controls for the failure-detection tests (process-wide, host side,
 * applied to subsequent launches).  wait_limit_ns = 0 restores the default.
 * inject: 0 = none; 1 = the TMA producer withholds the first Q-tile arrival
 * of each CTA, so the MMA issuer's bounded wait runs out (no GPU fault).
 */
FA_API void fa_debug_set(uint64_t wait_limit_ns, uint32_t inject);

/*
 * Debug: which kernel instance bf16 head_dim-128 launches without a key/value cache
 * use (process-wide, host side, applied to subsequent launches).  Those launches
 * (fixed-length or packed varlen) have two instances with identical results: one for
 * short launches and one whose MMA issuer runs the middle key blocks of a work item
 * without per-block tests, which the library picks once a launch holds at least 128
 * (query tile, key block) steps per CTA (varlen: counted from the longest sequence).  mode: 0 = by that size (the default),
 * 1 = always the steady-block instance, -1 = never.  Other values: as 0.  For
 * tests that exercise both instances on small shapes.
 */
FA_API void fa_debug_select_steady(int mode);

/*
 * Debug: event trace of the forward kernel, for a library built with -DFA_TRACE
 * (a variant build; the default library returns FA_ERR_UNSUPPORTED and its kernel
 * holds no trace code).  buf: device memory of at least fa_debug_trace_bytes()
 * bytes, 16-byte aligned, owned by the caller (NULL stops tracing); later launches
 * make 8 CTAs spread over the grid (slot k: CTA k * (grid - 1) / 7) log up to 8192
 * events per role into it: word (slot * 4 + role) * 8192 + i = tag << 56 | clock64
 * (low 56 bits), roles 0 the TMA producer, 1 the MMA issuer, 2 and 3 the softmax
 * warps of query tiles 0 and 1 (tags: see the kernel header).  Unwritten words keep
 * what the caller put there.
 */
FA_API fa_status fa_debug_trace(void* buf, size_t bytes);
FA_API size_t fa_debug_trace_bytes(void);

#ifdef __cplusplus
}
#endif

#endif /* FA_GB300_H */
