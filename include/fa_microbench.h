/*
 * fa_microbench.h -- C ABI of the throughput probes (_fa_microbench.so) that
 * measure the two ceilings of the attention forward kernel on this GPU: the
 * MUFU exponential rate and the tcgen05 tensor-pipe rate.
 *
 * A third probe measures how fast shared memory is fed from L2 (and HBM) by
 * bulk copies, the path every K/V block of the forward kernel takes.
 *
 * Why: the page "Dissecting the SM_120 Microarchitecture" (section 11.2,
 * Fig. 12) finds exp2 on the special-function unit, not the MMAs, to dominate
 * a key block of fused attention on a GPU without Tensor Memory.  A forward
 * pass computes one exp2 per visible (query row, key) pair and
 * 4 * head_dim FLOPs per pair, so its attainable time is the larger of the
 * two quotients; these probes supply both denominators, measured.
 *
 * All pointers are device pointers owned by the caller; all launches are
 * asynchronous on `stream` (a cudaStream_t).  Every wait inside a kernel is
 * bounded (limit_ns of %globaltimer); a wait that runs out sets *err != 0.
 * The return value is a cudaError_t (0 = launched).
 */
#ifndef FA_MICROBENCH_H
#define FA_MICROBENCH_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define FA_MB_API __attribute__((visibility("default")))
#else
#define FA_MB_API
#endif

/*
 * ex2.approx.ftz.f32 throughput.  `grid` CTAs of 1024 threads (one per SM),
 * each thread `iters` x 32 exponentials in 8 independent chains.  Writes the
 * SM cycles of each CTA to cycles[grid] (uint64); sink[1024] is never written
 * in practice (it keeps the chains from being optimised away).
 */
FA_MB_API int fa_mb_ex2(int grid, int iters, unsigned long long* cycles, float* sink,
                        void* stream);
/* exponentials one CTA of fa_mb_ex2 evaluates */
FA_MB_API long long fa_mb_ex2_per_cta(int iters);
/*
 * The same for ex2.approx.f16x2 (two fp16 exponentials per instruction): the CTAs
 * evaluate 2 x fa_mb_ex2_per_cta(iters) exponentials in as many instructions as
 * fa_mb_ex2.
 */
FA_MB_API int fa_mb_ex2_f16x2(int grid, int iters, unsigned long long* cycles, float* sink,
                              void* stream);

/*
 * tcgen05.mma issue rate.  `grid` CTAs (one per SM); in each one thread
 * issues 4 x `iters` MMAs of M = 128, N = n (64, 128 or 256 for bf16; 128 or
 * 256 for e4m3) and K = 16 (bf16, kind::f16) or 32 (e4m3, kind::f8f6f4), A and
 * B K-major from shared memory, fp32 accumulate in Tensor Memory, then waits
 * for their completion.  n = -128: N = 128 with A read from Tensor Memory and
 * B MN-major in shared memory (the form of the P V product).  Writes each
 * CTA's SM cycles to cycles[grid].
 */
FA_MB_API int fa_mb_mma(int grid, int n, int fp8, int iters, unsigned long long* cycles,
                        uint32_t* err, unsigned long long limit_ns, void* stream);
/* FLOPs one CTA of fa_mb_mma performs (2 * M * N * K per MMA) */
FA_MB_API long long fa_mb_mma_flops_per_cta(int n, int fp8, int iters);

/*
 * Bulk-copy (cp.async.bulk) throughput into shared memory.  `grid` CTAs; in each one
 * thread keeps four 32 KiB copies in flight, `iters` copies in all, each from the CTA's
 * own window of `window` bytes at src + cta * window (read cyclically; window a multiple
 * of 32 KiB, src 16-byte aligned, grid * window bytes readable).  A window set that fits
 * L2, read once beforehand, measures the L2 -> shared-memory rate; a larger one the HBM
 * read rate.  Writes each CTA's SM cycles to cycles[grid].
 */
FA_MB_API int fa_mb_load(int grid, const void* src, unsigned long long window, int iters,
                         unsigned long long* cycles, uint32_t* err, unsigned long long limit_ns,
                         void* stream);
/* bytes one CTA of fa_mb_load copies */
FA_MB_API long long fa_mb_load_bytes_per_cta(int iters);

/*
 * The tensor pipe and the bulk-copy engine sharing shared memory: in each of `grid` CTAs
 * one thread issues 4 x `iters` bf16 MMAs (M = N = 128, K = 16, A and B K-major in
 * shared memory: the QK^T form) while another keeps two 32 KiB bulk copies in flight from
 * the CTA's own window (as fa_mb_load) until the MMAs complete.  Writes each CTA's MMA
 * cycles to cycles[grid] and the bytes copied meanwhile to bytes[grid] (uint64).
 */
FA_MB_API int fa_mb_mma_with_load(int grid, const void* src, unsigned long long window, int iters,
                                  unsigned long long* cycles, unsigned long long* bytes,
                                  uint32_t* err, unsigned long long limit_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* FA_MICROBENCH_H */
