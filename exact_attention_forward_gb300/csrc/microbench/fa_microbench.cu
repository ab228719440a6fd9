// fa_microbench.cu -- throughput probes of the two units that bound the attention
// forward kernel on this GPU, built as a library of its own (_fa_microbench.so):
//
//  * the MUFU exponential: ex2.approx.ftz.f32 issued by every thread of one
//    1024-thread CTA per SM, eight independent dependency chains per thread, so the
//    unit's issue rate (not its latency) sets the time.  Result: ex2 per SM clock.
//  * the tensor pipe: one thread per SM issuing tcgen05.mma (cta_group::1, A and B
//    from 128-byte-swizzled shared memory, fp32 accumulator in Tensor Memory) back to
//    back, M = 128 and N = 64 / 128 / 256 with bf16 (kind::f16, K = 16 per MMA) or
//    e4m3 (kind::f8f6f4, K = 32), one commit at the end.  Result: FLOP per SM clock.
//
// Each CTA times itself with clock64 (SM cycles), so the rates do not depend on the
// clock the GPU happens to run at.  Why they matter: the page "Dissecting the SM_120
// Microarchitecture" (section 11.2, Fig. 12) finds the softmax's exponentials, not the
// MMAs, to dominate a key block of fused attention on a GPU without Tensor Memory; the
// attainable time of a forward pass is the larger of (exponentials / ex2 rate) and
// (FLOPs / tensor rate), and both rates are measured here rather than assumed.
//
// Every wait is bounded by %globaltimer; a wait that runs out sets *err and the CTA
// still waits (bounded again) for its MMAs before freeing Tensor Memory.
#include <cuda_bf16.h>
#include <cstdint>

#include "fa_microbench.h"
#include "../sm103_ptx.cuh"

namespace {

using namespace fa;

constexpr int kEx2Threads = 1024;
constexpr int kEx2Chains = 8;

__global__ void __launch_bounds__(kEx2Threads, 1)
    mb_ex2_kernel(int iters, unsigned long long* cycles, float* sink) {
    float x[kEx2Chains];
#pragma unroll
    for (int u = 0; u < kEx2Chains; ++u) x[u] = 0.25f + 0.01f * (float)((threadIdx.x + u) & 31);
    __syncthreads();
    const unsigned long long t0 = clock64();
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int u = 0; u < kEx2Chains; ++u) x[u] = ex2_approx(-x[u]);  // stays in (0.5, 1)
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    float s = 0.f;
#pragma unroll
    for (int u = 0; u < kEx2Chains; ++u) s += x[u];
    if (s == -1.0f) sink[threadIdx.x] = s;  // never true; keeps the chains alive
}

// The same with ex2.approx.f16x2: two fp16 exponentials per instruction.
__global__ void __launch_bounds__(kEx2Threads, 1)
    mb_ex2_f16x2_kernel(int iters, unsigned long long* cycles, float* sink) {
    uint32_t x[kEx2Chains];
#pragma unroll
    for (int u = 0; u < kEx2Chains; ++u) {
        const float f = 0.25f + 0.01f * (float)((threadIdx.x + u) & 31);
        asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(x[u]) : "f"(f), "f"(f + 0.125f));
    }
    __syncthreads();
    const unsigned long long t0 = clock64();
#pragma unroll 1
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int r = 0; r < 4; ++r)
#pragma unroll
            for (int u = 0; u < kEx2Chains; ++u)  // 2^-x for both halves: stays in (0.5, 1)
                asm volatile("ex2.approx.f16x2 %0, %1;" : "=r"(x[u]) : "r"(x[u] ^ 0x80008000u));
    }
    __syncthreads();
    const unsigned long long t1 = clock64();
    if (threadIdx.x == 0) cycles[blockIdx.x] = t1 - t0;
    uint32_t s = 0;
#pragma unroll
    for (int u = 0; u < kEx2Chains; ++u) s ^= x[u];
    if (s == 0xFFFFFFFFu) sink[threadIdx.x] = (float)s;  // never true; keeps the chains alive
}

constexpr int kMmaSmem = 120 * 1024;  // > half the SM's shared memory: one CTA per SM

// FORM 0: A and B K-major in shared memory (the QK^T form); FORM 1: A from Tensor Memory,
// B MN-major in shared memory (the PV form: P from TMEM, V as stored, d contiguous)
template <int N, bool FP8, int FORM>
__global__ void __launch_bounds__(128, 1)
    mb_mma_kernel(int iters, unsigned long long* cycles, uint32_t* err, unsigned long long limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    // FORM 0 -- A: 128 rows x 128 bytes, B: N rows x 128 bytes (one swizzle atom column
    // each, i.e. K = 64 bf16 or 128 e4m3 elements: four MMAs of K = 16 / 32).
    // FORM 1 -- B: 64 K rows x N columns, MN-major: N / (128 bytes) atom columns of 64 rows
    // x 128 bytes each (8 KiB apart); A: 128 lanes x 64 K elements in TMEM columns [256, ...).
    // All zeros.
    uint8_t* a = smem;
    uint8_t* b = smem + 128 * 128;
    uint64_t* bar = reinterpret_cast<uint64_t*>(b + N * 128);
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
    for (int i = threadIdx.x; i < (128 + N) * 128 / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(bar), 1);
        fence_barrier_init();
    }
    fence_proxy_async_smem();  // the zeros are visible to the tensor pipe
    if (threadIdx.x < 32) {
        tmem_alloc(smem_u32(tslot), 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (threadIdx.x == 0) {
        const uint32_t idesc = make_idesc(128, N, FP8 ? 0u : 1u, FORM == 1);
        const uint64_t da = sdesc_sw128(smem_u32(a), 16, 1024);
        // MN-major B: leading offset = the next 128-byte atom column along N (8 KiB: 64 K
        // rows of 128 bytes), stride offset = the next 8 K rows
        const uint64_t db = FORM == 1 ? sdesc_sw128(smem_u32(b), 8192, 1024)
                                      : sdesc_sw128(smem_u32(b), 16, 1024);
        const unsigned long long t0 = clock64();
#pragma unroll 1
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                // k step: 32 bytes (16 bf16 / 32 e4m3 elements) along the 128-byte rows
                const uint64_t off = (uint64_t)((kk * 32) >> 4);
                if constexpr (FORM == 1) {
                    // B: the next 16 (bf16) / 32 (e4m3) K rows of 128 bytes; A: the next 8
                    // TMEM columns (32 bytes of each lane's row)
                    const uint64_t boff = (uint64_t)((kk * (FP8 ? 32 : 16) * 128) >> 4);
                    if constexpr (FP8)
                        umma_f8_ts(tmem, tmem + 256u + 8u * kk, db + boff, idesc, (i | kk) != 0);
                    else
                        umma_f16_ts(tmem, tmem + 256u + 8u * kk, db + boff, idesc, (i | kk) != 0);
                } else if constexpr (FP8) {
                    umma_f8_ss(tmem, da + off, db + off, idesc, (i | kk) != 0);
                } else {
                    umma_f16_ss(tmem, da + off, db + off, idesc, (i | kk) != 0);
                }
            }
        }
        umma_commit(smem_u32(bar));
        const unsigned long long g0 = globaltimer_ns();
        bool ok = true;
        while (!mbar_try_wait(smem_u32(bar), 0u)) {
            if (globaltimer_ns() - g0 > limit_ns) {
                ok = false;
                break;
            }
        }
        const unsigned long long t1 = clock64();
        if (!ok) {
            atomicOr(err, 1u);
            // the MMAs still read shared memory and write TMEM: wait for them once more
            const unsigned long long g1 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(bar), 0u) && globaltimer_ns() - g1 < limit_ns) {
            }
        }
        cycles[blockIdx.x] = t1 - t0;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

template <int N, bool FP8, int FORM = 0>
cudaError_t launch_mma(int grid, int iters, unsigned long long* cycles, uint32_t* err,
                       unsigned long long limit_ns, cudaStream_t s) {
    cudaError_t e = cudaFuncSetAttribute(mb_mma_kernel<N, FP8, FORM>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kMmaSmem);
    if (e != cudaSuccess) return e;
    mb_mma_kernel<N, FP8, FORM><<<grid, 128, kMmaSmem, s>>>(iters, cycles, err, limit_ns);
    return cudaGetLastError();
}

// Bulk-copy throughput into shared memory: one thread per CTA keeps kLoadSlots copies of
// kLoadBytes in flight (cp.async.bulk, completion counted on one mbarrier per slot), each
// from the CTA's own window of `window` bytes of `src`, read cyclically.  With a window set
// that fits L2 (after a first pass) this is the L2 -> shared-memory rate; with a larger one,
// the HBM read rate.
constexpr int kLoadSlots = 4;
constexpr int kLoadBytes = 32 * 1024;
constexpr int kLoadSmem = kLoadSlots * kLoadBytes + 1024 + 64;

__global__ void __launch_bounds__(32, 1)
    mb_load_kernel(const uint8_t* src, unsigned long long window, int iters, unsigned long long* cycles,
                   uint32_t* err, unsigned long long limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kLoadSlots * kLoadBytes);
    if (threadIdx.x != 0) return;
    for (int s = 0; s < kLoadSlots; ++s) mbar_init(smem_u32(bars + s), 1);
    fence_barrier_init();
    const uint8_t* base = src + (size_t)blockIdx.x * window;
    const unsigned long long nchunks = window / kLoadBytes;
    const unsigned long long t0 = clock64();
    bool ok = true;
    for (int i = 0; i < iters && ok; ++i) {
        const int s = i % kLoadSlots;
        const uint32_t bar = smem_u32(bars + s);
        if (i >= kLoadSlots) {  // the slot's previous copy has landed
            const uint32_t parity = (uint32_t)((i / kLoadSlots) - 1) & 1u;
            const unsigned long long g0 = globaltimer_ns();
            while (!mbar_try_wait(bar, parity)) {
                if (globaltimer_ns() - g0 > limit_ns) {
                    ok = false;
                    break;
                }
            }
        }
        if (!ok) break;
        mbar_arrive_expect_tx(bar, kLoadBytes);
        const uint8_t* g = base + (size_t)(i % nchunks) * kLoadBytes;
        asm volatile(
            "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                smem_u32(smem + s * kLoadBytes)),
            "l"(g), "r"(kLoadBytes), "r"(bar)
            : "memory");
    }
    // the last copies have landed (bounded), before the time is taken and the CTA retires
    for (int i = (iters > kLoadSlots ? iters - kLoadSlots : 0); i < iters; ++i) {
        const uint32_t bar = smem_u32(bars + (i % kLoadSlots));
        const uint32_t parity = (uint32_t)(i / kLoadSlots) & 1u;
        const unsigned long long g0 = globaltimer_ns();
        while (!mbar_try_wait(bar, parity)) {
            if (globaltimer_ns() - g0 > limit_ns) {
                ok = false;
                break;
            }
        }
    }
    const unsigned long long t1 = clock64();
    if (!ok) atomicOr(err, 1u);
    cycles[blockIdx.x] = t1 - t0;
}

// The tensor pipe and the bulk-copy engine sharing one SM's shared memory: thread 0
// issues SS-form MMAs (M = 128, N = 128, bf16, as the QK^T product) for `iters` x 4
// instructions while thread 32 keeps two 32 KiB bulk copies in flight from the CTA's own
// L2-resident window (as the K/V stream) until the MMAs are done.  Reports the MMA cycles
// and the bytes copied meanwhile.
__global__ void __launch_bounds__(64, 1)
    mb_mma_load_kernel(const uint8_t* src, unsigned long long window, int iters,
                       unsigned long long* cycles, unsigned long long* bytes, uint32_t* err,
                       unsigned long long limit_ns) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* a = smem;                    // 16 KiB
    uint8_t* b = smem + 16384;            // 16 KiB
    uint8_t* ld = smem + 32768;           // 2 x 32 KiB copy slots
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 32768 + 2 * kLoadBytes);  // mma, 2 copies
    uint32_t* tslot = reinterpret_cast<uint32_t*>(bars + 3);
    volatile uint32_t* done = reinterpret_cast<volatile uint32_t*>(bars + 4);
    for (int i = threadIdx.x; i < 32768 / 16; i += blockDim.x)
        reinterpret_cast<uint4*>(smem)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) {
        for (int s = 0; s < 3; ++s) mbar_init(smem_u32(bars + s), 1);
        *done = 0u;
        fence_barrier_init();
    }
    fence_proxy_async_smem();
    if (threadIdx.x < 32) {
        tmem_alloc(smem_u32(tslot), 512);
        tmem_relinquish();
        tc_fence_before();
    }
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tslot;
    if (threadIdx.x == 0) {
        const uint32_t idesc = make_idesc(128, 128, 1u, false);
        const uint64_t da = sdesc_sw128(smem_u32(a), 16, 1024);
        const uint64_t db = sdesc_sw128(smem_u32(b), 16, 1024);
        const unsigned long long t0 = clock64();
#pragma unroll 1
        for (int i = 0; i < iters; ++i) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
                const uint64_t off = (uint64_t)((kk * 32) >> 4);
                umma_f16_ss(tmem, da + off, db + off, idesc, (i | kk) != 0);
            }
        }
        umma_commit(smem_u32(bars));
        const unsigned long long g0 = globaltimer_ns();
        bool ok = true;
        while (!mbar_try_wait(smem_u32(bars), 0u)) {
            if (globaltimer_ns() - g0 > limit_ns) {
                ok = false;
                break;
            }
        }
        const unsigned long long t1 = clock64();
        if (!ok) {
            atomicOr(err, 1u);
            const unsigned long long g1 = globaltimer_ns();
            while (!mbar_try_wait(smem_u32(bars), 0u) && globaltimer_ns() - g1 < limit_ns) {
            }
        }
        cycles[blockIdx.x] = t1 - t0;
        *done = 1u;
    } else if (threadIdx.x == 32) {
        const uint8_t* base = src + (size_t)blockIdx.x * window;
        const unsigned long long nchunks = window / kLoadBytes;
        // copy i uses slot i & 1 and completes that slot's phase i >> 1; two in flight
        unsigned long long issued = 0, landed = 0;
        bool ok = true;
        const unsigned long long g0 = globaltimer_ns();
        while (ok) {
            if (issued - landed == 2 || (*done && issued > landed)) {  // wait for the oldest
                const uint32_t bar = smem_u32(bars + 1 + (landed & 1));
                while (!mbar_try_wait(bar, (uint32_t)(landed >> 1) & 1u)) {
                    if (globaltimer_ns() - g0 > limit_ns) {
                        ok = false;
                        break;
                    }
                }
                if (ok) ++landed;
                continue;
            }
            if (*done) break;  // (nothing in flight)
            const int s = (int)(issued & 1);
            const uint32_t bar = smem_u32(bars + 1 + s);
            mbar_arrive_expect_tx(bar, kLoadBytes);
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                    smem_u32(ld + s * kLoadBytes)),
                "l"(base + (size_t)(issued % nchunks) * kLoadBytes), "r"(kLoadBytes), "r"(bar)
                : "memory");
            ++issued;
        }
        if (!ok) atomicOr(err, 2u);
        bytes[blockIdx.x] = landed * (unsigned long long)kLoadBytes;
    }
    __syncthreads();
    if (threadIdx.x < 32) {
        tc_fence_after();
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

extern "C" {

int fa_mb_load(int grid, const void* src, unsigned long long window, int iters, unsigned long long* cycles,
               uint32_t* err, unsigned long long limit_ns, void* stream) {
    if (grid < 1 || iters < 1 || !src || !cycles || !err || window < (unsigned long long)kLoadBytes ||
        window % kLoadBytes != 0 || (reinterpret_cast<uintptr_t>(src) & 15u) != 0)
        return (int)cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(mb_load_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kLoadSmem);
    if (e != cudaSuccess) return (int)e;
    mb_load_kernel<<<grid, 32, kLoadSmem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(src), window, iters, cycles, err, limit_ns);
    return (int)cudaGetLastError();
}

long long fa_mb_load_bytes_per_cta(int iters) { return (long long)iters * kLoadBytes; }

int fa_mb_mma_with_load(int grid, const void* src, unsigned long long window, int iters,
                        unsigned long long* cycles, unsigned long long* bytes, uint32_t* err,
                        unsigned long long limit_ns, void* stream) {
    if (grid < 1 || iters < 1 || !src || !cycles || !bytes || !err ||
        window < (unsigned long long)kLoadBytes || window % kLoadBytes != 0 ||
        (reinterpret_cast<uintptr_t>(src) & 15u) != 0)
        return (int)cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(mb_mma_load_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kMmaSmem);
    if (e != cudaSuccess) return (int)e;
    mb_mma_load_kernel<<<grid, 64, kMmaSmem, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint8_t*>(src), window, iters, cycles, bytes, err, limit_ns);
    return (int)cudaGetLastError();
}

int fa_mb_ex2(int grid, int iters, unsigned long long* cycles, float* sink, void* stream) {
    if (grid < 1 || iters < 1 || !cycles || !sink) return (int)cudaErrorInvalidValue;
    mb_ex2_kernel<<<grid, kEx2Threads, 0, static_cast<cudaStream_t>(stream)>>>(iters, cycles, sink);
    return (int)cudaGetLastError();
}

int fa_mb_ex2_f16x2(int grid, int iters, unsigned long long* cycles, float* sink, void* stream) {
    if (grid < 1 || iters < 1 || !cycles || !sink) return (int)cudaErrorInvalidValue;
    mb_ex2_f16x2_kernel<<<grid, kEx2Threads, 0, static_cast<cudaStream_t>(stream)>>>(iters, cycles, sink);
    return (int)cudaGetLastError();
}

long long fa_mb_ex2_per_cta(int iters) { return (long long)kEx2Threads * kEx2Chains * 4 * iters; }

int fa_mb_mma(int grid, int n, int fp8, int iters, unsigned long long* cycles, uint32_t* err,
              unsigned long long limit_ns, void* stream) {
    if (grid < 1 || iters < 1 || !cycles || !err) return (int)cudaErrorInvalidValue;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (!fp8 && n == 64) return (int)launch_mma<64, false>(grid, iters, cycles, err, limit_ns, s);
    if (!fp8 && n == 128) return (int)launch_mma<128, false>(grid, iters, cycles, err, limit_ns, s);
    if (!fp8 && n == 256) return (int)launch_mma<256, false>(grid, iters, cycles, err, limit_ns, s);
    if (fp8 && n == 128) return (int)launch_mma<128, true>(grid, iters, cycles, err, limit_ns, s);
    if (fp8 && n == 256) return (int)launch_mma<256, true>(grid, iters, cycles, err, limit_ns, s);
    // the PV form (A from TMEM, B MN-major), N = head dim 128
    if (!fp8 && n == -128) return (int)launch_mma<128, false, 1>(grid, iters, cycles, err, limit_ns, s);
    if (fp8 && n == -128) return (int)launch_mma<128, true, 1>(grid, iters, cycles, err, limit_ns, s);
    return (int)cudaErrorInvalidValue;
}

long long fa_mb_mma_flops_per_cta(int n, int fp8, int iters) {
    if (n < 0) n = -n;  // (the PV form)
    // 4 MMAs per iteration (the 128-byte rows hold K = 64 bf16 or K = 128 e4m3), each
    // 2 * M * N * K FLOPs with M = 128
    const long long k_per_mma = fp8 ? 32 : 16;
    return 4LL * iters * 2LL * 128 * n * k_per_mma;
}

}  // extern "C"
