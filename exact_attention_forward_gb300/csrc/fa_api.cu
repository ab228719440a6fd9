// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// validation, work decomposition (query-tile pairs, optional key splits),
// TMA tensor-map encoding, launches, the split merge kernel and the
// device-side failure word.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_internal.h"

namespace fa {

__device__ uint32_t g_fa_error_word;

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 4000000000ull;  // 4 s

thread_local char t_detail[512] = "";
std::mutex g_mu;
uint64_t g_wait_limit_ns = kDefaultWaitNs;
uint32_t g_inject = 0;
int g_num_sms[kMaxDevices] = {0};
uint32_t* g_err_addr[kMaxDevices] = {nullptr};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

fa_status fail(fa_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_detail, sizeof t_detail, fmt, ap);
    va_end(ap);
    return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

fa_status device_info(int* dev, int* sms, uint32_t** err) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return fail(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (*dev < 0 || *dev >= kMaxDevices) return fail(FA_ERR_CUDA, "device index %d out of range", *dev);
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_num_sms[*dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_fa_error_word);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "error word: %s", cudaGetErrorString(e));
        g_err_addr[*dev] = static_cast<uint32_t*>(addr);
        g_num_sms[*dev] = n;
    }
    if (!g_encode) {
        cudaDriverEntryPointQueryResult q;
        void* fn = nullptr;
        e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
        if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
            return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    *sms = g_num_sms[*dev];
    *err = g_err_addr[*dev];
    return FA_OK;
}

// 4-D view (d, head, row, batch) of a [batch, rows, heads, d] tensor; box =
// one 128-byte swizzle atom of d by 128 rows of one head.
fa_status encode_map(CUtensorMap* m, const void* base, bool fp8, int d, int heads, int rows,
                     int batch) {
    const int elem = fp8 ? 1 : 2;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1),
                          (cuuint64_t)(batch > 0 ? batch : 1)};
    cuuint64_t strides[3] = {(cuuint64_t)d * elem, (cuuint64_t)heads * d * elem,
                             (cuuint64_t)(rows > 0 ? rows : 1) * heads * d * elem};
    cuuint32_t box[4] = {(cuuint32_t)(128 / elem), 1u, 128u, 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                          const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FA_OK;
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// Key splits for a fixed-length shape: only when the (batch, head, tile-pair)
// items cannot fill the GPU and the key range is long.
int choose_splits(int batch, int heads, int sq, int sk, int causal, int sms) {
    (void)causal;
    const long long items = (long long)ceil_div(sq, 256) * batch * heads;
    const int nblk = ceil_div(sk, 128);
    if (items <= 0 || nblk < 8 || items * 2 > sms) return 1;
    int s = ceil_div(sms, items);
    s = s < nblk / 4 ? s : nblk / 4;  // at least 4 key blocks per split
    if (s < 2) return 1;
    const int bps = ceil_div(nblk, s);
    return ceil_div(nblk, bps);
}

size_t workspace_bytes_for(int splits, int batch, int heads, int sq, int dv) {
    if (splits <= 1) return 0;
    const size_t rows = (size_t)splits * batch * heads * sq;
    return rows * (size_t)dv * sizeof(float) + rows * sizeof(float);
}

}  // namespace

// ---------------------------------------------------------------- split merge
// One warp per output row.  LSE = ln sum_s exp(LSE_s) and O = sum_s exp(LSE_s - LSE) O_s.
// Lanes own splits for the LSE reductions (warp shuffles; for <= 32 splits each lane keeps
// its weight in a register and broadcasts it), then own 4 (Dv = 128) or 2 (Dv = 64)
// columns of O; the split loop is unrolled so several partial rows are in flight at once.
template <int DV>
__global__ void __launch_bounds__(256) fa_combine_kernel(const float* __restrict__ ws_o,
                                                         const float* __restrict__ ws_lse,
                                                         __nv_bfloat16* __restrict__ o,
                                                         float* __restrict__ lse, int batch,
                                                         int heads, int sq, int splits) {
    constexpr int kCols = DV / 32;  // columns per lane
    const long long rows = (long long)batch * heads * sq;
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int i = (int)(row % sq);
    const long long bh = row / sq;
    const int h = (int)(bh % heads);
    const long long b = bh / heads;
    const size_t stride = (size_t)rows;  // rows per split
    // launched as a programmatic dependent of the forward kernel: wait for its
    // completion (and memory) before reading the partial results
    asm volatile("griddepcontrol.wait;" ::: "memory");
    float mx = -INFINITY;
    for (int s = lane; s < splits; s += 32) mx = fmaxf(mx, __ldg(ws_lse + s * stride + row));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    __nv_bfloat16* out = o + (((size_t)b * sq + i) * heads + h) * DV + lane * kCols;
    float* lse_out = lse + ((size_t)b * heads + h) * sq + i;
    if (mx == -INFINITY) {  // no split saw a key: O = 0, LSE = -inf
#pragma unroll
        for (int c = 0; c < kCols; ++c) out[c] = __float2bfloat16(0.f);
        if (lane == 0) *lse_out = -INFINITY;
        return;
    }
    float w_lane = 0.f, tot = 0.f;
    for (int s = lane; s < splits; s += 32) {
        const float e = expf(__ldg(ws_lse + s * stride + row) - mx);
        if (s < 32) w_lane = e;
        tot += e;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    const float inv = 1.0f / tot;
    float acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
    const float* src = ws_o + (size_t)row * DV + lane * kCols;
    // batches of 8 splits: all 8 partial-row loads are issued before any is used
    constexpr int kBatch = 8;
    for (int s0 = 0; s0 < splits; s0 += kBatch) {
        float v[kBatch][kCols];
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int s = s0 + u;
#pragma unroll
            for (int c = 0; c < kCols; ++c) v[u][c] = 0.f;
            if (s < splits) {
                if constexpr (kCols == 4) {
                    const float4 t = __ldg(reinterpret_cast<const float4*>(src + s * stride * DV));
                    v[u][0] = t.x; v[u][1] = t.y; v[u][2] = t.z; v[u][3] = t.w;
                } else {
                    const float2 t = __ldg(reinterpret_cast<const float2*>(src + s * stride * DV));
                    v[u][0] = t.x; v[u][1] = t.y;
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int s = s0 + u;  // uniform across the warp
            float w = 0.f;
            if (s < 32)
                w = __shfl_sync(0xffffffffu, w_lane, s) * inv;  // 0 past the last split
            else if (s < splits)
                w = expf(__ldg(ws_lse + s * stride + row) - mx) * inv;
#pragma unroll
            for (int c = 0; c < kCols; ++c) acc[c] = fmaf(w, v[u][c], acc[c]);
        }
    }
    if constexpr (kCols == 4) {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc[0], acc[1]);
        __nv_bfloat162 hi = __floats2bfloat162_rn(acc[2], acc[3]);
        uint2 pk;
        pk.x = *reinterpret_cast<uint32_t*>(&lo);
        pk.y = *reinterpret_cast<uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out) = pk;
    } else {
        *reinterpret_cast<__nv_bfloat162*>(out) = __floats2bfloat162_rn(acc[0], acc[1]);
    }
    if (lane == 0) *lse_out = mx + logf(tot);
}

cudaError_t launch_combine(const float* ws_o, const float* ws_lse, void* o, float* lse, int batch,
                           int heads, int seqlen_q, int dv, int n_splits, cudaStream_t s) {
    const long long rows = (long long)batch * heads * seqlen_q;
    const int threads = 256;
    const long long blocks = (rows * 32 + threads - 1) / threads;
    // programmatic dependent launch: the merge grid is set up while the forward
    // kernel drains; griddepcontrol.wait in the merge orders it after the forward
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks);
    cfg.blockDim = dim3(threads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    __nv_bfloat16* ob = static_cast<__nv_bfloat16*>(o);
    if (dv == 128)
        return cudaLaunchKernelEx(&cfg, fa_combine_kernel<128>, ws_o, ws_lse, ob, lse, batch, heads,
                                  seqlen_q, n_splits);
    return cudaLaunchKernelEx(&cfg, fa_combine_kernel<64>, ws_o, ws_lse, ob, lse, batch, heads,
                              seqlen_q, n_splits);
}

}  // namespace fa

using namespace fa;

extern "C" {

const char* fa_status_string(fa_status s) {
    switch (s) {
    case FA_OK: return "ok";
    case FA_ERR_INVALID_ARG: return "invalid argument";
    case FA_ERR_UNSUPPORTED: return "unsupported configuration";
    case FA_ERR_CUDA: return "CUDA error";
    case FA_ERR_WORKSPACE: return "workspace too small";
    case FA_ERR_DEVICE_TIMEOUT: return "device-side wait timed out";
    }
    return "unknown status";
}

const char* fa_last_error_detail(void) { return t_detail; }

void fa_debug_set(uint64_t wait_limit_ns, uint32_t inject) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_wait_limit_ns = wait_limit_ns ? wait_limit_ns : kDefaultWaitNs;
    g_inject = inject;
}

fa_status fa_device_error(uint32_t* flags, int clear) {
    int dev, sms;
    uint32_t* err;
    fa_status st = device_info(&dev, &sms, &err);
    if (st != FA_OK) return st;
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return fail(FA_ERR_CUDA, "synchronize: %s", cudaGetErrorString(e));
    uint32_t w = 0;
    e = cudaMemcpy(&w, err, sizeof w, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return fail(FA_ERR_CUDA, "read error word: %s", cudaGetErrorString(e));
    if (clear) {
        e = cudaMemset(err, 0, sizeof w);
        if (e == cudaSuccess) e = cudaDeviceSynchronize();
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "clear error word: %s", cudaGetErrorString(e));
    }
    if (flags) *flags = w;
    if (w & kErrTimeout)
        return fail(FA_ERR_DEVICE_TIMEOUT, "device wait timed out at site %u", (w >> 8) & 0xFFu);
    return FA_OK;
}

int fa_fwd_num_splits(int batch, int heads, int seqlen_q, int seqlen_k, int causal) {
    int dev, sms;
    uint32_t* err;
    if (batch < 1 || heads < 1 || seqlen_q < 1 || seqlen_k < 1) return 1;
    if (device_info(&dev, &sms, &err) != FA_OK) return 1;
    return choose_splits(batch, heads, seqlen_q, seqlen_k, causal, sms);
}

size_t fa_fwd_workspace_size(int batch, int heads, int seqlen_q, int seqlen_k, int head_dim_v,
                             int causal) {
    const int s = fa_fwd_num_splits(batch, heads, seqlen_q, seqlen_k, causal);
    if (head_dim_v < 1) return 0;
    return workspace_bytes_for(s, batch, heads, seqlen_q, head_dim_v);
}

fa_status fa_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int batch,
                 int heads, int seqlen_q, int seqlen_k, const int32_t* cu_seqlens_q,
                 const int32_t* cu_seqlens_k, int max_seqlen_q, int max_seqlen_k, int head_dim,
                 int head_dim_v, float softmax_scale, int causal, fa_dtype dtype,
                 const float* q_descale, const float* k_descale, const float* v_descale,
                 void* workspace, size_t workspace_bytes, void* stream) {
    return fa_fwd_gqa(q, k, v, o, lse, batch, heads, heads, seqlen_q, seqlen_k, cu_seqlens_q,
                      cu_seqlens_k, max_seqlen_q, max_seqlen_k, head_dim, head_dim_v, softmax_scale,
                      causal, dtype, q_descale, k_descale, v_descale, workspace, workspace_bytes,
                      stream);
}

fa_status fa_fwd_gqa(const void* q, const void* k, const void* v, void* o, float* lse, int batch,
                     int heads, int heads_k, int seqlen_q, int seqlen_k,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int max_seqlen_q,
                     int max_seqlen_k, int head_dim, int head_dim_v, float softmax_scale,
                     int causal, fa_dtype dtype, const float* q_descale, const float* k_descale,
                     const float* v_descale, void* workspace, size_t workspace_bytes,
                     void* stream) {
    t_detail[0] = '\0';
    // ---------------------------------------------------------------- validation
    const bool varlen = cu_seqlens_q != nullptr || cu_seqlens_k != nullptr;
    // with no key rows at all (fixed length seqlen_k == 0, or varlen total 0) K and V may be NULL
    const bool no_keys = seqlen_k == 0;
    if (!q || !o || !lse || (!no_keys && (!k || !v)))
        return fail(FA_ERR_INVALID_ARG, "q, k, v, o and lse must be non-NULL device pointers");
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
        return fail(FA_ERR_INVALID_ARG, "q, k, v, o and lse must be 16-byte aligned");
    if (batch < 0 || heads < 1 || seqlen_q < 0 || seqlen_k < 0)
        return fail(FA_ERR_INVALID_ARG, "need batch >= 0, heads >= 1, seqlen_q/k >= 0");
    if (heads_k < 1 || heads % heads_k != 0)
        return fail(FA_ERR_INVALID_ARG, "heads_k (%d) must be >= 1 and divide heads (%d)", heads_k,
                    heads);
    if (causal != 0 && causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (!(softmax_scale > 0.0f) || !std::isfinite(softmax_scale))
        return fail(FA_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
    if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_E4M3)
        return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    if (dtype == FA_DTYPE_BF16 && (q_descale || k_descale || v_descale))
        return fail(FA_ERR_INVALID_ARG, "descale pointers are only meaningful for FA_DTYPE_E4M3");
    if ((q_descale && (reinterpret_cast<uintptr_t>(q_descale) & 3u)) ||
        (k_descale && (reinterpret_cast<uintptr_t>(k_descale) & 3u)) ||
        (v_descale && (reinterpret_cast<uintptr_t>(v_descale) & 3u)))
        return fail(FA_ERR_INVALID_ARG, "descale pointers must be 4-byte aligned");
    if (varlen && (!cu_seqlens_q || !cu_seqlens_k))
        return fail(FA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must both be given");
    if (varlen && (max_seqlen_q < 0 || max_seqlen_k < 0))
        return fail(FA_ERR_INVALID_ARG, "max_seqlen_q/k must be >= 0 for varlen");
    if (head_dim != head_dim_v)
        return fail(FA_ERR_UNSUPPORTED, "head_dim (%d) != head_dim_v (%d) is not built", head_dim,
                    head_dim_v);
    if (dtype == FA_DTYPE_BF16 && head_dim != 64 && head_dim != 128)
        return fail(FA_ERR_UNSUPPORTED, "bf16 head_dim %d not built (64, 128)", head_dim);
    if (dtype == FA_DTYPE_E4M3 && head_dim != 128)
        return fail(FA_ERR_UNSUPPORTED, "e4m3 head_dim %d not built (128)", head_dim);
    const long long rows_q = varlen ? seqlen_q : (long long)batch * seqlen_q;
    const long long rows_k = varlen ? seqlen_k : (long long)batch * seqlen_k;
    if (rows_q * heads * head_dim >= (1ll << 40) || rows_k * heads_k * head_dim >= (1ll << 40))
        return fail(FA_ERR_INVALID_ARG, "tensor too large");
    if (rows_q >= (1ll << 31) || rows_k >= (1ll << 31))
        return fail(FA_ERR_INVALID_ARG, "row count must fit in int32");
    const int mq = varlen ? max_seqlen_q : seqlen_q;
    const int mk = varlen ? max_seqlen_k : seqlen_k;
    if (batch == 0 || rows_q == 0 || mq == 0) return FA_OK;  // nothing to compute

    int dev, sms;
    uint32_t* err;
    fa_status st = device_info(&dev, &sms, &err);
    if (st != FA_OK) return st;

    // ---------------------------------------------------------------- decomposition
    int splits = 1;
    if (!varlen && workspace) {
        splits = choose_splits(batch, heads, seqlen_q, seqlen_k, causal, sms);
        const size_t need = workspace_bytes_for(splits, batch, heads, seqlen_q, head_dim_v);
        if (workspace_bytes < need)
            return fail(FA_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed", workspace_bytes,
                        need);
        if (!aligned16(workspace)) return fail(FA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    }
    FwdParams p{};
    p.o = o;
    p.lse = lse;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.q_descale = q_descale;
    p.k_descale = k_descale;
    p.v_descale = v_descale;
    p.err = err;
    p.batch = batch;
    p.heads = heads;
    p.kv_group = heads / heads_k;
    p.seqlen_q = mq;
    p.seqlen_k = mk;
    p.total_q = varlen ? seqlen_q : 0;
    p.n_mpairs = ceil_div(mq, 256);
    p.n_splits = splits;
    const int nblk = ceil_div(mk > 0 ? mk : 1, 128);
    p.blocks_per_split = splits > 1 ? ceil_div(nblk, splits) : (1 << 29);
    const long long n_items = (long long)p.n_mpairs * batch * heads * splits;
    if (n_items >= (1ll << 31)) return fail(FA_ERR_INVALID_ARG, "too many work items");
    p.n_items = (int)n_items;
    p.scale_log2 = softmax_scale * 1.4426950408889634f;
    p.causal = causal;
    p.varlen = varlen ? 1 : 0;
    p.split = splits > 1 ? 1 : 0;
    if (p.split) {
        const size_t rows = (size_t)splits * batch * heads * seqlen_q;
        p.ws_o = static_cast<float*>(workspace);
        p.ws_lse = p.ws_o + rows * head_dim_v;
    }
    {
        std::lock_guard<std::mutex> lk(g_mu);
        p.wait_limit_ns = g_wait_limit_ns;
        p.inject = g_inject;
    }

    // ---------------------------------------------------------------- tensor maps
    const bool fp8 = dtype == FA_DTYPE_E4M3;
    CUtensorMap tq, tk, tv;
    // fixed length: (d, head, seq row, batch); varlen: (d, head, packed row, 1)
    const int nbat = varlen ? 1 : batch;
    if ((st = encode_map(&tq, q, fp8, head_dim, heads, seqlen_q, nbat)) != FA_OK) return st;
    if (no_keys) {  // no key block is ever loaded; any valid map will do
        tk = tq;
        tv = tq;
    } else {
        if ((st = encode_map(&tk, k, fp8, head_dim, heads_k, seqlen_k, nbat)) != FA_OK) return st;
        if ((st = encode_map(&tv, v, fp8, head_dim, heads_k, seqlen_k, nbat)) != FA_OK) return st;
    }

    // ---------------------------------------------------------------- launch
    const int grid = (int)(n_items < sms ? n_items : sms);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (fp8)
        e = launch_fwd_e4m3_d128(tq, tk, tv, p, grid, s);
    else if (head_dim == 64)
        e = launch_fwd_bf16_d64(tq, tk, tv, p, grid, s);
    else
        e = launch_fwd_bf16_d128(tq, tk, tv, p, grid, s);
    if (e != cudaSuccess) return fail(FA_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
    if (p.split) {
        e = launch_combine(p.ws_o, p.ws_lse, o, lse, batch, heads, seqlen_q, head_dim_v, splits, s);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
    }
    return FA_OK;
}

}  // extern "C"
