// fa_api.cu -- host side of the C ABI declared in include/fa.h: argument
// validation, work decomposition (query-tile pairs, optional key splits),
// TMA tensor-map encoding, launches, the split merge kernel and the
// device-side failure word.
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <atomic>
#include <mutex>

#include <cuda_bf16.h>
#include <cudaTypedefs.h>

#include "fa.h"
#include "fa_internal.h"

namespace fa {

__device__ uint32_t g_fa_error_word;

// Work counters of the greedy item scheduler (varlen launches): one {next item, CTAs
// done} pair per launch slot.  Each launch takes the next slot of its range round-robin
// (eager launches and launches captured into CUDA graphs have separate ranges) and its
// last CTA returns the pair to zero, so up to 192 eager launches may be in flight on a
// device at once.  A captured launch keeps its slot in every replay: two replays of one
// graph, or of two graphs whose varlen launches drew the same captured slot (64 apart),
// must not run at the same time.
constexpr int kSchedSlots = 256;
__device__ uint32_t g_fa_sched[2 * kSchedSlots];

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kDefaultWaitNs = 4000000000ull;  // 4 s

thread_local char t_detail[512] = "";
std::mutex g_mu;
uint64_t g_wait_limit_ns = kDefaultWaitNs;
uint32_t g_inject = 0;
int g_steady_mode = 0;  // fa_debug_select_steady
uint64_t* g_trace = nullptr;  // event log of a FA_TRACE build (fa_debug_trace)
int g_num_sms[kMaxDevices] = {0};
// Device addresses of the library's __device__ variables, valid for the context they were
// looked up in: a cudaDeviceReset (or any new context) reloads the module at other
// addresses, so they are looked up again whenever the current context's id changes.
unsigned long long g_addr_ctx[kMaxDevices] = {0};
uint32_t* g_err_addr[kMaxDevices] = {nullptr};
uint32_t* g_sched_addr[kMaxDevices] = {nullptr};
// Counter slots: eager launches take [0, kEagerSlots) round-robin; launches recorded into
// a CUDA graph keep their slot for every replay, so they take theirs from the separate
// range [kEagerSlots, kSchedSlots) and never share one with an eager launch.
constexpr int kEagerSlots = 192;
// (tile, key block) steps per CTA from which a bf16 D = 128 launch without a cache takes the
// kernel instance specialised for steady key blocks.  Measured, both instances from one
// library, L2 flushed: +5.5 % at 54 per CTA (causal 2K), even at 108-121, -2.8 to -4 % at
// 215-243, -5.8 % at 431.
constexpr double kSteadyMinTileBlocksPerCta = 128.0;
std::atomic<uint32_t> g_sched_next{0};
std::atomic<uint32_t> g_sched_next_captured{0};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
PFN_cuCtxGetId_v12000 g_ctx_get_id = nullptr;

fa_status fail(fa_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(t_detail, sizeof t_detail, fmt, ap);
    va_end(ap);
    return s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Driver entry points, resolved once (g_mu held).
bool driver_entry(const char* name, int version, void** fn) {
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion(name, fn, version, cudaEnableDefault, &q);
    return e == cudaSuccess && q == cudaDriverEntryPointSuccess && *fn;
}

// Unique id of the calling thread's current context, 0 if there is none yet (g_mu held).
unsigned long long context_id_locked() {
    if (!g_ctx_current || !g_ctx_get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (g_ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return 0;
    if (g_ctx_get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

fa_status resolve_driver_entries() {
    if (!g_encode) {
        void* fn = nullptr;
        if (!driver_entry("cuTensorMapEncodeTiled", 12000, &fn))
            return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled entry point unavailable");
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    if (!g_ctx_current || !g_ctx_get_id) {
        void *f1 = nullptr, *f2 = nullptr;
        if (!driver_entry("cuCtxGetCurrent", 4000, &f1) || !driver_entry("cuCtxGetId", 12000, &f2))
            return fail(FA_ERR_CUDA, "cuCtxGetCurrent / cuCtxGetId entry points unavailable");
        g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(f1);
        g_ctx_get_id = reinterpret_cast<PFN_cuCtxGetId_v12000>(f2);
    }
    return FA_OK;
}

fa_status device_info(int* dev, int* sms, uint32_t** err) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return fail(FA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (*dev < 0 || *dev >= kMaxDevices) return fail(FA_ERR_CUDA, "device index %d out of range", *dev);
    std::lock_guard<std::mutex> lk(g_mu);
    fa_status st = resolve_driver_entries();
    if (st != FA_OK) return st;
    if (g_num_sms[*dev] == 0) {
        int n = 0;
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, *dev);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "SM count: %s", cudaGetErrorString(e));
        g_num_sms[*dev] = n;
    }
    const unsigned long long ctx = context_id_locked();
    if (ctx == 0 || ctx != g_addr_ctx[*dev]) {
        // (the lookup also creates the device's primary context if nothing has yet)
        void* addr = nullptr;
        e = cudaGetSymbolAddress(&addr, g_fa_error_word);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "error word: %s", cudaGetErrorString(e));
        g_err_addr[*dev] = static_cast<uint32_t*>(addr);
        e = cudaGetSymbolAddress(&addr, g_fa_sched);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "work counters: %s", cudaGetErrorString(e));
        g_sched_addr[*dev] = static_cast<uint32_t*>(addr);
        g_addr_ctx[*dev] = context_id_locked();
    }
    *sms = g_num_sms[*dev];
    *err = g_err_addr[*dev];
    return FA_OK;
}

uint32_t* next_sched_slot(int dev, cudaStream_t s) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const bool captured = cudaStreamIsCapturing(s, &cap) == cudaSuccess &&
                          cap == cudaStreamCaptureStatusActive;
    const uint32_t slot =
        captured ? (uint32_t)kEagerSlots +
                       g_sched_next_captured.fetch_add(1u) % (uint32_t)(kSchedSlots - kEagerSlots)
                 : g_sched_next.fetch_add(1u) % (uint32_t)kEagerSlots;
    std::lock_guard<std::mutex> lk(g_mu);
    return g_sched_addr[dev] + 2 * slot;
}

// 4-D view (d, head, row, batch) of a [batch, rows, heads, d] tensor; box =
// one 128-byte swizzle atom of d by 128 rows of one head, or (box_heads > 1) by
// box_heads heads x 128 / box_heads rows -- 128 shared-memory rows either way.
// box_rows > 0 overrides the rows of a box (a CTA pair loads 64-key halves of K blocks).
fa_status encode_map(CUtensorMap* m, const void* base, bool fp8, int d, int heads, int rows,
                     int batch, int box_heads = 1, int box_rows = 0) {
    const int elem = fp8 ? 1 : 2;
    cuuint64_t dims[4] = {(cuuint64_t)d, (cuuint64_t)heads, (cuuint64_t)(rows > 0 ? rows : 1),
                          (cuuint64_t)(batch > 0 ? batch : 1)};
    cuuint64_t strides[3] = {(cuuint64_t)d * elem, (cuuint64_t)heads * d * elem,
                             (cuuint64_t)(rows > 0 ? rows : 1) * heads * d * elem};
    cuuint32_t box[4] = {(cuuint32_t)(128 / elem), (cuuint32_t)box_heads,
                         (cuuint32_t)(box_rows > 0 ? box_rows : 128 / box_heads), 1u};
    cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
    CUresult r = g_encode(m, fp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                          const_cast<void*>(base), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(FA_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return FA_OK;
}

int ceil_div(long long a, long long b) { return (int)((a + b - 1) / b); }

// CTA pairs of the pair kernel that fit on the device at once (cached per device).
int g_pairs[kMaxDevices] = {0};
fa_status resident_pairs(int dev, int* pairs) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_pairs[dev] == 0) {
        int n = 0;
        cudaError_t e = max_resident_pairs_bf16_d128(&n);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "cluster occupancy: %s", cudaGetErrorString(e));
        if (n < 1) return fail(FA_ERR_UNSUPPORTED, "no CTA pair of the kernel fits on this device");
        g_pairs[dev] = n;
    }
    *pairs = g_pairs[dev];
    return FA_OK;
}

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

// Grouped-query packing: the query heads that share a K/V head are packed into the
// rows of one tile (row = query row x head) when a whole group of short query blocks
// fits one tile pair -- decoding and short prefill chunks, where one head per tile
// would leave most tile rows empty and stream each K/V head once per query head.
int choose_pack(int heads, int heads_k, int sq, bool varlen) {
    const int group = heads / heads_k;
    if (varlen || group <= 1 || 128 % group != 0 || (long long)sq * group > 256) return 1;
    return group;
}

// Splits of the key range for a fixed-length shape, taking packing into account.
int plan_splits(int batch, int heads, int heads_k, int sq, int sk, int causal, int sms) {
    const int pack = choose_pack(heads, heads_k, sq, false);
    return choose_splits(batch, heads / pack, sq * pack, sk, causal, sms);
}

// Balanced plan for key/value-cache launches (cache lengths live on the device, so items
// differ in cost in ways the host cannot see): when the fixed-length rule does not split,
// the items are few (< 2 waves) and long, every CTA takes an equal share of the key
// blocks of all items, concatenated -- at most kStreamSlots pieces per item, merged by the
// LSE identity.  The batch's lengths are read into shared memory by each CTA (<= 64).
constexpr int kStreamSlots = 4;
constexpr int kStreamMaxBatch = 64;
bool use_stream_plan(int batch, int heads, int heads_k, int sq, int cap, int causal, int sms) {
    const int pack = choose_pack(heads, heads_k, sq, false);
    const long long mpairs = ceil_div((long long)sq * pack, 256);
    const long long items = mpairs * batch * (heads / pack);
    // (rows that see only part of their item's keys -- a causal mask over several query
    // rows -- would leave pieces without work: not planned this way)
    return batch <= kStreamMaxBatch && mpairs == 1 && items < 2LL * sms && ceil_div(cap, 128) >= 8 &&
           (!causal || sq == 1) && plan_splits(batch, heads, heads_k, sq, cap, causal, sms) == 1;
}

// L2-aware order for static schedules.  Taken level by level (all (batch, head) pairs of
// one pair index, then the next), the ~2 rounds of items running at one time span every
// (batch, head): at B=2, H=32, S=8192 that is 64 K/V streams of 4 MiB, twice what L2
// holds, and each K/V block came from DRAM about once per round (reads 4.8x the Q/K/V
// bytes).  Bands of consecutive levels per (batch, head) put a few heads' items side by
// side instead.  Item costs: equal without a causal mask, so all levels form one band
// (head-major).  Under a causal mask the cost falls with the level, and the snake
// balances it by giving each CTA complementary costs in paired rounds (positions c and
// 2P-1-c of a run of 2P items, P = CTAs).  A band of g levels keeps that pairing when g
// divides 2P and a band's items (g x items per level) are a multiple of 2P: g =
// 2P / gcd(items per level, 2P).  The last ~35 % of the levels (small items, the end of
// the schedule) stay in plain LPT order.
void set_item_bands(FwdParams& p, int nunits) {
    p.band_levels = p.band_items = p.band_lv = 0;
    if (p.greedy || p.stream || p.varlen || p.seqused_k || p.n_splits != 1 || nunits < 1 ||
        p.n_items <= nunits)
        return;
    const long long per_m = (long long)p.batch * p.item_heads;
    long long g = p.n_mpairs, bands = 1;
    if (p.causal) {
        long long a = per_m, b = 2LL * nunits;
        while (b) { const long long t = a % b; a = b; b = t; }
        g = 2LL * nunits / a;
        const long long tail = (p.n_mpairs * 35LL + 99) / 100;
        bands = g > 1 ? (p.n_mpairs - tail) / g : 0;
    }
    if (bands < 1 || g < 2) return;
    p.band_levels = (int)g;
    p.band_lv = (int)(bands * g);
    p.band_items = (int)(bands * g * per_m);
}

// Without a causal mask a static schedule's items (tile pairs) cost the same, so a
// part-filled last round leaves CTAs idle for a whole item: 2048 pairs on 152 CTAs take
// 14 rounds where 13.5 would do.  When the last round holds at most half as many pairs
// as there are CTAs, its pairs run as single tiles, two items each, one per CTA.  A tile
// alone costs ~0.8 of a pair (its softmax has no second tile's MMAs to hide behind), so
// the last round shortens by ~20 %.  Only for the one-CTA kernel.
void set_half_tail(FwdParams& p, int nunits) {
    p.half_from = 0;
    if (p.causal || p.greedy || p.stream || p.varlen || p.seqused_k || p.n_splits != 1 ||
        nunits < 1 || p.n_items <= nunits)
        return;
    const int tail = p.n_items % nunits;
    if (tail == 0 || 2 * tail > nunits) return;
    p.half_from = p.n_items - tail;
    p.n_items += tail;
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
// columns of O.  The partial rows of the first batch of splits are requested together
// with the LSEs (they do not depend on the weights), and a batch holds 12 splits, so up
// to 12 splits take one memory round trip and up to 24 take two.
// Packed variable-length batches (cu_q != nullptr): the partial rows are laid out by
// (sequence, head, row < sq = the longest sequence's length); rows past a sequence's own
// length hold nothing and are skipped, and the results go to the packed O [total_q, H, Dv]
// and LSE [H, total_q].
template <int DV>
__global__ void __launch_bounds__(256) fa_combine_kernel(const float* __restrict__ ws_o,
                                                         const float* __restrict__ ws_lse,
                                                         __nv_bfloat16* __restrict__ o,
                                                         float* __restrict__ lse, int batch,
                                                         int heads, int sq, int splits,
                                                         const int32_t* __restrict__ cu_q,
                                                         int total_q) {
    constexpr int kCols = DV / 32;  // columns per lane
    constexpr int kBatch = 12;
    const long long rows = (long long)batch * heads * sq;
    const long long row = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (row >= rows) return;
    const int i = (int)(row % sq);
    const long long bh = row / sq;
    const int h = (int)(bh % heads);
    const long long b = bh / heads;
    const size_t stride = (size_t)rows;  // rows per split
    const float* src = ws_o + (size_t)row * DV + lane * kCols;
    size_t out_row = ((size_t)b * sq + i) * heads + h;     // row of O (in units of DV)
    size_t lse_idx = ((size_t)b * heads + h) * sq + i;
    if (cu_q) {
        const int q0 = __ldg(cu_q + b);
        if (i >= __ldg(cu_q + b + 1) - q0) return;  // past this sequence's rows
        out_row = ((size_t)q0 + i) * heads + h;
        lse_idx = (size_t)h * total_q + q0 + i;
    }
    // launched as a programmatic dependent of the forward kernel: wait for its
    // completion (and memory) before reading the partial results
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // partial rows of splits [s0, s0 + kBatch): all loads issued before any is used
    auto load_batch = [&](int s0, float (&v)[kBatch][kCols]) {
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
    };
    const float lse_lane = lane < splits ? __ldg(ws_lse + lane * stride + row) : -INFINITY;
    float v[kBatch][kCols];
    load_batch(0, v);
    float mx = lse_lane;
    for (int s = lane + 32; s < splits; s += 32) mx = fmaxf(mx, __ldg(ws_lse + s * stride + row));
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
    __nv_bfloat16* out = o + out_row * DV + lane * kCols;
    float* lse_out = lse + lse_idx;
    if (mx == -INFINITY) {  // no split saw a key: O = 0, LSE = -inf
#pragma unroll
        for (int c = 0; c < kCols; ++c) out[c] = __float2bfloat16(0.f);
        if (lane == 0) *lse_out = -INFINITY;
        return;
    }
    const float w_lane = lane < splits ? expf(lse_lane - mx) : 0.f;
    float tot = w_lane;
    for (int s = lane + 32; s < splits; s += 32) tot += expf(__ldg(ws_lse + s * stride + row) - mx);
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tot += __shfl_xor_sync(0xffffffffu, tot, off);
    const float inv = 1.0f / tot;
    float acc[kCols];
#pragma unroll
    for (int c = 0; c < kCols; ++c) acc[c] = 0.f;
    for (int s0 = 0; s0 < splits; s0 += kBatch) {
        if (s0 > 0) load_batch(s0, v);
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            const int s = s0 + u;  // uniform across the warp
            float w = 0.f;
            if (s < 32)
                w = __shfl_sync(0xffffffffu, w_lane, s) * inv;  // 0 past the last split
            else if (s < splits)
                w = expf(__ldg(ws_lse + s * stride + row) - mx) * inv;
            // (a slot of weight 0 -- an empty split, or a piece slot the balanced cache plan
            // did not use -- adds nothing, and its O is not trusted: never written for unused
            // slots)
            if (w != 0.f) {
#pragma unroll
                for (int c = 0; c < kCols; ++c) acc[c] = fmaf(w, v[u][c], acc[c]);
            }
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
                           int heads, int seqlen_q, int dv, int n_splits, const int32_t* cu_q,
                           int total_q, cudaStream_t s) {
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
                                  seqlen_q, n_splits, cu_q, total_q);
    return cudaLaunchKernelEx(&cfg, fa_combine_kernel<64>, ws_o, ws_lse, ob, lse, batch, heads,
                              seqlen_q, n_splits, cu_q, total_q);
}

// Every entry point fills one of these; fwd_impl validates and launches.
struct FwdArgs {
    const void *q, *k, *v;
    void* o;
    float* lse;
    int batch, heads, heads_k, seqlen_q, seqlen_k;
    const int32_t *cu_q, *cu_k;
    int max_q, max_k, head_dim, head_dim_v;
    float scale;
    int causal;
    fa_dtype dtype, v_dtype;
    const float *qd, *kd, *vd;
    long long ds_b, ds_h;
    const int32_t* seqused_k;   // key/value cache: filled lengths (device, [batch])
    int seqused_add;            //   + the rows appended by this call
    const void *k_new, *v_new;  // rows to append first (n_new of them per sequence)
    int n_new;
    void* workspace;
    size_t workspace_bytes;
    void* stream;
    bool cta_pair;              // run the CTA-pair (cta_group::2) kernel
};

fa_status fwd_impl(const FwdArgs& a) {
    // ---------------------------------------------------------------- validation
    const bool varlen = a.cu_q != nullptr || a.cu_k != nullptr;
    const bool fp8 = a.dtype == FA_DTYPE_E4M3;
    // with no key rows at all (fixed length seqlen_k == 0, or varlen total 0) K and V may be NULL
    const bool no_keys = a.seqlen_k == 0;
    if (!a.q || !a.o || !a.lse || (!no_keys && (!a.k || !a.v)))
        return fail(FA_ERR_INVALID_ARG, "q, k, v, o and lse must be non-NULL device pointers");
    if (!aligned16(a.q) || !aligned16(a.k) || !aligned16(a.v) || !aligned16(a.o) ||
        !aligned16(a.lse))
        return fail(FA_ERR_INVALID_ARG, "q, k, v, o and lse must be 16-byte aligned");
    if (a.batch < 0 || a.heads < 1 || a.seqlen_q < 0 || a.seqlen_k < 0)
        return fail(FA_ERR_INVALID_ARG, "need batch >= 0, heads >= 1, seqlen_q/k >= 0");
    if (a.heads_k < 1 || a.heads % a.heads_k != 0)
        return fail(FA_ERR_INVALID_ARG, "heads_k (%d) must be >= 1 and divide heads (%d)",
                    a.heads_k, a.heads);
    if (a.causal != 0 && a.causal != 1) return fail(FA_ERR_INVALID_ARG, "causal must be 0 or 1");
    if (!(a.scale > 0.0f) || !std::isfinite(a.scale))
        return fail(FA_ERR_INVALID_ARG, "softmax_scale must be finite and > 0");
    if (fp8 ? (a.v_dtype != FA_DTYPE_E4M3 && a.v_dtype != FA_DTYPE_E5M2)
            : a.v_dtype != FA_DTYPE_BF16)
        return fail(FA_ERR_INVALID_ARG, "v dtype %d does not go with q/k dtype %d",
                    (int)a.v_dtype, (int)a.dtype);
    if (!fp8 && (a.qd || a.kd || a.vd))
        return fail(FA_ERR_INVALID_ARG, "descale pointers are only meaningful for FP8 inputs");
    if ((a.qd && (reinterpret_cast<uintptr_t>(a.qd) & 3u)) ||
        (a.kd && (reinterpret_cast<uintptr_t>(a.kd) & 3u)) ||
        (a.vd && (reinterpret_cast<uintptr_t>(a.vd) & 3u)))
        return fail(FA_ERR_INVALID_ARG, "descale pointers must be 4-byte aligned");
    if (a.ds_b < 0 || a.ds_h < 0)
        return fail(FA_ERR_INVALID_ARG, "descale strides must be >= 0");
    if (varlen && (!a.cu_q || !a.cu_k))
        return fail(FA_ERR_INVALID_ARG, "cu_seqlens_q and cu_seqlens_k must both be given");
    if (varlen && (a.max_q < 0 || a.max_k < 0))
        return fail(FA_ERR_INVALID_ARG, "max_seqlen_q/k must be >= 0 for varlen");
    if (a.head_dim != a.head_dim_v)
        return fail(FA_ERR_UNSUPPORTED, "head_dim (%d) != head_dim_v (%d) is not built",
                    a.head_dim, a.head_dim_v);
    if (!fp8 && a.head_dim != 64 && a.head_dim != 128)
        return fail(FA_ERR_UNSUPPORTED, "bf16 head_dim %d not built (64, 128)", a.head_dim);
    if (fp8 && a.head_dim != 128)
        return fail(FA_ERR_UNSUPPORTED, "fp8 head_dim %d not built (128)", a.head_dim);
    if (a.cta_pair && (fp8 || a.head_dim != 128 || a.seqused_k || a.n_new > 0 || a.workspace))
        return fail(FA_ERR_UNSUPPORTED, "the CTA-pair kernel is built for bf16, head_dim 128, "
                                        "without caches or key splits");
    const long long rows_q = varlen ? a.seqlen_q : (long long)a.batch * a.seqlen_q;
    const long long rows_k = varlen ? a.seqlen_k : (long long)a.batch * a.seqlen_k;
    if (rows_q * a.heads * a.head_dim >= (1ll << 40) ||
        rows_k * a.heads_k * a.head_dim >= (1ll << 40))
        return fail(FA_ERR_INVALID_ARG, "tensor too large");
    if (rows_q >= (1ll << 31) || rows_k >= (1ll << 31))
        return fail(FA_ERR_INVALID_ARG, "row count must fit in int32");
    const int mq = varlen ? a.max_q : a.seqlen_q;
    const int mk = varlen ? a.max_k : a.seqlen_k;
    const bool append = a.n_new > 0;
    if (a.batch == 0 || ((rows_q == 0 || mq == 0) && !append)) return FA_OK;  // nothing to do

    int dev, sms;
    uint32_t* err;
    fa_status st = device_info(&dev, &sms, &err);
    if (st != FA_OK) return st;

    // ---------------------------------------------------------------- decomposition
    const int pack = a.cta_pair ? 1 : choose_pack(a.heads, a.heads_k, mq, varlen);
    int splits = 1;
    const bool stream = a.seqused_k && a.workspace && mq > 0 &&
                        use_stream_plan(a.batch, a.heads, a.heads_k, a.seqlen_q, a.seqlen_k, a.causal, sms);
    if (a.workspace && mq > 0 && !a.cta_pair) {
        // (varlen: the longest lengths decide, and the partial rows are laid out by sequence
        // with max_seqlen_q rows each; packed grouped-query tiles are not used for varlen)
        splits = stream   ? kStreamSlots
                 : varlen ? choose_splits(a.batch, a.heads, mq, mk, a.causal, sms)
                          : plan_splits(a.batch, a.heads, a.heads_k, a.seqlen_q, a.seqlen_k, a.causal, sms);
        const size_t need = workspace_bytes_for(splits, a.batch, a.heads, mq, a.head_dim_v);
        if (a.workspace_bytes < need)
            return fail(FA_ERR_WORKSPACE, "workspace holds %zu bytes, %zu needed",
                        a.workspace_bytes, need);
        if (!aligned16(a.workspace))
            return fail(FA_ERR_INVALID_ARG, "workspace must be 16-byte aligned");
    }
    FwdParams p{};
    p.o = a.o;
    p.lse = a.lse;
    p.cu_q = a.cu_q;
    p.cu_k = a.cu_k;
    p.q_descale = a.qd;
    p.k_descale = a.kd;
    p.v_descale = a.vd;
    p.descale_sb = a.ds_b;
    p.descale_sh = a.ds_h;
    p.seqused_k = a.seqused_k;
    p.seqused_add = a.seqused_add;
    p.err = err;
    p.sched = next_sched_slot(dev, static_cast<cudaStream_t>(a.stream));
    p.batch = a.batch;
    p.heads = a.heads;
    p.kv_group = a.heads / a.heads_k;
    p.pack = pack;
    p.pack_shift = 0;
    while ((1 << p.pack_shift) < pack) ++p.pack_shift;
    if ((1 << p.pack_shift) != pack) return fail(FA_ERR_INVALID_ARG, "internal: pack %d", pack);
    p.item_heads = a.heads / pack;
    p.seqlen_q = mq;
    p.seqlen_k = mk;
    p.total_q = varlen ? a.seqlen_q : 0;
    p.n_mpairs = ceil_div((long long)mq * pack, a.cta_pair ? 512 : 256);
    p.n_splits = splits;
    const int nblk = ceil_div(mk > 0 ? mk : 1, 128);
    p.blocks_per_split = splits > 1 ? ceil_div(nblk, splits) : (1 << 29);
    const long long n_items = (long long)p.n_mpairs * a.batch * p.item_heads * splits;
    if (n_items >= (1ll << 31)) return fail(FA_ERR_INVALID_ARG, "too many work items");
    p.n_items = (int)n_items;
    p.scale_log2 = a.scale * 1.4426950408889634f;
    p.causal = a.causal;
    p.varlen = varlen ? 1 : 0;
    p.greedy = varlen && !a.cta_pair ? 1 : 0;  // varlen item costs are unknown on the host
    p.split = splits > 1 ? 1 : 0;
    p.stream = stream ? 1 : 0;
    if (stream) p.n_items = 1;  // pieces are published as index 0, the end as index 1
    p.v_e5m2 = a.v_dtype == FA_DTYPE_E5M2 ? 1 : 0;
    if (p.split) {
        const size_t rows = (size_t)splits * a.batch * a.heads * mq;
        p.ws_o = static_cast<float*>(a.workspace);
        p.ws_lse = p.ws_o + rows * a.head_dim_v;
    }
    int steady_mode = 0;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        p.wait_limit_ns = g_wait_limit_ns;
        p.inject = g_inject;
        p.trace = g_trace;
        steady_mode = g_steady_mode;
    }

    // ---------------------------------------------------------------- tensor maps
    CUtensorMap tq, tk, tv;
    // fixed length: (d, head, seq row, batch); varlen: (d, head, packed row, 1)
    const int nbat = varlen ? 1 : a.batch;
    // packed: one box spans the group's `pack` heads x 128 / pack rows, which lands in
    // shared memory as 128 tile rows ordered (query row, head)
    if ((st = encode_map(&tq, a.q, fp8, a.head_dim, a.heads, a.seqlen_q, nbat, pack)) != FA_OK)
        return st;
    if (no_keys) {  // no key block is ever loaded; any valid map will do
        tk = tq;
        tv = tq;
    } else {
        if ((st = encode_map(&tk, a.k, fp8, a.head_dim, a.heads_k, a.seqlen_k, nbat, 1,
                             a.cta_pair ? 64 : 0)) != FA_OK)
            return st;
        if ((st = encode_map(&tv, a.v, fp8, a.head_dim, a.heads_k, a.seqlen_k, nbat)) != FA_OK)
            return st;
    }

    // O (bf16) is stored by TMA from 128-row staging tiles: the same 4-D view and box as Q
    CUtensorMap to;
    if ((st = encode_map(&to, a.o, false, a.head_dim_v, a.heads, a.seqlen_q, nbat, pack)) != FA_OK)
        return st;

    // ---------------------------------------------------------------- launches
    cudaStream_t s = static_cast<cudaStream_t>(a.stream);
    cudaError_t e;
    // Few new rows (decoding): written by the forward kernel's producers, each the rows in
    // the key blocks it loads, right before loading them -- no copy kernel.  Otherwise a
    // copy kernel runs first on the same stream.
    const bool fused_append = append && rows_q > 0 && mq > 0 && a.n_new <= 4;
    if (fused_append) {
        p.k_cache = const_cast<void*>(a.k);
        p.v_cache = const_cast<void*>(a.v);
        p.k_new = a.k_new;
        p.v_new = a.v_new;
        p.append_rows = a.n_new;
    }
    if (append && !fused_append) {  // the new rows go into the cache first (ordered before the reads)
        const long long row_bytes = (long long)a.heads_k * a.head_dim * (fp8 ? 1 : 2);
        e = launch_append_kv(const_cast<void*>(a.k), const_cast<void*>(a.v), a.k_new, a.v_new,
                             a.seqused_k, a.batch, a.seqlen_k, a.n_new, row_bytes, err, s);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "append launch: %s", cudaGetErrorString(e));
    }
    if (rows_q == 0 || mq == 0) return FA_OK;
    if (a.cta_pair) {
        int pairs = 0;
        if ((st = resident_pairs(dev, &pairs)) != FA_OK) return st;
        const int grid2 = 2 * (int)(n_items < pairs ? n_items : pairs);
        set_item_bands(p, grid2 / 2);
        e = launch_fwd_pair_bf16_d128(tq, tk, tv, to, p, grid2, s);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
        return FA_OK;
    }
    const int grid = stream ? sms : (int)(n_items < sms ? n_items : sms);
    set_item_bands(p, grid);
    set_half_tail(p, grid);
    const bool cache = a.seqused_k != nullptr;  // the kernel instance with the cache code
    // the instance with packed variable-length batches (and debug injection)
    const bool var = p.varlen || p.inject != 0u;
    // Long bf16 D = 128 launches (fixed length or varlen) take the instance whose issuer runs the middle
    // key blocks of an item without per-block tests.  Its extra code is fetched from DRAM on
    // every launch after an L2 flush, so it pays off only over enough (tile, key block)
    // steps per CTA (kSteadyMinTileBlocksPerCta).
    // (varlen: from the longest sequence's lengths, an upper bound)
    const double tile_blocks = (double)a.batch * p.item_heads * (double)ceil_div((long long)mq * pack, 128) *
                               (double)nblk * (a.causal ? 0.5 : 1.0);
    const bool steady = !fp8 && a.head_dim == 128 && p.inject == 0u && !cache && steady_mode >= 0 &&
                        (steady_mode == 1 || tile_blocks >= kSteadyMinTileBlocksPerCta * (double)grid);
    if (fp8)
        e = launch_fwd_e4m3_d128(tq, tk, tv, to, p, grid, s, append && !fused_append, cache, var);
    else if (a.head_dim == 64)
        e = launch_fwd_bf16_d64(tq, tk, tv, to, p, grid, s, append && !fused_append, cache, var);
    else
        e = launch_fwd_bf16_d128(tq, tk, tv, to, p, grid, s, append && !fused_append, cache, var, steady);
    if (e != cudaSuccess) return fail(FA_ERR_CUDA, "forward launch: %s", cudaGetErrorString(e));
    if (p.split) {
        e = launch_combine(p.ws_o, p.ws_lse, a.o, a.lse, a.batch, a.heads, mq, a.head_dim_v, splits,
                           varlen ? a.cu_q : nullptr, varlen ? a.seqlen_q : 0, s);
        if (e != cudaSuccess) return fail(FA_ERR_CUDA, "combine launch: %s", cudaGetErrorString(e));
    }
    return FA_OK;
}

fa_status set_error_detail(fa_status status, const char* msg) { return fail(status, "%s", msg); }

unsigned long long current_context_id() {
    std::lock_guard<std::mutex> lk(g_mu);
    if (resolve_driver_entries() != FA_OK) return 0;
    return context_id_locked();
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
    case FA_ERR_DEVICE_ARG: return "device-resident length out of range";
    }
    return "unknown status";
}

const char* fa_last_error_detail(void) { return t_detail; }

void fa_debug_set(uint64_t wait_limit_ns, uint32_t inject) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_wait_limit_ns = wait_limit_ns ? wait_limit_ns : kDefaultWaitNs;
    g_inject = inject;
}

void fa_debug_select_steady(int mode) {
    std::lock_guard<std::mutex> lk(g_mu);
    g_steady_mode = (mode == 1 || mode == -1) ? mode : 0;
}

fa_status fa_debug_trace(void* buf, size_t bytes) {
#ifdef FA_TRACE
    if (buf && (bytes < kTraceBytes || !aligned16(buf)))
        return fail(FA_ERR_INVALID_ARG, "trace buffer needs %zu bytes, 16-byte aligned", kTraceBytes);
    std::lock_guard<std::mutex> lk(g_mu);
    g_trace = static_cast<uint64_t*>(buf);
    return FA_OK;
#else
    (void)buf;
    (void)bytes;
    return fail(FA_ERR_UNSUPPORTED, "this library was built without FA_TRACE");
#endif
}

size_t fa_debug_trace_bytes(void) { return kTraceBytes; }

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
    if (w & kErrBadLength)
        return fail(FA_ERR_DEVICE_ARG, "a cache length was out of range (rows computed with it clamped)");
    return FA_OK;
}

int fa_fwd_num_splits_gqa(int batch, int heads, int heads_k, int seqlen_q, int seqlen_k,
                          int causal) {
    int dev, sms;
    uint32_t* err;
    if (batch < 1 || heads < 1 || seqlen_q < 1 || seqlen_k < 1) return 1;
    if (heads_k < 1 || heads % heads_k != 0) return 1;
    if (device_info(&dev, &sms, &err) != FA_OK) return 1;
    return plan_splits(batch, heads, heads_k, seqlen_q, seqlen_k, causal, sms);
}

int fa_fwd_num_splits(int batch, int heads, int seqlen_q, int seqlen_k, int causal) {
    return fa_fwd_num_splits_gqa(batch, heads, heads, seqlen_q, seqlen_k, causal);
}

size_t fa_fwd_workspace_size_gqa(int batch, int heads, int heads_k, int seqlen_q, int seqlen_k,
                                 int head_dim_v, int causal) {
    const int s = fa_fwd_num_splits_gqa(batch, heads, heads_k, seqlen_q, seqlen_k, causal);
    if (head_dim_v < 1) return 0;
    // also enough for a packed varlen batch whose longest sequences have these lengths
    int sv = 1, dev, sms;
    uint32_t* err;
    if (batch >= 1 && heads >= 1 && seqlen_q >= 1 && seqlen_k >= 1 &&
        device_info(&dev, &sms, &err) == FA_OK)
        sv = choose_splits(batch, heads, seqlen_q, seqlen_k, causal, sms);
    const size_t fixed = workspace_bytes_for(s, batch, heads, seqlen_q, head_dim_v);
    const size_t packed = workspace_bytes_for(sv, batch, heads, seqlen_q, head_dim_v);
    return fixed > packed ? fixed : packed;
}

int fa_fwd_kvcache_num_splits(int batch, int heads, int heads_k, int seqlen_q, int cache_capacity,
                              int causal) {
    int dev, sms;
    uint32_t* err;
    if (batch < 1 || heads < 1 || seqlen_q < 1 || cache_capacity < 1) return 1;
    if (heads_k < 1 || heads % heads_k != 0) return 1;
    if (device_info(&dev, &sms, &err) != FA_OK) return 1;
    if (use_stream_plan(batch, heads, heads_k, seqlen_q, cache_capacity, causal, sms)) return kStreamSlots;
    return plan_splits(batch, heads, heads_k, seqlen_q, cache_capacity, causal, sms);
}

size_t fa_fwd_kvcache_workspace_size(int batch, int heads, int heads_k, int seqlen_q,
                                     int cache_capacity, int head_dim, int causal) {
    const int s = fa_fwd_kvcache_num_splits(batch, heads, heads_k, seqlen_q, cache_capacity, causal);
    if (head_dim < 1) return 0;
    return workspace_bytes_for(s, batch, heads, seqlen_q, head_dim);
}

size_t fa_fwd_workspace_size(int batch, int heads, int seqlen_q, int seqlen_k, int head_dim_v,
                             int causal) {
    return fa_fwd_workspace_size_gqa(batch, heads, heads, seqlen_q, seqlen_k, head_dim_v, causal);
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
    if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_E4M3)
        return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
    a.batch = batch; a.heads = heads; a.heads_k = heads_k;
    a.seqlen_q = seqlen_q; a.seqlen_k = seqlen_k;
    a.cu_q = cu_seqlens_q; a.cu_k = cu_seqlens_k;
    a.max_q = max_seqlen_q; a.max_k = max_seqlen_k;
    a.head_dim = head_dim; a.head_dim_v = head_dim_v;
    a.scale = softmax_scale; a.causal = causal;
    a.dtype = dtype; a.v_dtype = dtype;
    a.qd = q_descale; a.kd = k_descale; a.vd = v_descale;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.stream = stream;
    return fwd_impl(a);
}

fa_status fa_fwd_2cta(const void* q, const void* k, const void* v, void* o, float* lse, int batch,
                      int heads, int heads_k, int seqlen_q, int seqlen_k,
                      const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int max_seqlen_q,
                      int max_seqlen_k, int head_dim, float softmax_scale, int causal,
                      void* stream) {
    t_detail[0] = '\0';
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
    a.batch = batch; a.heads = heads; a.heads_k = heads_k;
    a.seqlen_q = seqlen_q; a.seqlen_k = seqlen_k;
    a.cu_q = cu_seqlens_q; a.cu_k = cu_seqlens_k;
    a.max_q = max_seqlen_q; a.max_k = max_seqlen_k;
    a.head_dim = head_dim; a.head_dim_v = head_dim;
    a.scale = softmax_scale; a.causal = causal;
    a.dtype = FA_DTYPE_BF16; a.v_dtype = FA_DTYPE_BF16;
    a.stream = stream;
    a.cta_pair = true;
    return fwd_impl(a);
}

fa_status fa_fwd_fp8(const void* q, const void* k, const void* v, void* o, float* lse, int batch,
                     int heads, int heads_k, int seqlen_q, int seqlen_k,
                     const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k, int max_seqlen_q,
                     int max_seqlen_k, int head_dim, float softmax_scale, int causal,
                     fa_dtype v_dtype, const float* q_descale, const float* k_descale,
                     const float* v_descale, int64_t descale_stride_b, int64_t descale_stride_h,
                     void* workspace, size_t workspace_bytes, void* stream) {
    t_detail[0] = '\0';
    FwdArgs a{};
    a.q = q; a.k = k; a.v = v; a.o = o; a.lse = lse;
    a.batch = batch; a.heads = heads; a.heads_k = heads_k;
    a.seqlen_q = seqlen_q; a.seqlen_k = seqlen_k;
    a.cu_q = cu_seqlens_q; a.cu_k = cu_seqlens_k;
    a.max_q = max_seqlen_q; a.max_k = max_seqlen_k;
    a.head_dim = head_dim; a.head_dim_v = head_dim;
    a.scale = softmax_scale; a.causal = causal;
    a.dtype = FA_DTYPE_E4M3; a.v_dtype = v_dtype;
    a.qd = q_descale; a.kd = k_descale; a.vd = v_descale;
    a.ds_b = descale_stride_b; a.ds_h = descale_stride_h;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.stream = stream;
    return fwd_impl(a);
}

fa_status fa_fwd_kvcache(const void* q, void* k_cache, void* v_cache, const void* k_new,
                         const void* v_new, void* o, float* lse, int batch, int heads, int heads_k,
                         int seqlen_q, int cache_capacity, const int32_t* cache_seqlens,
                         int seqlen_new, int head_dim, float softmax_scale, int causal,
                         fa_dtype dtype, fa_dtype v_dtype, const float* q_descale,
                         const float* k_descale, const float* v_descale,
                         int64_t descale_stride_b, int64_t descale_stride_h, void* workspace,
                         size_t workspace_bytes, void* stream) {
    t_detail[0] = '\0';
    if (!k_cache || !v_cache || !cache_seqlens)
        return fail(FA_ERR_INVALID_ARG, "k_cache, v_cache and cache_seqlens must be non-NULL");
    if (cache_capacity < 1 || seqlen_new < 0 || seqlen_new > cache_capacity)
        return fail(FA_ERR_INVALID_ARG, "need cache_capacity >= 1 and 0 <= seqlen_new <= capacity");
    if (seqlen_new > 0 && (!k_new || !v_new))
        return fail(FA_ERR_INVALID_ARG, "k_new and v_new must be given when seqlen_new > 0");
    if (seqlen_new > 0 && (!aligned16(k_new) || !aligned16(v_new)))
        return fail(FA_ERR_INVALID_ARG, "k_new and v_new must be 16-byte aligned");
    if ((reinterpret_cast<uintptr_t>(cache_seqlens) & 3u) != 0)
        return fail(FA_ERR_INVALID_ARG, "cache_seqlens must be 4-byte aligned");
    if (dtype != FA_DTYPE_BF16 && dtype != FA_DTYPE_E4M3)
        return fail(FA_ERR_INVALID_ARG, "unknown dtype %d", (int)dtype);
    FwdArgs a{};
    a.q = q; a.k = k_cache; a.v = v_cache; a.o = o; a.lse = lse;
    a.batch = batch; a.heads = heads; a.heads_k = heads_k;
    a.seqlen_q = seqlen_q; a.seqlen_k = cache_capacity;
    a.head_dim = head_dim; a.head_dim_v = head_dim;
    a.scale = softmax_scale; a.causal = causal;
    a.dtype = dtype; a.v_dtype = v_dtype;
    a.qd = q_descale; a.kd = k_descale; a.vd = v_descale;
    a.ds_b = descale_stride_b; a.ds_h = descale_stride_h;
    a.seqused_k = cache_seqlens; a.seqused_add = seqlen_new;
    a.k_new = k_new; a.v_new = v_new; a.n_new = seqlen_new;
    a.workspace = workspace; a.workspace_bytes = workspace_bytes;
    a.stream = stream;
    return fwd_impl(a);
}

}  // extern "C"
