// fa_fwd_kernel.cuh -- the attention forward kernel for GB300 (sm_103a).
//
// Method (exact attention, computed block by block with an online softmax,
// so S and P never leave the SM): "FlashAttention: Fast and Memory-Efficient
// Exact Attention with IO-Awareness" (arXiv:2205.14135), as its forward pass
// is walked through on the page "FlashAttention core algorithm: forward
// pass" (inference.lei6393.com, flash_fwd_kernel_sm90.h excerpts):
//   * a persistent tile-scheduler loop whose next work item is known before
//     the epilogue runs (scheduler loop and "get_next_work before the
//     epilogue" excerpts);
//   * a producer that loads Q once per item and streams K/V blocks through
//     full/empty pipelines (SharedStorage / PipelineStorage excerpt);
//   * consumers that run the two GEMMs and the softmax with exp2 and a
//     pre-multiplied softmax_scale_log2, FP8 descales folded into that scale,
//     a running row maximum and row_sum, iterating key blocks from
//     n_block_max - 1 down to n_block_min;
//   * an epilogue that stores O and LSE, or zeros and -inf (store_zero).
// The page "Dissecting the SM_120 Microarchitecture" (section 11.2, Fig. 12)
// finds the softmax (exp2 on the SFU) rather than the MMAs to dominate a
// key block on a GPU without TMEM, and lists overlapping MMA with softmax
// across warps and keeping accumulators in Tensor Memory as the remedies;
// both are the structure of this kernel.
//
// GB300 design (not a port of the pages' SM80/SM90 kernels):
//   * 384 threads, one CTA per SM (persistent, grid = #SMs):
//       warp 0      TMA producer (one elected thread)
//       warp 1      TMEM allocator and tcgen05.mma issuer (one elected thread)
//       warps 4-7   softmax + lazy correction + epilogue for query tile 0
//       warps 8-11  the same for query tile 1
//   * a work item is (batch, head, 256 query rows = two 128-row tiles, key
//     split); both tiles consume every K/V block loaded, halving K/V traffic;
//     for short query blocks of grouped-query attention an item is (batch, K/V
//     head, ...) and the group's query heads share the tile rows (row = query
//     row x head), so a K/V block is streamed once per K/V head;
//   * S_t = Q_t K^T and O_t += P_t V are tcgen05.mma (M=128) with fp32
//     accumulators in TMEM: S_t at columns [128t, 128t+128), O_t at
//     [256+128t, 256+128t+Dv); P_t (bf16 or e4m3) is written back over the
//     first columns of S_t and fed to the PV MMA straight from TMEM;
//   * the MMA issue order per key block j (reverse order) is
//       PV_0(j), S_0(j-1), PV_1(j), S_1(j-1)
//     so the tensor pipe works on one tile while the other tile's softmax
//     runs (ping-pong); the tensor pipe executes one thread's MMAs in issue
//     order, so S_t(j-1) overwriting P_t(j) after PV_t(j) is safe, and S_t(j)
//     being complete implies PV_t(j+1) is complete -- which is what lets the
//     softmax warps rescale O_t in place (lazily, only when the running max
//     grows by more than 2^16 for bf16 P, 2^8 for e4m3 P) without a separate
//     correction warpgroup;
//   * the MMA issuer is one thread whose bookkeeping between MMA batches is kept
//     minimal (compile-time tile indices, phase bits in registers, descriptors
//     built once): measured, a second issuer thread per tile interleaving MMA
//     streams is slower, and so is moving part of exp2 to the FMA pipe -- on
//     GB300 the MUFU is not the limit;
//   * the producer decides each CTA's next item (static LPT snake for fixed
//     length, a device-wide counter for varlen), decodes it once and hands the
//     decoded record to the other roles through a two-entry ring in shared memory,
//     before the current item's epilogue;
//   * static schedules run their items in L2 bands: several consecutive query
//     tile pairs of one (batch, head) side by side (all of them without a causal
//     mask; a band sized to keep the snake balanced, then plain LPT, under one),
//     so the CTAs running at one time read few heads' K/V and find it in L2;
//     without a causal mask, a last round holding at most half as many pairs as
//     CTAs runs its pairs as single tiles, two items each;
//   * key/value-cache launches with few, long items (decoding) use a balanced
//     plan instead: every producer reads the cache lengths, and each CTA takes
//     an equal share of the key blocks of all items, concatenated, as pieces
//     that leave partial results in their own slots (merged by the LSE identity
//     in a second, programmatically dependent kernel);
//   * up to 4 new cache rows per sequence are written into the caches by the
//     producers themselves (each the rows inside a key block it loads, just
//     before loading it), so a decoding step needs no copy kernel;
//   * the epilogue reads O out of TMEM (normalised, packed to bf16) and returns the
//     TMEM columns to the MMA issuer at once, then writes O out through a
//     128-byte-swizzled staging tile with TMA stores (plain stores only where a
//     varlen tile crosses its sequence end, and for the fp32 split partials);
//   * every wait is bounded by wall clock; a timeout sets the device error
//     word and all roles abandon the launch cleanly (TMEM released);
//   * CTA-pair variant (PAIR, bf16, D = 128): a cluster of two CTAs on two SMs
//     runs M = 256 tcgen05 MMAs (cta_group::2) issued by one thread of the even
//     CTA; a work item is 512 query rows, each of the pair's two MMA row slots
//     covering 256 rows (128 in each CTA).  Each CTA loads its own halves of the
//     operands -- its Q rows, keys [64r, 64r+64) of every K block and head-dim
//     columns [64r, 64r+64) of every V block -- so each SM streams half of each
//     K/V block through shared memory; the loads complete on the even CTA's
//     barriers, MMA completions are multicast to both CTAs, and the odd CTA's
//     softmax warps hand P back to the even CTA's barrier.
#pragma once

#include <cuda_bf16.h>

#include <atomic>
#include <type_traits>

#include "fa_internal.h"
#include "sm103_ptx.cuh"

namespace fa {
constexpr int kBM = 128;          // query rows per tile (one TMEM lane per row)
constexpr int kBN = 128;          // keys per K/V block
constexpr int kTiles = 2;         // query tiles per work item
constexpr int kThreads = 384;
constexpr uint32_t kTmemCols = 512;
// Pairs (of every 16) of exp2 evaluated on the FMA pipe instead of the MUFU, in
// blocks without masking.  0 by default: on GB300 the MUFU keeps up (measured), and
// the extra instructions only lengthen the softmax; kept as a build option.
#ifndef FA_EXP2_EMU_PAIRS
#define FA_EXP2_EMU_PAIRS 0
#endif
// Lazy-rescale threshold (log2 units): P stays <= 2^tau.  e4m3 P must stay below its
// 448 maximum; bf16 P has fp32's exponent range, so a larger threshold only trades
// (rare) rescales for larger -- still exactly representable -- P values.
template <bool FP8>
__host__ __device__ constexpr float lazy_tau() { return FP8 ? 8.0f : 16.0f; }

// exp2 on the FMA pipe (for part of the columns, relieving the MUFU): Cody-Waite
// style range reduction x = n + f with n = round(x), |f| <= 1/2, then 2^f by a
// degree-3 polynomial, minimax in relative error on [-1/2, 1/2] (coefficients
// derived by linear programming in exact_attention_forward_gb300/exp2_poly.py;
// max relative error 7.5e-5, below bf16's 2^-9 rounding of P), and 2^n added to
// the exponent field.  Inputs are clamped to >= -125 so the result stays normal.
constexpr float kExp2C0 = 0.9999279975891113f;
constexpr float kExp2C1 = 0.6932609677314758f;
constexpr float kExp2C2 = 0.2426113784313202f;
constexpr float kExp2C3 = 0.05517187342047691f;
constexpr float kRoundMagic = 12582912.0f;  // 1.5 * 2^23: x + magic rounds x to an integer

// Optional event trace (built with -DFA_TRACE; without it every hook below compiles to
// nothing).  kTraceCtas CTAs spread over the grid (slot k: CTA k * (grid - 1) /
// (kTraceCtas - 1)) log (tag << 56 | clock64) words per role -- 0 the producer, 1 the MMA
// issuer, 2 + t the first thread of tile t's softmax warps -- into
// p.trace[(slot * kTraceRoles + role) * kTraceCap + i], up to kTraceCap events each.  Tags:
//   producer: 1 item start, 2 + t Q_EMPTY[t] passed, 4 K/V group issued, 5 next item published
//   issuer:   1 item read, 2 Q ready, 3 K/V group ready, 4 + t P[t] ready, 6 + t tile t's
//             MMAs of a block issued, 8 item done; just before the K/V-group and P waits,
//             11 / 12 the group had / had not landed, 13 / 14 P was / was not handed over
//   softmax:  1 item read, 2 S ready, 3 P handed over, 4 O ready, 5 O released (TMEM),
//             6 epilogue done; within a block, 7 S in registers, 8 max and rescale done,
//             9 exponentials done, 10 P stored to TMEM
//   every role, first and last: 15 %globaltimer (ns), then 14 clock64 -- ties the SM's
//   cycle count to wall time across SMs
struct Tracer {
#ifdef FA_TRACE
    uint64_t* buf = nullptr;
    uint32_t n = 0;
    __device__ __forceinline__ void init(uint64_t* base, int role) {
        // traced CTAs spread over the grid: slot k is CTA k * (grid - 1) / (kTraceCtas - 1)
        const int g1 = (int)gridDim.x - 1, c = (int)blockIdx.x;
        const int k = g1 > 0 ? (c * (kTraceCtas - 1) + g1 / 2) / g1 : 0;
        const bool on = base && k < kTraceCtas && (g1 > 0 ? k * g1 / (kTraceCtas - 1) : 0) == c;
        buf = on ? base + ((size_t)k * kTraceRoles + role) * kTraceCap : nullptr;
        fin();
    }
    __device__ __forceinline__ void fin() {
        if (buf && n + 2 <= (uint32_t)kTraceCap) {
            buf[n++] = (15ull << 56) | (globaltimer_ns() & 0xFFFFFFFFFFFFFFull);
            buf[n++] = (14ull << 56) | (clock64() & 0xFFFFFFFFFFFFFFull);
        }
    }
    __device__ __forceinline__ void ev(uint32_t tag) {
        if (buf && n < (uint32_t)kTraceCap) buf[n++] = ((uint64_t)tag << 56) | (clock64() & 0xFFFFFFFFFFFFFFull);
    }
#else
    __device__ __forceinline__ void init(uint64_t*, int) {}
    __device__ __forceinline__ void fin() {}
    __device__ __forceinline__ void ev(uint32_t) {}
#endif
};

// Register split: launched at 168 per thread (384 x 168 = 64512); the producer /
// MMA warpgroup gives up 64 per thread, the two softmax warpgroups take 32 more.
constexpr uint32_t kRegsLoadMma = 104;
constexpr uint32_t kRegsSoftmax = 200;
static_assert(128 * kRegsLoadMma + 256 * kRegsSoftmax <= 384 * 168, "register split exceeds launch");

template <int D, bool FP8, bool PAIR = false>
struct Cfg {
    static_assert(!PAIR || (!FP8 && D == 128), "the CTA-pair variant is built for bf16, D = 128");
    static constexpr int kElem = FP8 ? 1 : 2;
    static constexpr int kRowBytes = D * kElem;
    static constexpr int kChunks = kRowBytes / 128;        // 128-byte swizzle atoms per row
    static constexpr int kChunkElems = 128 / kElem;
    static constexpr int kChunkBytes = kBM * 128;          // one atom column of a tile: 16 KiB
    static constexpr int kTileBytes = kBM * kRowBytes;     // Q tile == K/V block (BM == BN)
    static constexpr int kUmmaK = 32 / kElem;              // reduction depth of one MMA
    // a K/V ring slot holds one K or V block, or (CTA pair) this CTA's half of one:
    // 64 keys of K, or 64 head-dim columns of V
    static constexpr int kSlotBytes = PAIR ? kTileBytes / 2 : kTileBytes;
    static constexpr int kKChunkBytes = PAIR ? kBN / 2 * 128 : kChunkBytes;  // atom column of a K slot
    static constexpr int kStages = (FP8 || D == 64 || PAIR) ? 8 : 4;
    static constexpr int kPCols = kBN * kElem / 4;         // TMEM columns of a P tile
    static constexpr int kQOff = 0;
    static constexpr int kKVOff = kTiles * kTileBytes;
    // epilogue staging: per tile, 128 rows x 64 bf16 columns of O (one 128-byte swizzle atom
    // wide), stored to HBM by TMA; a D = 128 tile goes out in two halves
    static constexpr int kStageBytes = kBM * 128;
    static constexpr int kStageOff = kKVOff + kStages * kSlotBytes;
    static constexpr int kBarOff = kStageOff + kTiles * kStageBytes;
    enum {
        Q_FULL = 0, Q_EMPTY = 2, S_FULL = 4, P_FULL = 6, O_FULL = 8, O_EMPTY = 10, STG_FULL = 12,
        STG_EMPTY = 14, ITEM_FULL = 16, ITEM_EMPTY = 18, DRAIN = 20, KV_FULL = 21,
        KV_EMPTY = 21 + kStages, NUM_BARS = 21 + 2 * kStages
    };
    static constexpr int kMiscOff = kBarOff + NUM_BARS * 8;
    // misc: TMEM address, abort flag, item ring indices (16 B); then the two decoded item
    // records of the ring (64 B each, 16-byte aligned)
    static constexpr int kItemRecOff = (kMiscOff + 16 + 15) / 16 * 16;
    // balanced cache plan: the batch's clamped cache lengths (<= 64 sequences), producer only
    static constexpr int kLenOff = kItemRecOff + 2 * 64;
    static constexpr int kMaxPlanBatch = 64;
    static constexpr int kSmemBytes = kLenOff + kMaxPlanBatch * 4 + 1024;  // + slack to align the base to 1 KiB
    static constexpr int kMmaM = PAIR ? 2 * kBM : kBM;  // rows of one MMA (both CTAs of a pair)
    static constexpr uint32_t kIdescQK = make_idesc(kMmaM, kBN, 0u + (FP8 ? 0u : 1u), false);
    static constexpr uint32_t kIdescPV = make_idesc(kMmaM, D, 0u + (FP8 ? 0u : 1u), true);
    // FP8 with an E5M2 V: P (A operand) stays E4M3, B = V is E5M2 (kind::f8f6f4 codes 0 / 1)
    static constexpr uint32_t kIdescPV5 = make_idesc2(kBM, D, 0u, 1u, true);
    static constexpr uint32_t kColO = 256;
    static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte swizzle atoms");
    static_assert(kSmemBytes <= 232448, "exceeds the 227 KiB per-block shared memory");
    static_assert(kSmemBytes > 232448 / 2, "must keep one CTA (and one 512-column TMEM) per SM");
};

// One unit of work: a pair of 128-row query tiles of one (batch, head) and a
// range of key blocks.  Decoded identically by every role from its index.  In a CTA
// pair an item is two 256-row MMA slots; m0 is then this CTA's half of slot t, and the
// key ranges and `active` belong to the slot (both CTAs visit the same blocks).
struct Item {
    int b, h, split;
    int sq, sk;          // this sequence's lengths
    int q_row0, k_row0;  // first row of this sequence in the packed / fixed tensors
    int m0[kTiles];      // first query row (within the sequence) of each tile
    int n_lo, n_hi;      // key blocks [n_lo, n_hi) are visited, in reverse
    int n_hi_t[kTiles];  // tile t visits [n_lo, n_hi_t[t]); none if n_hi_t[t] <= n_lo
    bool active[kTiles]; // tile t has at least one row inside the sequence
    bool bad_len;        // the per-sequence key length was out of range (clamped)
    int fill;            // balanced plan: partial slots after this piece's to mark empty
};

// Features that only the variable-length kernel instances carry (VAR = true): packed
// variable-length batches with their greedy hand-out, and debug injection.  With
// VAR = false the accessors return the defaults (fixed length, no injection) as
// compile-time constants, and the code behind them drops out.
template <bool VAR>
struct Var {
    static __device__ __forceinline__ bool varlen(const FwdParams& p) { return VAR && p.varlen; }
    static __device__ __forceinline__ uint32_t inject(const FwdParams& p) { return VAR ? p.inject : 0u; }
};

// Tile rows and visited key blocks [n_lo, n_hi_t[t]) of an item whose rows start at
// (packed) row mp * kTiles * kSlotRows and whose key range is [n_lo, n_end), under the
// causal mask when set (bottom-right aligned).
template <bool PAIR>
__device__ __forceinline__ void set_tile_ranges(const FwdParams& p, Item& it, int mp, int n_end,
                                                uint32_t rank) {
    constexpr int kSlotRows = PAIR ? 2 * kBM : kBM;  // query rows of one MMA row slot
    const int G = p.pack;
    it.n_hi = it.n_lo;
#pragma unroll
    for (int t = 0; t < kTiles; ++t) {
        const int s0 = mp * (kTiles * kSlotRows) + t * kSlotRows;  // first (packed) row of slot t
        it.m0[t] = s0 + (PAIR ? (int)rank * kBM : 0);               // ... of this CTA's tile
        it.active[t] = s0 < it.sq * G;
        int hi = n_end;
        if (p.causal) {
            const int rmax = (min(s0 + kSlotRows, it.sq * G) - 1) / G;  // last query row
            const int last = rmax + it.sk - it.sq;  // last visible key of the tile's last row
            hi = last < 0 ? 0 : min(hi, last / kBN + 1);
        }
        if (!it.active[t]) hi = it.n_lo;
        it.n_hi_t[t] = max(hi, it.n_lo);
        it.n_hi = max(it.n_hi, it.n_hi_t[t]);
    }
}

// Item index -> (pair level, batch, head, split).  Longest-processing-time order:
// pair index descending (under a causal mask later pairs see more key blocks), then
// (batch, head, split).  Taken level by level, the items running at one time span
// every (batch, head), whose K/V streams together outgrow L2.  So a static schedule
// may first run bands (set by the host): `band_levels` consecutive levels of one
// (batch, head, split), then the next (batch, head, split).  The host sizes a causal
// band so that the snake's paired rounds still balance (see fa_api.cu) and leaves the
// last levels, the small items, in plain LPT order.  Query heads sharing a K/V head
// (grouped-query attention) are consecutive items, so they stream the same K/V at
// about the same time and share it in L2.
template <bool PAIR, bool CACHE, bool VAR>
__device__ __forceinline__ Item decode_item(const FwdParams& p, int w, uint32_t rank) {
    using V = Var<VAR>;
    Item it;
    it.fill = 0;
    int half = -1;  // a single query tile (0 or 1) of a tile pair item, or -1: the pair
    if (!PAIR && p.half_from > 0 && w >= p.half_from) {
        const int d = w - p.half_from;
        half = d & 1;
        w = p.half_from + (d >> 1);
    }
    // packed grouped-query mode (p.pack = G > 1): an item serves one K/V head, and its
    // tile rows are (query row, query head of the group) pairs, row-major: packed row
    // r = i * G + g.  it.h is then the group's first query head.
    const int G = p.pack;
    const int per_m = p.batch * p.item_heads * p.n_splits;
    int level, r;  // level 0 = the last pair (the most key blocks under a causal mask)
    if (w < p.band_items) {  // band_levels consecutive levels of one (batch, head, split)
        const int per_band = p.band_levels * per_m;
        const int bi = w / per_band;
        const int rem = w - bi * per_band;
        r = rem / p.band_levels;
        level = bi * p.band_levels + (rem - r * p.band_levels);
    } else {  // level by level, all (batch, head, split) of a level together
        const int w2 = w - p.band_items;
        const int l2 = w2 / per_m;
        level = p.band_lv + l2;
        r = w2 - l2 * per_m;
    }
    const int mp = p.n_mpairs - 1 - level;
    it.split = r % p.n_splits;
    const int bh = r / p.n_splits;
    it.h = (bh % p.item_heads) * G;
    it.b = bh / p.item_heads;
    if (V::varlen(p)) {
        it.q_row0 = __ldg(p.cu_q + it.b);
        it.sq = __ldg(p.cu_q + it.b + 1) - it.q_row0;
        it.k_row0 = __ldg(p.cu_k + it.b);
        it.sk = __ldg(p.cu_k + it.b + 1) - it.k_row0;
    } else {
        it.q_row0 = it.b * p.seqlen_q;
        it.sq = p.seqlen_q;
        it.k_row0 = it.b * p.seqlen_k;
        it.sk = p.seqlen_k;
    }
    it.bad_len = false;
    if (CACHE && p.seqused_k) {  // a cache of capacity seqlen_k filled to this sequence's length
        const int u = __ldg(p.seqused_k + it.b) + p.seqused_add;
        it.bad_len = u < 0 || u > p.seqlen_k;
        it.sk = min(max(u, 0), p.seqlen_k);
    }
    const int nblk = (it.sk + kBN - 1) / kBN;
    it.n_lo = it.split * p.blocks_per_split;
    set_tile_ranges<PAIR>(p, it, mp, min(nblk, it.n_lo + p.blocks_per_split), rank);
    if (half >= 0) {  // run tile `half` alone, as tile 0; tile 1 does nothing
        if (half == 1) {
            it.m0[0] = it.m0[1];
            it.active[0] = it.active[1];
            it.n_hi_t[0] = it.n_hi_t[1];
        }
        it.active[1] = false;
        it.n_hi_t[1] = it.n_lo;
        it.n_hi = max(it.n_hi_t[0], it.n_lo);
    }
    return it;
}

// The producer decodes each item once and passes it to the other roles in a 64-byte
// shared-memory record (sixteen 32-bit words), next to the index in the item ring.
__device__ __forceinline__ void store_item(uint8_t* rec, int w, const Item& it) {
    int4* r = reinterpret_cast<int4*>(rec);
    const int flags = (it.active[0] ? 1 : 0) | (it.active[1] ? 2 : 0) | (it.bad_len ? 4 : 0);
    r[0] = make_int4(w, it.b, it.h, it.split);
    r[1] = make_int4(it.sq, it.sk, it.q_row0, it.k_row0);
    r[2] = make_int4(it.m0[0], it.m0[1], it.n_lo, it.n_hi);
    r[3] = make_int4(it.n_hi_t[0], it.n_hi_t[1], flags, it.fill);
}
__device__ __forceinline__ int load_item(const uint8_t* rec, Item& it) {
    const int4* r = reinterpret_cast<const int4*>(rec);
    const int4 a = r[0], b = r[1], c = r[2], d = r[3];
    it.b = a.y; it.h = a.z; it.split = a.w;
    it.sq = b.x; it.sk = b.y; it.q_row0 = b.z; it.k_row0 = b.w;
    it.m0[0] = c.x; it.m0[1] = c.y; it.n_lo = c.z; it.n_hi = c.w;
    it.n_hi_t[0] = d.x; it.n_hi_t[1] = d.y;
    it.active[0] = (d.z & 1) != 0; it.active[1] = (d.z & 2) != 0; it.bad_len = (d.z & 4) != 0;
    it.fill = d.w;
    return a.x;
}

// Which item a CTA takes next is decided by its producer thread, which passes the
// index to the MMA issuer and the softmax warps through a two-entry ring in shared
// memory (ITEM_FULL / ITEM_EMPTY mbarriers), published once the current item's loads
// are issued -- before the current item's epilogue.  CTA c starts with item c; then
//  * fixed length (item costs known from the index): a static snake -- round r hands
//    items [r*G, (r+1)*G) to the CTAs in forward order on even rounds and in reverse
//    order on odd ones, which balances the descending item costs;
//  * varlen (costs depend on lengths that live on the device): greedy -- the next index
//    comes from a device-wide counter (atomicAdd), so a CTA that finishes early takes
//    the next (in LPT order: the next most expensive) item.
constexpr uint32_t kItemConsumers = 1 + 2 * (kBM / 32);  // issuer + one arrival per softmax warp
// `unit`: this CTA (or CTA pair) among `nunits`
__device__ __forceinline__ int item_of_round(int round, int unit, int nunits) {
    const int pos = (round & 1) ? (nunits - 1 - unit) : unit;
    return round * nunits + pos;
}

struct WaitCtx {
    uint64_t limit_ns;
    uint32_t* err;
    volatile uint32_t* abort_flag;  // shared memory
};

// cluster: acquire at cluster scope (barriers that the peer CTA of a pair arrives on)
static __device__ __forceinline__ bool wait_slow(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                                 uint32_t site, bool honor_abort = true,
                                                 bool cluster = false) {
    const uint64_t t0 = globaltimer_ns();
    while (true) {
#pragma unroll 1
        for (int i = 0; i < 128; ++i)
            if (cluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity)) return true;
        if (honor_abort && *w.abort_flag) return false;
        if (globaltimer_ns() - t0 > w.limit_ns) {
            atomicCAS(w.err, 0u, kErrTimeout | (site << 8));
            atomicOr(w.err, kErrTimeout);
            *w.abort_flag = 1u;
            __threadfence_block();
            return false;
        }
    }
}
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                         uint32_t site) {
    if (mbar_try_wait(bar, parity)) return true;
    return wait_slow(bar, parity, w, site);
}
__device__ __forceinline__ bool wait_bar_cluster(uint32_t bar, uint32_t parity, const WaitCtx& w,
                                                 uint32_t site) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    return wait_slow(bar, parity, w, site, true, true);
}

// Wait-site codes reported in bits 8..15 of the error word.
enum : uint32_t {
    SITE_Q_EMPTY = 1, SITE_KV_EMPTY = 2, SITE_Q_FULL = 3, SITE_KV_FULL = 4, SITE_P_FULL = 5,
    SITE_O_EMPTY = 6, SITE_S_FULL = 7, SITE_O_FULL = 8, SITE_DRAIN = 9, SITE_STG_FULL = 10,
    SITE_STG_EMPTY = 11, SITE_ITEM_FULL = 12, SITE_ITEM_EMPTY = 13, SITE_LOAD_DRAIN = 14
};

// CACHE: the instance for key/value-cache calls (per-sequence cache lengths, new rows
// written by the producers, the balanced plan); the other instances hold none of that code
// -- measured, the smaller kernel starts its launches faster (causal 2K -8 %).
// VAR: the instance for packed variable-length batches (and debug injection); the
// fixed-length instance (VAR = false) leaves their code out -- measured, same-run A/B with
// bit-identical outputs: causal 2K -1 %, FP8 4K -1.3 %, short-q/long-k -1.5 %, a
// launch-bound B=1 H=2 S=256 call -15 to -24 %, the 8K shapes within +-0.6 %.  (Folding key
// splits and packed rows as well made the code smaller still but the 8K launches 1.4-4 %
// slower.)
// STEADY: the instance for long bf16 launches (fixed length or varlen), whose MMA issuer runs key
// blocks in the middle of an item (both tiles active, past their first PV) without the
// per-block tests of the edge blocks.  The single issuing thread paces the tensor pipe, so
// those tests cost time: same-run A/B, bit-identical outputs, causal and grouped-query 8K
// -4 %, non-causal 8K -4.7 %, and -1.4 to -1.9 % more once its MMA descriptors stopped
// spilling.  Its extra code (~9 KB, fetched from DRAM after every L2 flush) made short
// launches 1-3 % slower, so the host picks it by size.
template <int D, bool FP8, bool PAIR = false, bool CACHE = false, bool VAR = true, bool STEADY = false>
__global__ void __launch_bounds__(kThreads, 1)
    fa_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                  const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                  const FwdParams p) {
    using C = Cfg<D, FP8, PAIR>;
    using V = Var<VAR>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    const uint32_t s_base = smem_u32(smem);
    const uint32_t s_q = s_base + C::kQOff;
    const uint32_t s_kv = s_base + C::kKVOff;
    const uint32_t s_bar = s_base + C::kBarOff;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + C::kMiscOff);
    volatile uint32_t* abort_flag = reinterpret_cast<volatile uint32_t*>(smem + C::kMiscOff + 4);
    auto bar = [&](int i) -> uint32_t { return s_bar + 8u * (uint32_t)i; };

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    // CTA pair: rank 0 issues the MMAs and owns the barriers the pair's loads and P / O
    // hand-offs complete; `leader(b)` is that barrier's shared::cluster address
    const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
    // (the barrier array is contiguous in each CTA's window, so one mapping serves all)
    const uint32_t s_bar_lead = PAIR ? mapa_shared(s_bar, 0u) : s_bar;
    auto leader = [&](uint32_t b) -> uint32_t { return PAIR ? s_bar_lead + (b - s_bar) : b; };
    // the unit the static schedule hands items to: this CTA, or this CTA's pair
    const int unit = PAIR ? (int)cluster_id_x() : (int)blockIdx.x;
    const int nunits = PAIR ? (int)ncluster_x() : (int)gridDim.x;

    if (threadIdx.x == 0) {
        for (int t = 0; t < kTiles; ++t) {
            mbar_init(bar(C::Q_FULL + t), 1);
            mbar_init(bar(C::Q_EMPTY + t), 1);
            mbar_init(bar(C::S_FULL + t), 1);
            // one arrival per softmax warp (of both CTAs of a pair)
            mbar_init(bar(C::P_FULL + t), (PAIR ? 2 : 1) * kBM / 32);
            mbar_init(bar(C::O_FULL + t), 1);
            mbar_init(bar(C::O_EMPTY + t), (PAIR ? 2 : 1) * kBM / 32);
            mbar_init(bar(C::STG_FULL + t), kBM / 32);  // every warp of the tile wrote its rows
            mbar_init(bar(C::STG_EMPTY + t), 1);        // the store has read the staging rows
        }
        mbar_init(bar(C::DRAIN), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(C::ITEM_FULL + i), 1);
            mbar_init(bar(C::ITEM_EMPTY + i), kItemConsumers);
        }
        for (int s = 0; s < C::kStages; ++s) {
            mbar_init(bar(C::KV_FULL + s), 1);
            mbar_init(bar(C::KV_EMPTY + s), kTiles);  // one release per query tile
        }
        *abort_flag = 0u;
        fence_barrier_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        if constexpr (PAIR) {
            tmem_alloc_pair(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish_pair();
        } else {
            tmem_alloc(smem_u32(tmem_slot), kTmemCols);
            tmem_relinquish();
        }
        tc_fence_before();
    }
    // a pair's barriers are initialised before the other CTA's loads, commits or arrivals
    // can reach them
    if constexpr (PAIR) {
        __syncwarp();  // the .aligned cluster barrier wants converged warps
        cluster_sync();
    } else {
        __syncthreads();
    }
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const WaitCtx wc{p.wait_limit_ns, p.err, abort_flag};
    // consumer side of the item ring: the next item index (n_items = no more work)
    uint32_t items_read = 0;
    // (the index, and for an index below p.n_items the decoded item)
    auto read_item = [&](int& w, Item& it) -> bool {
        const uint32_t slot = items_read & 1u;
        if (!wait_bar(bar(C::ITEM_FULL + slot), (items_read >> 1) & 1u, wc, SITE_ITEM_FULL)) return false;
        w = load_item(smem + C::kItemRecOff + 64 * slot, it);
        ++items_read;
        return true;
    };

    if (warp < 4) {
    setmaxnreg_dec<kRegsLoadMma>();
    if (warp == 0) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_q);
            tma_prefetch_desc(&tm_k);
            tma_prefetch_desc(&tm_v);
            tma_prefetch_desc(&tm_o);
            // launched as a programmatic dependent of the cache append (key/value cache
            // calls): its writes are complete and visible before any load below; a no-op
            // for other launches
            asm volatile("griddepcontrol.wait;" ::: "memory");
            const uint64_t pol_q = l2_policy_evict_first();
            const uint64_t pol_kv = l2_policy_evict_last();
            Tracer tr;
            tr.init(p.trace, 0);
            uint32_t ring = 0, ph_qe = 0;  // bit t: parity of the last Q_EMPTY wait of tile t
            // loads in flight: bit t / s toggles whenever Q_FULL[t] / KV_FULL[s] is armed
            // (its phase parity), and stays set in the *_any masks once it has been armed
            uint32_t q_par = 0, q_any = 0, kv_par = 0, kv_any = 0;
            bool withheld = false;
            bool aborted = false;
            uint32_t published = 0;
            // a pair's two producers follow one static order (no device counter)
            const bool greedy = !PAIR && VAR && p.greedy;
            // decodes item w (an index below p.n_items) into `it` and publishes both; in the
            // greedy hand-out an item with no rows (a tile pair past a short sequence's end) is
            // passed over for the next ticket instead of going round the item ring (varlen
            // -3 %; not in the FP8 instance, whose code measured 2.3 % slower with it)
            auto publish = [&](int& w, Item& it) -> bool {
                const uint32_t slot = published & 1u;
                if (!(CACHE && p.stream)) {
                    while (w < p.n_items) {
                        it = decode_item<PAIR, CACHE, VAR>(p, w, rank);
                        if (FP8 || !greedy || it.active[0] || it.active[1]) break;
                        w = min((int)(gridDim.x + atomicAdd(p.sched, 1u)), p.n_items);
                    }
                }
                if (published >= 2 &&
                    !wait_bar(bar(C::ITEM_EMPTY + slot), ((published >> 1) - 1) & 1u, wc, SITE_ITEM_EMPTY))
                    return false;
                store_item(smem + C::kItemRecOff + 64 * slot, w, it);
                mbar_arrive(bar(C::ITEM_FULL + slot));  // release: the record is visible to waiters
                ++published;
                return true;
            };
            // Every CTA counts itself once when it will fetch no more (its last fetch, or an
            // abort); the last one returns the counter pair to zero for the next launch that
            // uses it -- by then no CTA of this launch touches the counter again.
            bool counted = false;
            auto fetching_done = [&]() {
                if (counted) return;
                counted = true;
                if (atomicAdd(p.sched + 1, 1u) == gridDim.x - 1) {
                    p.sched[0] = 0u;
                    p.sched[1] = 0u;
                }
            };
            // Balanced cache plan (p.stream): the key blocks of all items, concatenated in
            // (batch, item head) order, are cut into equal shares of T blocks, one per CTA:
            // this CTA runs the pieces of the items that overlap [lo_g, hi_g), each in its own
            // partial slot (the CTA index minus that of the item's first share), and finishes
            // the empty items whose position falls in its share (the last CTA any beyond).
            // T is at least a third of a full cache, so no item needs more than four slots.
            // (The plan is used where every row sees every key of its item -- non-causal, or
            // one query row -- so a piece always has work for its active tiles.)
            uint32_t* const plan_len = reinterpret_cast<uint32_t*>(smem + C::kLenOff);
            long long plan_T = 1, lo_g = 0, hi_g = 0, ppos = 0;
            int pb = 0, ph = 0;  // next item (batch, item head) of the walk, at block ppos
            if (CACHE && p.stream) {
                long long W = 0;
                for (int b = 0; b < p.batch; ++b) {
                    const int u = __ldg(p.seqused_k + b) + p.seqused_add;
                    const int L = min(max(u, 0), p.seqlen_k);
                    plan_len[b] = (uint32_t)L | ((u < 0 || u > p.seqlen_k) ? 0x80000000u : 0u);
                    W += (long long)((L + kBN - 1) / kBN) * p.item_heads;
                }
                const long long G = gridDim.x;
                const long long capblk = (p.seqlen_k + kBN - 1) / kBN;
                plan_T = max(max((W + G - 1) / G, (capblk + p.n_splits - 2) / (p.n_splits - 1)), 1LL);
                lo_g = (long long)blockIdx.x * plan_T;
                hi_g = min(lo_g + plan_T, W);
            }
            auto next_piece = [&](Item& it) -> bool {
                const long long G = gridDim.x, c = blockIdx.x, T = plan_T;
                while (pb < p.batch) {
                    const uint32_t rec = plan_len[pb];
                    const int L = (int)(rec & 0x7fffffffu);
                    const long long nb = (L + kBN - 1) / kBN;
                    if (ph == 0) {
                        // nothing from here on is this CTA's (the last CTA also owns any
                        // empty items beyond the total)
                        if (ppos >= (c + 1) * T && c != G - 1) return false;
                        // the whole sequence lies before this CTA's share, or is empty and
                        // owned by another CTA
                        if ((nb > 0 && ppos + nb * p.item_heads <= lo_g) ||
                            (nb == 0 && min(ppos / T, G - 1) != c)) {
                            ppos += nb * p.item_heads;
                            ++pb;
                            continue;
                        }
                    }
                    const int b = pb, h = ph;
                    const long long s0 = ppos;
                    ppos += nb;
                    if (++ph == p.item_heads) {
                        ph = 0;
                        ++pb;
                    }
                    if (nb == 0) {
                        // an empty cache (this CTA's to finish): every partial slot of the
                        // item's rows is marked empty, and the merge writes O = 0, LSE = -inf
                        const size_t slot_rows = (size_t)p.batch * p.heads * p.seqlen_q;
                        for (int prow = 0; prow < (p.seqlen_q << p.pack_shift); ++prow) {
                            const int hrow = h * p.pack + (prow & (p.pack - 1));
                            const size_t rid = ((size_t)b * p.heads + hrow) * p.seqlen_q + (prow >> p.pack_shift);
                            for (int k = 0; k < p.n_splits; ++k) p.ws_lse[k * slot_rows + rid] = -INFINITY;
                        }
                        continue;
                    }
                    const long long a = max(s0, lo_g), e = min(s0 + nb, hi_g);
                    if (a >= e) continue;  // this item does not reach into the share
                    const int n_lo = (int)(a - s0), n_end = (int)(e - s0);
                    const int slot = (int)(c - s0 / T);
                    const int fill = (e == s0 + nb) ? p.n_splits - 1 - slot : 0;  // the item's last piece
                    it.b = b;
                    it.h = h * p.pack;
                    it.split = slot;
                    it.fill = fill;
                    it.q_row0 = b * p.seqlen_q;
                    it.sq = p.seqlen_q;
                    it.k_row0 = b * p.seqlen_k;
                    it.sk = L;
                    it.bad_len = (rec >> 31) != 0u;
                    it.n_lo = n_lo;
                    set_tile_ranges<PAIR>(p, it, 0, n_end, rank);
                    return true;
                }
                return false;
            };
            int w_next = unit;
            int round_no = 0;  // static order: rounds of the snake
            Item it_next{};
            if constexpr (CACHE) {
                if (p.stream) w_next = next_piece(it_next) ? 0 : 1;  // (index 1 = p.n_items: the end)
            }
            if (!publish(w_next, it_next)) aborted = true;
            for (int w = w_next; !aborted && w < p.n_items; w = w_next) {
                // the next index is requested now and published once this item's loads have
                // been issued, so the counter's round trip overlaps them
                ++round_no;
                tr.ev(1);
                const uint32_t ticket = greedy ? atomicAdd(p.sched, 1u) : 0u;
                const Item it = it_next;
                const int bc = V::varlen(p) ? 0 : it.b;  // batch coordinate of the 4-D view
                auto load_q = [&](auto tc) -> bool {
                    constexpr int t = decltype(tc)::value;
                    if (it.n_hi_t[t] <= it.n_lo) return true;
                    if (!wait_bar(bar(C::Q_EMPTY + t), ((ph_qe >> t) & 1u) ^ 1u, wc, SITE_Q_EMPTY))
                        return false;
                    tr.ev(2 + t);
                    ph_qe ^= 1u << t;
                    if (V::inject(p) == 1u && !withheld) {  // debug: never arrive on this Q tile
                        withheld = true;
                        return true;
                    }
                    // packed mode: the map's box spans G heads x 128/G rows
                    const int qrow = (V::varlen(p) ? it.q_row0 : 0) + it.m0[t] / p.pack;
                    // a pair's Q tiles both land on the even CTA's barrier, which expects them
                    if (rank == 0u) {
                        mbar_arrive_expect_tx(bar(C::Q_FULL + t), (PAIR ? 2 : 1) * C::kTileBytes);
                        q_par ^= 1u << t;
                        q_any |= 1u << t;
                    }
#pragma unroll
                    for (int c = 0; c < C::kChunks; ++c) {
                        if constexpr (PAIR)
                            tma_load_4d_pair(s_q + t * C::kTileBytes + c * C::kChunkBytes, &tm_q,
                                             leader(bar(C::Q_FULL + t)), c * C::kChunkElems, it.h, qrow,
                                             bc, pol_q);
                        else
                            tma_load_4d(s_q + t * C::kTileBytes + c * C::kChunkBytes, &tm_q,
                                        bar(C::Q_FULL + t), c * C::kChunkElems, it.h, qrow, bc, pol_q);
                    }
                    return true;
                };
                const bool has_work = it.n_hi > it.n_lo;
                if (has_work &&
                    (!load_q(std::integral_constant<int, 0>{}) || !load_q(std::integral_constant<int, 1>{}))) {
                    aborted = true;
                    break;
                }
                const int kv_head = it.h / p.kv_group;  // grouped-query: shared K/V head
                // K/V go through the ring in the order K(n_hi-1), V(n_hi-1), K(n_hi-2), ...,
                // V(n_lo), one slot each, and are signalled in groups: {K(n_hi-1)},
                // {V(j), K(j-1)} for each later block, {V(n_lo)} -- the MMA issuer needs V(j)
                // and K(j-1) at the same point, so one wait covers both.  A group completes
                // the KV_FULL barrier of its first slot.
                auto free_slot = [&](uint32_t pos) -> bool {
                    return wait_bar(bar(C::KV_EMPTY + pos % C::kStages),
                                    ((pos / C::kStages) & 1u) ^ 1u, wc, SITE_KV_EMPTY);
                };
                auto load_kv = [&](uint32_t pos, bool is_v, int j, uint32_t full) {
                    const uint32_t dst = s_kv + (pos % C::kStages) * C::kSlotBytes;
                    const int row = (V::varlen(p) ? it.k_row0 : 0) + j * kBN;
                    if constexpr (PAIR) {
                        // this CTA's half: head-dim columns [64r, 64r+64) of V(j) (one atom
                        // column, 128 keys), or keys [64r, 64r+64) of K(j) (64-row boxes)
                        const uint32_t fl = leader(full);
                        if (is_v) {
                            tma_load_4d_pair(dst, &tm_v, fl, (int)rank * C::kChunkElems, kv_head, row, bc,
                                             pol_kv);
                        } else {
#pragma unroll
                            for (int c = 0; c < C::kChunks; ++c)
                                tma_load_4d_pair(dst + c * C::kKChunkBytes, &tm_k, fl, c * C::kChunkElems,
                                                 kv_head, row + (int)rank * (kBN / 2), bc, pol_kv);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < C::kChunks; ++c)
                            tma_load_4d(dst + c * C::kChunkBytes, is_v ? &tm_v : &tm_k, full,
                                        c * C::kChunkElems, kv_head, row, bc, pol_kv);
                    }
                };
                // bytes a group of n slots brings to its barrier (both CTAs' halves in a pair;
                // only the even CTA, which owns the barrier, announces them)
                auto expect_group = [&](uint32_t slot, uint32_t n) {
                    if (rank == 0u) {
                        mbar_arrive_expect_tx(bar(C::KV_FULL + slot), n * (PAIR ? 2u : 1u) * C::kSlotBytes);
                        kv_par ^= 1u << slot;
                        kv_any |= 1u << slot;
                    }
                };
                // Few new cache rows (decoding): the ones inside this item's key blocks go
                // into the caches now, before any of those blocks is loaded -- generic-proxy
                // writes, a proxy fence, then the TMA reads.  Every new row lies in one block,
                // and every item that reads that block writes the row itself (items of other
                // query heads of the same K/V head write the same bytes).  A sequence whose
                // filled length leaves no room gets no rows; the error word records it.
                if (CACHE && !PAIR && p.append_rows > 0 && has_work) {  // (pairs take no cache calls)
                    const int len = __ldg(p.seqused_k + it.b);
                    if (len < 0 || len > p.seqlen_k - p.append_rows) {
                        atomicOr(p.err, kErrBadLength);
                    } else {
                        constexpr int kVecs = D * C::kElem / 16;  // 16-byte vectors in one head's row
                        const int hk = p.heads / p.kv_group;
                        const int r0 = max(len, it.n_lo * kBN);
                        const int r1 = min(len + p.append_rows, it.n_hi * kBN);
                        const uint4* kn = static_cast<const uint4*>(p.k_new);
                        const uint4* vn = static_cast<const uint4*>(p.v_new);
                        uint4* kc = static_cast<uint4*>(p.k_cache);
                        uint4* vc = static_cast<uint4*>(p.v_cache);
                        for (int r = r0; r < r1; ++r) {
                            const size_t src = (((size_t)it.b * p.append_rows + (r - len)) * hk + kv_head) * kVecs;
                            const size_t dst = (((size_t)it.b * p.seqlen_k + r) * hk + kv_head) * kVecs;
                            for (int c = 0; c < kVecs; ++c) {
                                kc[dst + c] = __ldg(kn + src + c);
                                vc[dst + c] = __ldg(vn + src + c);
                            }
                        }
                        fence_proxy_async_global();
                    }
                }
                if (has_work) {
                    const int j0 = it.n_hi - 1;
                    if (!free_slot(ring)) {
                        aborted = true;
                        break;
                    }
                    uint32_t full = bar(C::KV_FULL + ring % C::kStages);
                    expect_group(ring % C::kStages, 1u);
                    load_kv(ring, false, j0, full);
                    ++ring;
                    for (int j = j0; j >= it.n_lo; --j) {
                        const bool pair = j > it.n_lo;  // V(j) with K(j-1), or V(n_lo) alone
                        if (!free_slot(ring) || (pair && !free_slot(ring + 1))) {
                            aborted = true;
                            break;
                        }
                        full = bar(C::KV_FULL + ring % C::kStages);
                        expect_group(ring % C::kStages, pair ? 2u : 1u);
                        load_kv(ring, true, j, full);
                        if (pair) load_kv(ring + 1, false, j - 1, full);
                        ring += pair ? 2u : 1u;
                        tr.ev(4);
                    }
                }
                if (aborted) break;
                if (CACHE && p.stream) {
                    if constexpr (CACHE) w_next = next_piece(it_next) ? 0 : 1;
                } else if (greedy) {
                    w_next = min((int)(gridDim.x + ticket), p.n_items);
                    if (w_next >= p.n_items) fetching_done();
                } else {
                    w_next = min(item_of_round(round_no, unit, nunits), p.n_items);
                }
                if (!publish(w_next, it_next)) {
                    aborted = true;
                    break;
                }
                tr.ev(5);
            }
            if (greedy) fetching_done();  // after an abort, or with no item beyond the first
            tr.fin();
            if (aborted) {
                // Loads already issued must land before the CTA retires (its shared memory
                // may go to the next CTA on this SM): wait, bounded and regardless of the
                // abort flag, for the last armed phase of every full barrier -- phases of one
                // barrier complete in order, so that covers every earlier load too.
#pragma unroll 1
                for (int t = 0; t < kTiles; ++t)
                    if ((q_any >> t) & 1u)
                        wait_slow(bar(C::Q_FULL + t), ((q_par >> t) & 1u) ^ 1u, wc, SITE_LOAD_DRAIN, false);
#pragma unroll 1
                for (int s = 0; s < C::kStages; ++s)
                    if ((kv_any >> s) & 1u)
                        wait_slow(bar(C::KV_FULL + s), ((kv_par >> s) & 1u) ^ 1u, wc, SITE_LOAD_DRAIN, false);
                if constexpr (PAIR) {
                    // the odd CTA's halves complete on the even CTA's barriers, which it
                    // cannot watch, and it may have run ahead of the arming: a grace period
                    const uint64_t t0 = globaltimer_ns();
                    while (globaltimer_ns() - t0 < 200000ull) {
                    }
                }
            }
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // One thread issues every MMA.  Its bookkeeping sits between MMA batches, so
        // it is kept lean: tiles are unrolled at compile time (phase bits live in
        // registers), and descriptors are built once -- per MMA only the 32-bit low
        // word (start address) advances.
        if (PAIR && rank != 0u && lane == 0) {
            // the odd CTA of a pair issues nothing; it only keeps its item ring turning
            for (;;) {
                int w;
                Item it;
                if (!read_item(w, it)) break;
                mbar_arrive(bar(C::ITEM_EMPTY + ((items_read - 1) & 1u)));
                if (w >= p.n_items) break;
            }
        } else if (lane == 0) {
            // descriptor words: high word (SBO = 1024 B, version 1, 128B swizzle) is common
            const uint32_t d_hi = (uint32_t)(sdesc_sw128(0, 16, 1024) >> 32);
            const uint32_t q_lo = (uint32_t)sdesc_sw128(s_q, 16, 1024);          // + t*tile
            const uint32_t k_lo = (uint32_t)sdesc_sw128(s_kv, 16, 1024);         // + slot*slot bytes
            const uint32_t v_lo = (uint32_t)sdesc_sw128(s_kv, C::kChunkBytes, 1024);
            constexpr uint32_t kTile16 = C::kTileBytes >> 4;
            constexpr uint32_t kSlot16 = C::kSlotBytes >> 4;
            // MMA completions reach both CTAs of a pair
            auto commit = [&](uint32_t b) {
                if constexpr (PAIR)
                    umma_commit_pair_mc(b, (uint16_t)0x3);
                else
                    umma_commit(b);
            };
            // a K/V slot that a tile does not read is released for it (in both CTAs of a pair)
            const uint32_t kv_empty_peer = PAIR ? mapa_shared(bar(C::KV_EMPTY), 1u) : 0u;
            auto release_slot = [&](uint32_t slot) {
                mbar_arrive(bar(C::KV_EMPTY + slot));
                if constexpr (PAIR) mbar_arrive_cluster(kv_empty_peer + 8u * slot);
            };
            // P and O hand-offs: a pair's odd CTA arrives from the other SM
            auto wait_handoff = [&](uint32_t b, uint32_t parity, uint32_t site) -> bool {
                return PAIR ? wait_bar_cluster(b, parity, wc, site) : wait_bar(b, parity, wc, site);
            };
            auto desc = [&](uint32_t lo) -> uint64_t { return ((uint64_t)d_hi << 32) | lo; };
            uint32_t ring = 0;
            uint32_t ph_q = 0, ph_p = 0, ph_o = 0;  // bit t: parity of the next wait on tile t
            Tracer tr;
            tr.init(p.trace, 1);
            uint32_t ph_kv = 0;  // bit s: parity of the next wait on KV_FULL[s] (armed per group)
            auto wait_kv = [&](uint32_t slot) -> bool {
                if (!wait_bar(bar(C::KV_FULL + slot), (ph_kv >> slot) & 1u, wc, SITE_KV_FULL)) return false;
                ph_kv ^= 1u << slot;
                return true;
            };
            bool aborted = false;
            // S_t = Q_t K^T : A = Q (K-major), B = K (K-major), both 128B-swizzled.
            auto issue_qk = [&](auto tc, uint32_t kslot) {
                constexpr int t = decltype(tc)::value;
                uint32_t a0 = q_lo + t * kTile16, b0 = k_lo + kslot * kSlot16;
                // STEADY: bases taken per call, so the compiler keeps no per-item set of 64-bit
                // descriptors live across blocks (it spilled them: 60 bytes; without, -1.4 %)
                if constexpr (STEADY) asm volatile("" : "+r"(a0), "+r"(b0));
#pragma unroll
                for (int kk = 0; kk < D / C::kUmmaK; ++kk) {
                    // k step kk: 32 bytes further along the row, next 128-byte atom column
                    // (a K slot's atom columns are 64 rows deep in a pair)
                    constexpr uint32_t kAtomA = C::kChunkBytes >> 4, kAtomB = C::kKChunkBytes >> 4;
                    const uint32_t col = (uint32_t)((kk * C::kUmmaK) / C::kChunkElems);
                    const uint32_t in_row = (uint32_t)((kk * 32) % 128 >> 4);
                    const uint32_t a_off = col * kAtomA + in_row, b_off = col * kAtomB + in_row;
                    if constexpr (PAIR)
                        umma_f16_ss_pair(tmem_base + 128u * t, desc(a0 + a_off), desc(b0 + b_off), C::kIdescQK,
                                         kk > 0);
                    else if constexpr (FP8)
                        umma_f8_ss(tmem_base + 128u * t, desc(a0 + a_off), desc(b0 + b_off), C::kIdescQK, kk > 0);
                    else
                        umma_f16_ss(tmem_base + 128u * t, desc(a0 + a_off), desc(b0 + b_off), C::kIdescQK, kk > 0);
                }
            };
            // O_t += P_t V : A = P_t from TMEM, B = V (MN-major, 128B-swizzled):
            // leading offset = next 128-byte column atom, stride offset = next 8 keys.
            const uint32_t idesc_pv = (FP8 && p.v_e5m2) ? C::kIdescPV5 : C::kIdescPV;
            auto issue_pv = [&](auto tc, uint32_t vslot, uint32_t acc) {
                constexpr int t = decltype(tc)::value;
                uint32_t b0 = v_lo + vslot * kSlot16;
                if constexpr (STEADY) asm volatile("" : "+r"(b0));
#pragma unroll
                for (int kk = 0; kk < kBN / C::kUmmaK; ++kk) {
                    const uint32_t off = (uint32_t)(kk * C::kUmmaK * 128) >> 4;
                    const uint32_t a_tmem = tmem_base + 128u * t + 8u * kk;
                    if constexpr (PAIR)
                        umma_f16_ts_pair(tmem_base + C::kColO + 128u * t, a_tmem, desc(b0 + off), C::kIdescPV,
                                         kk > 0 ? 1u : acc);
                    else if constexpr (FP8)
                        umma_f8_ts(tmem_base + C::kColO + 128u * t, a_tmem, desc(b0 + off), idesc_pv,
                                   kk > 0 ? 1u : acc);
                    else
                        umma_f16_ts(tmem_base + C::kColO + 128u * t, a_tmem, desc(b0 + off), C::kIdescPV,
                                    kk > 0 ? 1u : acc);
                }
            };
            for (;;) {
                int w;
                Item it;
                if (!read_item(w, it)) {
                    aborted = true;
                    break;
                }
                mbar_arrive(bar(C::ITEM_EMPTY + ((items_read - 1) & 1u)));
                if (w >= p.n_items) break;
                if (it.n_hi <= it.n_lo) continue;
                tr.ev(1);
                const int hi0 = it.n_hi_t[0], hi1 = it.n_hi_t[1], lo = it.n_lo;
                const bool has0 = hi0 > lo, has1 = hi1 > lo;
                if (has0 && !wait_bar(bar(C::Q_FULL + 0), ph_q & 1u, wc, SITE_Q_FULL)) break;
                if (has1 && !wait_bar(bar(C::Q_FULL + 1), (ph_q >> 1) & 1u, wc, SITE_Q_FULL)) break;
                tc_fence_after();
                tr.ev(2);
                uint32_t acc0 = 0u, acc1 = 0u;  // becomes 1 after the tile's first PV
                const int j0 = it.n_hi - 1;
                const uint32_t kslot0 = ring % C::kStages;
                if (!wait_kv(kslot0)) break;  // group {K(j0)}
                ++ring;
                // FP8: a tile's last QK^T is the one for block lo; once it completes, the
                // producer may load the next item's Q over this one while the last PVs run
                // (measured: +5 % on FP8, -2 to -4 % on bf16, which releases Q at the item end)
                if (j0 < hi0) {
                    issue_qk(std::integral_constant<int, 0>{}, kslot0);
                    commit(bar(C::S_FULL + 0));
                    if (FP8 && j0 == lo) commit(bar(C::Q_EMPTY + 0));
                } else {
                    release_slot(kslot0);  // tile 0 never reads K(j0)
                }
                if (j0 < hi1) {
                    issue_qk(std::integral_constant<int, 1>{}, kslot0);
                    commit(bar(C::S_FULL + 1));
                    if (FP8 && j0 == lo) commit(bar(C::Q_EMPTY + 1));
                } else {
                    release_slot(kslot0);
                }
                if constexpr (STEADY) {
                    // STEADY instance: the body of one key block as a template on kSteady -- both
                    // tiles visit blocks j and j - 1 and are past their first PV, and no slot is
                    // released for a skipping tile.  The issuer's instruction stream paces the
                    // tensor pipe, and in steady blocks it then carries no per-block tests.
                    auto run_block = [&](const int j, auto steady_c) -> bool {
                        constexpr bool kSteady = decltype(steady_c)::value;
                        const uint32_t vslot = ring % C::kStages;
    #ifdef FA_TRACE  // had the group landed when the issuer got here?
                        tr.ev(mbar_test_wait(bar(C::KV_FULL + vslot), (ph_kv >> vslot) & 1u) ? 11 : 12);
    #endif
                        if (!wait_kv(vslot)) return false;  // group {V(j), K(j-1)} (or {V(lo)})
                        tr.ev(3);
                        ++ring;
                        // a tile that does not visit block j releases V(j) at once (its load has
                        // landed, so the arrival belongs to this phase of the slot)
                        if (!kSteady) {
                            if (j >= hi0) release_slot(vslot);
                            if (j >= hi1) release_slot(vslot);
                        }
                        const bool has_next = kSteady || j - 1 >= lo;
                        const uint32_t nslot = ring % C::kStages;  // K(j-1), landed with V(j)
                        if (has_next) ++ring;
                        // one tile: PV_t(j) if it visits block j, then S_t(j-1) if it visits j-1
                        auto tile_step = [&](auto tc, int hi, uint32_t& acc) -> bool {
                            constexpr int t = decltype(tc)::value;
                            const bool cur = kSteady || j < hi;
                            const bool nxt = kSteady || (has_next && (j - 1) < hi);
                            if (cur) {
    #ifdef FA_TRACE  // was P ready when the issuer got here?
                                tr.ev(mbar_test_wait(bar(C::P_FULL + t), (ph_p >> t) & 1u) ? 13 : 14);
    #endif
                                if (!wait_handoff(bar(C::P_FULL + t), (ph_p >> t) & 1u, SITE_P_FULL)) return false;
                                tr.ev(4 + t);
                                ph_p ^= 1u << t;
                                if (!kSteady && acc == 0u &&
                                    !wait_handoff(bar(C::O_EMPTY + t), ((ph_o >> t) & 1u) ^ 1u, SITE_O_EMPTY))
                                    return false;
                                tc_fence_after();
                                issue_pv(tc, vslot, kSteady ? 1u : acc);
                                acc = 1u;
                            }
                            if (nxt) {
                                issue_qk(tc, nslot);
                                commit(bar(C::S_FULL + t));
                                if (FP8 && j - 1 == lo) commit(bar(C::Q_EMPTY + t));
                            } else if (cur) {
                                commit(bar(C::O_FULL + t));  // last block of tile t
                            }
                            tr.ev(6 + t);
                            return true;
                        };
                        if (!tile_step(std::integral_constant<int, 0>{}, hi0, acc0) ||
                            !tile_step(std::integral_constant<int, 1>{}, hi1, acc1))
                            return false;
                        if (!kSteady && has_next) {  // K(j-1) has landed (some tile read it); skipping tiles release it
                            if (j - 1 >= hi0) release_slot(nslot);
                            if (j - 1 >= hi1) release_slot(nslot);
                        }
                        return true;
                    };
                    // steady blocks: lo < j <= min(hi0, hi1) - 2 (both tiles had their first PV at
                    // block hi_t - 1 > j)
                    const int j_steady = min(hi0, hi1) - 2;
                    for (int j = j0; j >= lo; --j) {
                        const bool ok = (j <= j_steady && j > lo) ? run_block(j, std::true_type{})
                                                                  : run_block(j, std::false_type{});
                        if (!ok) {
                            aborted = true;
                            break;
                        }
                    }
                } else {
                    // the other instances keep the block loop as it stood before the steady
                    // instance: routing them through run_block changes their code, and every
                    // change to the issuer's code moved their launches by 1-3 %
                    for (int j = j0; j >= lo; --j) {
                        const uint32_t vslot = ring % C::kStages;
    #ifdef FA_TRACE  // had the group landed when the issuer got here?
                        tr.ev(mbar_test_wait(bar(C::KV_FULL + vslot), (ph_kv >> vslot) & 1u) ? 11 : 12);
    #endif
                        if (!wait_kv(vslot)) {  // group {V(j), K(j-1)} (or {V(lo)})
                            aborted = true;
                            break;
                        }
                        tr.ev(3);
                        ++ring;
                        // a tile that does not visit block j releases V(j) at once (its load has
                        // landed, so the arrival belongs to this phase of the slot)
                        if (j >= hi0) release_slot(vslot);
                        if (j >= hi1) release_slot(vslot);
                        const bool has_next = j - 1 >= lo;
                        const uint32_t nslot = ring % C::kStages;  // K(j-1), landed with V(j)
                        if (has_next) ++ring;
                        // one tile: PV_t(j) if it visits block j, then S_t(j-1) if it visits j-1
                        auto tile_step = [&](auto tc, int hi, uint32_t& acc) -> bool {
                            constexpr int t = decltype(tc)::value;
                            const bool cur = j < hi;
                            const bool nxt = has_next && (j - 1) < hi;
                            if (cur) {
    #ifdef FA_TRACE  // was P ready when the issuer got here?
                                tr.ev(mbar_test_wait(bar(C::P_FULL + t), (ph_p >> t) & 1u) ? 13 : 14);
    #endif
                                if (!wait_handoff(bar(C::P_FULL + t), (ph_p >> t) & 1u, SITE_P_FULL)) return false;
                                tr.ev(4 + t);
                                ph_p ^= 1u << t;
                                if (acc == 0u &&
                                    !wait_handoff(bar(C::O_EMPTY + t), ((ph_o >> t) & 1u) ^ 1u, SITE_O_EMPTY))
                                    return false;
                                tc_fence_after();
                                issue_pv(tc, vslot, acc);
                                acc = 1u;
                            }
                            if (nxt) {
                                issue_qk(tc, nslot);
                                commit(bar(C::S_FULL + t));
                                if (FP8 && j - 1 == lo) commit(bar(C::Q_EMPTY + t));
                            } else if (cur) {
                                commit(bar(C::O_FULL + t));  // last block of tile t
                            }
                            tr.ev(6 + t);
                            return true;
                        };
                        if (!tile_step(std::integral_constant<int, 0>{}, hi0, acc0) ||
                            !tile_step(std::integral_constant<int, 1>{}, hi1, acc1)) {
                            aborted = true;
                            break;
                        }
                        if (has_next) {  // K(j-1) has landed (some tile read it); skipping tiles release it
                            if (j - 1 >= hi0) release_slot(nslot);
                            if (j - 1 >= hi1) release_slot(nslot);
                        }
                    }
                }
                if (aborted) break;
                tr.ev(8);
                if (!FP8 && has0) commit(bar(C::Q_EMPTY + 0));
                if (!FP8 && has1) commit(bar(C::Q_EMPTY + 1));
                ph_q ^= (has0 ? 1u : 0u) | (has1 ? 2u : 0u);
                ph_o ^= (has0 ? 1u : 0u) | (has1 ? 2u : 0u);
            }
            // Drain: every MMA issued by this thread has completed before TMEM is
            // released, also after an abort (bounded by the wait limit only).
            if constexpr (PAIR)
                umma_commit_pair(bar(C::DRAIN));
            else
                umma_commit(bar(C::DRAIN));
            if (!mbar_try_wait(bar(C::DRAIN), 0u)) wait_slow(bar(C::DRAIN), 0u, wc, SITE_DRAIN, false);
            tr.fin();
        }
        __syncwarp();
    }
    } else {
        setmaxnreg_inc<kRegsSoftmax>();
        // ------------------------------------------------------------ softmax / epilogue
        const int t = (warp - 4) >> 2;              // query tile of this warpgroup
        const int wq = warp & 3;                    // TMEM lane quarter of this warp
        const int r_in_tile = wq * 32 + lane;       // this thread's row within the tile
        const uint32_t t_lane = tmem_base + ((uint32_t)(wq * 32) << 16);
        const uint32_t t_s = t_lane + 128u * t;     // S_t (fp32) and, over it, P_t
        const uint32_t t_o = t_lane + C::kColO + 128u * t;
        uint32_t s_cnt = 0, o_cnt = 0;
        uint32_t stg_cnt = 0;  // staging-buffer passes of this tile so far (both barriers' phase)
        uint32_t kv_base = 0;  // ring position of the current item's first K/V load
        const bool releaser = wq == 0 && lane == 0;  // this warpgroup's slot-release thread
        bool aborted = false;
        uint32_t held = 0;  // 1 + the item-ring slot whose record this warp still reads (0: none)
        bool stg_owed = false;  // (thread 0 of the tile) its last O store's read is unconfirmed
        Tracer tr;
        tr.init(r_in_tile == 0 ? p.trace : nullptr, 2 + t);
        // output addresses of this thread's row of a tile starting at (packed) row m0 of the
        // item (b, h, split, first packed row q_row0); false past the sequence end
        auto out_addr = [&](int b, int h, int split, int q_row0, int sq, int m0, float*& lse_ptr,
                            float*& wso_ptr, __nv_bfloat16*& o_ptr) -> bool {
            const int prow = m0 + r_in_tile;               // (packed) tile row
            const int row = prow >> p.pack_shift;           // query row within the sequence
            const int hrow = h + (prow & (p.pack - 1));     // query head of this row
            wso_ptr = nullptr;
            o_ptr = nullptr;
            if (p.split) {
                const size_t rid = (((size_t)split * p.batch + b) * p.heads + hrow) * (size_t)p.seqlen_q + row;
                lse_ptr = p.ws_lse + rid;
                wso_ptr = p.ws_o + rid * D;
            } else if (V::varlen(p)) {
                lse_ptr = p.lse + (size_t)hrow * p.total_q + q_row0 + row;
                o_ptr = reinterpret_cast<__nv_bfloat16*>(p.o) + (((size_t)q_row0 + row) * p.heads + hrow) * D;
            } else {
                lse_ptr = p.lse + ((size_t)b * p.heads + hrow) * p.seqlen_q + row;
                o_ptr = reinterpret_cast<__nv_bfloat16*>(p.o) + (((size_t)b * p.seqlen_q + row) * p.heads + hrow) * D;
            }
            return prow < (sq << p.pack_shift);
        };
        // balanced cache plan: an item's last piece marks the item's later partial slots of
        // this row empty (LSE = -inf; the merge gives such slots weight 0 and never reads
        // their O), so the merge sees exactly the item's pieces (at most 3 later slots)
        auto mark_empty_slots = [&](float* lse_ptr, int fill) {
            const size_t slot_rows = (size_t)p.batch * p.heads * p.seqlen_q;
#pragma unroll
            for (int k2 = 1; k2 <= 3; ++k2)
                if (k2 <= fill) lse_ptr[k2 * slot_rows] = -INFINITY;
        };
        for (;;) {
            int w = 0;
            Item it;
            bool got = read_item(w, it);
            got = __all_sync(0xffffffffu, got);
            if (!got) {
                aborted = true;
                break;
            }
            // The previous item is finished: release its record.  This item's record is held
            // until then -- its epilogue reads its output coordinates back from it rather than
            // keeping them in registers through the key loop.  (The producer reuses a slot
            // only after issuing every load of the item in between.)
            __syncwarp();
            if (lane == 0 && held) mbar_arrive(bar(C::ITEM_EMPTY + (held - 1u)));
            held = 1u + ((items_read - 1) & 1u);
            if (w >= p.n_items) break;
            tr.ev(1);
            if (it.bad_len && r_in_tile == 0 && t == 0) atomicOr(p.err, kErrBadLength);
            const uint32_t item_base = kv_base;
            if (it.n_hi > it.n_lo) kv_base += 2u * (uint32_t)(it.n_hi - it.n_lo);
            // ring slots of this item's K(j) and V(j)
            auto k_slot = [&](int j) { return (item_base + 2u * (uint32_t)(it.n_hi - 1 - j)) % C::kStages; };
            auto v_slot = [&](int j) { return (item_base + 2u * (uint32_t)(it.n_hi - 1 - j) + 1u) % C::kStages; };
            // this warpgroup's tile, selected without indexing (keeps Item in registers)
            const bool t_active = t ? it.active[1] : it.active[0];
            const int t_m0 = t ? it.m0[1] : it.m0[0];
            const int t_hi = t ? it.n_hi_t[1] : it.n_hi_t[0];
            if (!t_active) continue;
            // FP8: q_descale * k_descale folded into the scale of this work tile, which
            // belongs to one (batch, head); v_descale scales its output
            float scale_log2 = p.scale_log2;
            float o_scale = 1.0f;
            if constexpr (FP8) {
                const long long ds = it.b * p.descale_sb + (long long)(it.h / p.kv_group) * p.descale_sh;
                const float qd = p.q_descale ? __ldg(p.q_descale + ds) : 1.0f;
                const float kd = p.k_descale ? __ldg(p.k_descale + ds) : 1.0f;
                scale_log2 *= qd * kd;
                o_scale = p.v_descale ? __ldg(p.v_descale + ds) : 1.0f;
            }
            const int row = (t_m0 + r_in_tile) >> p.pack_shift;  // query row within the sequence
            if (t_hi <= it.n_lo) {
                float* lse_ptr;
                float* wso_ptr;
                __nv_bfloat16* o_ptr;
                const bool row_ok =
                    out_addr(it.b, it.h, it.split, it.q_row0, it.sq, t_m0, lse_ptr, wso_ptr, o_ptr);
                // no visible key for any row of this tile: O = 0, LSE = -inf
                if (row_ok) {
                    if (p.split) {
                        for (int c = 0; c < D; c += 4)
                            *reinterpret_cast<float4*>(wso_ptr + c) = make_float4(0.f, 0.f, 0.f, 0.f);
                    } else {
                        for (int c = 0; c < D; c += 8)
                            *reinterpret_cast<uint4*>(o_ptr + c) = make_uint4(0u, 0u, 0u, 0u);
                    }
                    *lse_ptr = -INFINITY;
                }
                continue;
            }
            // visible keys of this row: [0, vis_end) with vis_end = min(sk, row + sk - sq + 1)
            const int vis_end = p.causal ? min(it.sk, row + it.sk - it.sq + 1) : it.sk;
            // a block needs masking iff some column of it is invisible to some row of the tile
            const int tile_rmin = t_m0 >> p.pack_shift;  // the tile's first query row
            const int tile_vis_min = p.causal ? min(it.sk, tile_rmin + it.sk - it.sq + 1) : it.sk;
            float m_run = -INFINITY;  // running max of scale_log2 * s (lazy reference)
            float l_run = 0.0f;       // running sum of exp2(scale_log2 * s - m_run)
            const int j_first = t_hi - 1;
            for (int j = j_first; j >= it.n_lo; --j) {
                bool ok = wait_bar(bar(C::S_FULL + t), s_cnt & 1u, wc, SITE_S_FULL);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    aborted = true;
                    break;
                }
                ++s_cnt;
                tc_fence_after();
                tr.ev(2);
                // S_t(j) is complete: K(j) is consumed, and so is V(j+1) (PV_t(j+1) was issued
                // before S_t(j) by the same thread, and MMAs complete in issue order)
                if (releaser) {
                    mbar_arrive(bar(C::KV_EMPTY + k_slot(j)));
                    if (j + 1 < t_hi) mbar_arrive(bar(C::KV_EMPTY + v_slot(j + 1)));
                }
                uint32_t sr[128];
                tmem_ld128(t_s, sr);
                tmem_wait_ld();
                tr.ev(7);
                float s[128];
#pragma unroll
                for (int q = 0; q < 4; ++q)
#pragma unroll
                    for (int i = 0; i < 32; ++i) s[q * 32 + i] = __uint_as_float(sr[q * 32 + i]);
                const int col0 = j * kBN;
                const bool masked = col0 + kBN > tile_vis_min;  // diagonal or key-tail block
                if (masked) {
                    const int lim = vis_end - col0;
#pragma unroll
                    for (int c = 0; c < 128; ++c)
                        if (c >= lim) s[c] = -INFINITY;
                }
                float mx0 = s[0], mx1 = s[1], mx2 = s[2], mx3 = s[3];
#pragma unroll
                for (int c = 4; c < 124; c += 8) {
                    mx0 = max3f(mx0, s[c], s[c + 1]);
                    mx1 = max3f(mx1, s[c + 2], s[c + 3]);
                    mx2 = max3f(mx2, s[c + 4], s[c + 5]);
                    mx3 = max3f(mx3, s[c + 6], s[c + 7]);
                }
                mx0 = max3f(mx0, s[124], s[125]);
                mx1 = max3f(mx1, s[126], s[127]);
                const float m_cand = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3)) * scale_log2;
                // Lazy rescale: the reference max moves only when it grows by more than
                // 2^tau.  tcgen05.ld/st are warp-collective (.sync.aligned), so the O
                // round trip is taken by the whole warp whenever any of its rows needs it;
                // rows that keep their reference scale by 1.
                const bool grow = m_cand > m_run + lazy_tau<FP8>();
                if (__any_sync(0xffffffffu, grow)) {
                    const float f = grow ? ex2_approx(m_run - m_cand) : 1.0f;  // 0 if m_run = -inf
                    if (j != j_first) {  // the first block's PV overwrites O (uniform per warp)
                        const uint64_t f2 = f32x2(f, f);
#pragma unroll 1
                        for (int c = 0; c < D; c += 32) {
                            uint32_t orr[32];
                            tmem_ld32(t_o + c, orr);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; i += 2) {
                                float a, b;
                                unpack_f32x2(mul_f32x2(f32x2(__uint_as_float(orr[i]),
                                                             __uint_as_float(orr[i + 1])), f2), a, b);
                                orr[i] = __float_as_uint(a);
                                orr[i + 1] = __float_as_uint(b);
                            }
                            tmem_st32(t_o + c, orr);
                        }
                    }
                    if (grow) {
                        l_run *= f;
                        m_run = m_cand;
                    }
                }
                const float mu = (m_run == -INFINITY) ? 0.0f : m_run;
                tr.ev(8);
                // exp2(s * scale_log2 - mu) on packed fp32 pairs (f32x2 FMA/add halve the
                // issue slots); P is converted to bf16x2 / e4m3x4 and stored to TMEM in one go.
                const uint64_t sc2 = f32x2(scale_log2, scale_log2);
                const uint64_t nm2 = f32x2(-mu, -mu);
                const uint64_t mg2 = f32x2(kRoundMagic, kRoundMagic);
                const uint64_t c0 = f32x2(kExp2C0, kExp2C0), c1 = f32x2(kExp2C1, kExp2C1);
                const uint64_t c2 = f32x2(kExp2C2, kExp2C2), c3 = f32x2(kExp2C3, kExp2C3);
                uint64_t acc0 = f32x2(0.f, 0.f), acc1 = acc0;
                constexpr int kPkPerChunk = FP8 ? 8 : 16;
                uint32_t pk_all[4 * kPkPerChunk];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float e[32];
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        const int c = 32 * q + 2 * i;
                        float a, b;
                        const uint64_t x2 = fma_f32x2(f32x2(s[c], s[c + 1]), sc2, nm2);
                        if (FA_EXP2_EMU_PAIRS > 0 && !masked && (i % 16) < FA_EXP2_EMU_PAIRS) {
                            unpack_f32x2(x2, a, b);
                            const uint64_t xc = f32x2(fmaxf(a, -125.0f), fmaxf(b, -125.0f));
                            const uint64_t r = add_f32x2(xc, mg2);          // magic + round(x)
                            const uint64_t fr = sub_f32x2(xc, sub_f32x2(r, mg2));
                            uint64_t pp = fma_f32x2(c3, fr, c2);
                            pp = fma_f32x2(pp, fr, c1);
                            pp = fma_f32x2(pp, fr, c0);
                            float p0, p1, r0, r1;
                            unpack_f32x2(pp, p0, p1);
                            unpack_f32x2(r, r0, r1);
                            e[2 * i] = __uint_as_float(__float_as_uint(p0) + (__float_as_uint(r0) << 23));
                            e[2 * i + 1] = __uint_as_float(__float_as_uint(p1) + (__float_as_uint(r1) << 23));
                        } else {
                            unpack_f32x2(x2, a, b);
                            e[2 * i] = ex2_approx(a);
                            e[2 * i + 1] = ex2_approx(b);
                        }
                        if (i & 1)
                            acc1 = add_f32x2(acc1, f32x2(e[2 * i], e[2 * i + 1]));
                        else
                            acc0 = add_f32x2(acc0, f32x2(e[2 * i], e[2 * i + 1]));
                    }
                    uint32_t pk[kPkPerChunk];
#pragma unroll
                    for (int i = 0; i < kPkPerChunk; ++i) {
                        if constexpr (FP8)
                            pk[i] = pack_e4m3x4(e[4 * i], e[4 * i + 1], e[4 * i + 2], e[4 * i + 3]);
                        else
                            pk[i] = pack_bf16x2(e[2 * i], e[2 * i + 1]);
                    }
#pragma unroll
                    for (int i = 0; i < kPkPerChunk; ++i) pk_all[q * kPkPerChunk + i] = pk[i];
                }
                tr.ev(9);
                if constexpr (FP8)
                    tmem_st32(t_s, *reinterpret_cast<const uint32_t(*)[32]>(pk_all));
                else
                    tmem_st64(t_s, pk_all);
                float l0, l1, l2, l3;
                unpack_f32x2(acc0, l0, l1);
                unpack_f32x2(acc1, l2, l3);
                l_run += (l0 + l1) + (l2 + l3);
                tmem_wait_st();
                tr.ev(10);
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        mbar_arrive_cluster(leader(bar(C::P_FULL + t)));
                    else
                        mbar_arrive(bar(C::P_FULL + t));
                }
                tr.ev(3);
            }
            if (aborted) break;
            // ---------------- epilogue: O = O_acc / l, LSE = ln2 * (m + log2 l)
            {
                bool ok = wait_bar(bar(C::O_FULL + t), o_cnt & 1u, wc, SITE_O_FULL);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) {
                    aborted = true;
                    break;
                }
                ++o_cnt;
            }
            tc_fence_after();
            tr.ev(4);
            if (releaser) mbar_arrive(bar(C::KV_EMPTY + v_slot(it.n_lo)));  // PV_t(n_lo) is complete
            const bool has_mass = l_run > 0.0f;
            const float inv_l = has_mass ? o_scale / l_run : 0.0f;
            // output coordinates, read back from this item's record
            Item io;
            load_item(smem + C::kItemRecOff + 64 * (held - 1u), io);
            const int o_m0 = t ? io.m0[1] : io.m0[0];
            float* lse_ptr;
            float* wso_ptr;
            __nv_bfloat16* o_ptr;
            const bool row_ok =
                out_addr(io.b, io.h, io.split, io.q_row0, io.sq, o_m0, lse_ptr, wso_ptr, o_ptr);
            // The O tile goes out by TMA store from a per-tile staging buffer (128 rows x 64
            // columns, 128-byte swizzled like the tensor map), in D / 64 passes.  Rows past a
            // fixed-length sequence's end fall outside the map and are clipped; a varlen tile
            // that crosses its sequence's end (the next rows belong to another sequence) and
            // the fp32 split partials use plain stores instead.
            // (in a pair, the odd CTA's tile of the last slot may lie wholly past the end)
            const int sq_rows = io.sq << p.pack_shift;
            const bool use_tma = !p.split && o_m0 < sq_rows && (!V::varlen(p) || o_m0 + kBM <= sq_rows);
            if (use_tma) {
                // O leaves TMEM first (normalised and packed to bf16 on the way), so the MMA
                // issuer gets it back (O_EMPTY) before any staging
                uint32_t pk[D / 2];
#pragma unroll
                for (int hh = 0; hh < D / 64; ++hh) {
                    uint32_t o0[32], o1[32];
                    tmem_ld32(t_o + hh * 64, o0);
                    tmem_ld32(t_o + hh * 64 + 32, o1);
                    tmem_wait_ld();
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        pk[hh * 32 + i] = pack_bf16x2(__uint_as_float(o0[2 * i]) * inv_l,
                                                      __uint_as_float(o0[2 * i + 1]) * inv_l);
                        pk[hh * 32 + 16 + i] = pack_bf16x2(__uint_as_float(o1[2 * i]) * inv_l,
                                                           __uint_as_float(o1[2 * i + 1]) * inv_l);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        mbar_arrive_cluster(leader(bar(C::O_EMPTY + t)));
                    else
                        mbar_arrive(bar(C::O_EMPTY + t));
                }
                tr.ev(5);
                // the last store of the previous epilogue out of this buffer: its issuing
                // thread confirms that the TMA engine has read it only now, when the buffer is
                // needed again, instead of waiting for it at the end of that epilogue
                if (r_in_tile == 0 && stg_owed) {
                    bulk_wait_group_read0();
                    mbar_arrive(bar(C::STG_EMPTY + t));
                    stg_owed = false;
                }
                const uint32_t stile = s_base + C::kStageOff + (uint32_t)t * C::kStageBytes;
                const uint32_t srow = stile + (uint32_t)r_in_tile * 128u;
                const uint32_t sw = (uint32_t)(r_in_tile & 7);
                bool bad = false;
#pragma unroll
                for (int hh = 0; hh < D / 64; ++hh) {
                    // the previous store out of this buffer has read it
                    if (stg_cnt > 0 &&
                        !wait_bar(bar(C::STG_EMPTY + t), (stg_cnt - 1) & 1u, wc, SITE_STG_EMPTY))
                        bad = true;
                    if (__any_sync(0xffffffffu, bad)) break;
                    // 16-byte chunk c of the row lands at chunk c ^ (row mod 8)
#pragma unroll
                    for (int k4 = 0; k4 < 8; ++k4)
                        st_shared_v4(srow + ((((uint32_t)k4) ^ sw) << 4), pk[hh * 32 + 4 * k4],
                                     pk[hh * 32 + 4 * k4 + 1], pk[hh * 32 + 4 * k4 + 2],
                                     pk[hh * 32 + 4 * k4 + 3]);
                    fence_proxy_async_smem();  // generic-proxy writes -> visible to the TMA engine
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(C::STG_FULL + t));
                    if (r_in_tile == 0) {
                        if (wait_bar(bar(C::STG_FULL + t), stg_cnt & 1u, wc, SITE_STG_FULL)) {
                            tma_store_4d(&tm_o, stile, hh * 64, io.h, (V::varlen(p) ? io.q_row0 : 0) +
                                         (o_m0 >> p.pack_shift), V::varlen(p) ? 0 : io.b);
                            bulk_commit_group();
                            if (hh + 1 < D / 64) {
                                bulk_wait_group_read0();
                                mbar_arrive(bar(C::STG_EMPTY + t));
                            } else {
                                stg_owed = true;
                            }
                        } else {
                            bad = true;
                        }
                    }
                    ++stg_cnt;
                }
                if (__any_sync(0xffffffffu, bad)) {
                    aborted = true;
                    break;
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < D; c += 32) {
                    uint32_t orr[32];
                    tmem_ld32(t_o + c, orr);
                    tmem_wait_ld();
                    if (row_ok) {
                        if (p.split) {
#pragma unroll
                            for (int i = 0; i < 32; i += 4)
                                *reinterpret_cast<float4*>(wso_ptr + c + i) = make_float4(
                                    __uint_as_float(orr[i]) * inv_l, __uint_as_float(orr[i + 1]) * inv_l,
                                    __uint_as_float(orr[i + 2]) * inv_l, __uint_as_float(orr[i + 3]) * inv_l);
                        } else {
                            uint32_t pk[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i)
                                pk[i] = pack_bf16x2(__uint_as_float(orr[2 * i]) * inv_l,
                                                    __uint_as_float(orr[2 * i + 1]) * inv_l);
#pragma unroll
                            for (int i = 0; i < 4; ++i)
                                *reinterpret_cast<uint4*>(o_ptr + c + 8 * i) =
                                    make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    if constexpr (PAIR)
                        mbar_arrive_cluster(leader(bar(C::O_EMPTY + t)));
                    else
                        mbar_arrive(bar(C::O_EMPTY + t));
                }
            }
            if (row_ok) {
                // (l_run >= 1 for a row with mass: the reference max never exceeds the row max)
                *lse_ptr = has_mass ? (m_run + lg2_approx(l_run)) * 0.69314718055994531f : -INFINITY;
                if (CACHE && p.split) mark_empty_slots(lse_ptr, io.fill);
            }
            tr.ev(6);
        }
#ifdef FA_TRACE
        if (r_in_tile == 0) bulk_wait_group0();  // (the trace's end: the tile's stores done)
#endif
        tr.fin();
    }

    // the TMA stores of O have completed before this CTA retires (their issuing threads wait)
    if (warp >= 4 && (threadIdx.x & (kBM - 1)) == 0) bulk_wait_group0();
    // a pair retires together: the even CTA's MMAs (drained above) no longer read the odd
    // CTA's shared memory or write its TMEM, and no load or arrival of one CTA is still
    // heading for the other's barriers
    if constexpr (PAIR) {
        __syncwarp();
        cluster_sync();
    } else {
        __syncthreads();
    }
    // lets a programmatically dependent grid (the split merge) be scheduled; it still
    // waits for this grid's completion before reading anything
    if (threadIdx.x == 0) asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    if (warp == 1) {
        __syncwarp();
        tc_fence_after();
        if constexpr (PAIR)
            tmem_dealloc_pair(tmem_base, kTmemCols);
        else
            tmem_dealloc(tmem_base, kTmemCols);
    }
}

template <int D, bool FP8, bool PAIR = false, bool CACHE = false, bool VAR = true, bool STEADY = false>
cudaError_t launch_fwd(const CUtensorMap& q, const CUtensorMap& k, const CUtensorMap& v,
                       const CUtensorMap& o, const FwdParams& p, int grid, cudaStream_t stream,
                       bool after_append) {
    using C = Cfg<D, FP8, PAIR>;
    // The shared-memory attribute is set once per device and context (devices 0-63; others
    // every launch): the context id it was set in is kept per device, so a new context
    // (after cudaDeviceReset) sets it again; concurrent host threads at worst set it twice.
    static std::atomic<unsigned long long> attr_ctx[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const unsigned long long ctx = current_context_id();
    if (dev < 0 || dev >= 64 || ctx == 0 || attr_ctx[dev].load(std::memory_order_acquire) != ctx) {
        e = cudaFuncSetAttribute(fa_fwd_kernel<D, FP8, PAIR, CACHE, VAR, STEADY>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 C::kSmemBytes);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_ctx[dev].store(ctx, std::memory_order_release);
    }
    if (!after_append && !PAIR) {
        fa_fwd_kernel<D, FP8, PAIR, CACHE, VAR, STEADY><<<grid, kThreads, C::kSmemBytes, stream>>>(q, k, v, o, p);
        return cudaGetLastError();
    }
    // after the cache append: programmatic dependent launch, so this grid's set-up
    // (barriers, TMEM, descriptor prefetch) overlaps the append; the producer waits for
    // the append's completion (griddepcontrol.wait) before its first load.
    // CTA pairs: clusters of two CTAs (grid = 2 x pairs)
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    int n = 0;
    if (after_append) {
        attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
    }
    if (PAIR) {
        attr[n].id = cudaLaunchAttributeClusterDimension;
        attr[n].val.clusterDim.x = 2;
        attr[n].val.clusterDim.y = 1;
        attr[n].val.clusterDim.z = 1;
        ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, fa_fwd_kernel<D, FP8, PAIR, CACHE, VAR, STEADY>, q, k, v, o, p);
}

// How many CTA pairs of the kernel can be resident at once (0 if none).
template <int D, bool FP8>
cudaError_t max_resident_pairs(int* pairs) {
    using C = Cfg<D, FP8, true>;
    cudaError_t e = cudaFuncSetAttribute(fa_fwd_kernel<D, FP8, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemBytes);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(2u);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = C::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaOccupancyMaxActiveClusters(pairs, fa_fwd_kernel<D, FP8, true>, &cfg);
}

}  // namespace fa
