/*
 * attn_oracle.c -- the parity oracle for the attention forward pass.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may call, link or
 * load this file: it exists so that tests, the smoke check and the CPU
 * baseline leg of the benchmark have an independent, obviously correct
 * answer to compare the CUDA path against.  It shares no code, header,
 * table or constant with the CUDA path.
 *
 * What it computes (plain definition, fp64, no tiling, no online softmax):
 * exact softmax attention, the method that the FlashAttention papers
 * reach tile by tile ("FlashAttention: Fast and Memory-Efficient Exact
 * Attention with IO-Awareness", arXiv:2205.14135, cited as the algorithmic
 * background by the page "FlashAttention SM120 forward reuses the SM80
 * mainloop", reference [8]).  For one query row i of head h in batch b:
 *
 *     s_j   = scale * sum_d q_id k_jd            for j in the visible set V_i
 *     M     = max_j s_j
 *     L     = sum_j exp(s_j - M)
 *     O_i   = sum_j exp(s_j - M) v_j / L
 *     LSE_i = M + ln L                            (natural log)
 *
 * V_i is {0..Sk-1} without a mask and {j : j <= i + Sk - Sq} with the
 * causal mask (bottom-right alignment; identical to top-left when Sq == Sk).
 * When V_i is empty, O_i = 0 and LSE_i = -inf: the "store_zero" rule of the
 * epilogue in the page "FlashAttention core algorithm: forward pass"
 * (epilogue excerpt: all-zero O, -inf LSE).
 *
 * Grouped-query attention: K and V may have fewer heads (heads_k) than Q;
 * query head h reads key/value head h / (heads / heads_k).  heads_k = heads is
 * ordinary multi-head attention.
 *
 * FP8 inputs: the page "FlashAttention core algorithm: forward pass"
 * (consumer mainloop excerpt, FP8 branch) folds q_descale * k_descale into
 * the softmax scale of a work tile and the output is scaled by the V descale.
 * Both are the same as attending over the dequantised values x8 * descale,
 * which is what this oracle does: every input element is decoded exactly to
 * fp64 and multiplied by its descale in fp64.  A work tile belongs to one
 * (batch, head), so a descale may differ per (batch, key/value head): the
 * descale of row (b, h) is descale[b * stride_b + (h / group) * stride_h]
 * (strides 0, 0: one value for the whole tensor).  Each of Q, K, V has its
 * own storage type, so V may be E5M2 while Q and K are E4M3.
 *
 * Per-batch key lengths (seqused_k, optional): sequence b attends over its
 * first seqused_k[b] keys only -- a key/value cache filled up to that length
 * inside a larger fixed-capacity buffer.  orc_append_kv writes new key/value
 * rows into such a cache at each sequence's current length ("load the new KV
 * before attention" in the page's AppendKV branch of the producer loop).
 *
 * Layouts: fixed length   Q [B, Sq, H, D], K/V [B, Sk, Hk, D]
 *          packed varlen  Q [total_q, H, D], K/V [total_k, Hk, D] with
 *                         cu_seqlens (host int32 [B + 1]).
 * The caller chooses which rows to evaluate as (b, h, i) triples.
 */
#include <math.h>
#include <stddef.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F64 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_E5M2 = 3 };

/* bf16 is the top half of an IEEE binary32: widen by placing the 16 bits
 * in the high half.  Exact. */
static double orc_bf16_to_f64(uint16_t bits) {
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn" variant): 1 sign, 4 exponent bits (bias 7), 3 mantissa
 * bits, no infinities, S.1111.111 is NaN.  Exponent field 0 is subnormal:
 * m/8 * 2^-6.  Otherwise (1 + m/8) * 2^(e-7).  Exact in fp64. */
static double orc_e4m3_to_f64(uint8_t bits) {
    int sign = (bits >> 7) & 1;
    int e = (bits >> 3) & 0xF;
    int m = bits & 0x7;
    double mag;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0) mag = ldexp((double)m / 8.0, -6);
    else mag = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -mag : mag;
}

/* OCP FP8 E5M2: 1 sign, 5 exponent bits (bias 15), 2 mantissa bits, with
 * infinities (exponent 31, m = 0) and NaNs (exponent 31, m != 0).  Exponent
 * field 0 is subnormal: m/4 * 2^-14.  Otherwise (1 + m/4) * 2^(e-15). */
static double orc_e5m2_to_f64(uint8_t bits) {
    int sign = (bits >> 7) & 1;
    int e = (bits >> 2) & 0x1F;
    int m = bits & 0x3;
    double mag;
    if (e == 0x1F) {
        if (m != 0) return NAN;
        mag = INFINITY;
    } else if (e == 0) {
        mag = ldexp((double)m / 4.0, -14);
    } else {
        mag = ldexp(1.0 + (double)m / 4.0, e - 15);
    }
    return sign ? -mag : mag;
}

static double orc_load(const void* base, int dtype, int64_t idx) {
    switch (dtype) {
    case ORC_F64: return ((const double*)base)[idx];
    case ORC_BF16: return orc_bf16_to_f64(((const uint16_t*)base)[idx]);
    case ORC_E4M3: return orc_e4m3_to_f64(((const uint8_t*)base)[idx]);
    case ORC_E5M2: return orc_e5m2_to_f64(((const uint8_t*)base)[idx]);
    default: return NAN;
    }
}

static int orc_elem_bytes(int dtype) {
    return dtype == ORC_F64 ? 8 : dtype == ORC_BF16 ? 2 : 1;
}

/* Decode n elements of the given storage type to fp64 (exposed so the
 * decoders can be pinned against independent library conversions). */
int orc_decode(int dtype, const void* src, double* dst, int64_t n) {
    if (dtype < ORC_F64 || dtype > ORC_E5M2) return 1;
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_load(src, dtype, i);
    return 0;
}

/*
 * Evaluate n_rows query rows.  rows[3r + 0..2] = (b, h, i).
 * q/k/v_dtype: storage type of each tensor (ORC_*).
 * q/k/v_descale: NULL (= 1) or fp64 arrays indexed b * descale_stride_b +
 *          (h / group) * descale_stride_h.
 * seqused_k: NULL, or host int32 [batch]: sequence b uses its first
 *          seqused_k[b] keys (at most its stored length).
 * o_out  : [n_rows, dv] fp64
 * lse_out: [n_rows]     fp64
 * p_out  : optional [n_rows, p_stride] fp64 softmax probabilities over key
 *          index j (masked keys get 0); p_stride >= the sequence's Sk.
 * Returns 0, or 1 on a bad argument (nothing written).
 */
int orc_attention_rows(const void* q, const void* k, const void* v,
                       int q_dtype, int k_dtype, int v_dtype,
                       const double* q_descale, const double* k_descale, const double* v_descale,
                       int64_t descale_stride_b, int64_t descale_stride_h,
                       int batch, int heads, int heads_k, int seqlen_q, int seqlen_k,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                       const int32_t* seqused_k,
                       int d, int dv, double softmax_scale, int causal,
                       const int64_t* rows, int64_t n_rows,
                       double* o_out, double* lse_out,
                       double* p_out, int64_t p_stride) {
    if (!q || !k || !v || !rows || !o_out || !lse_out) return 1;
    if (q_dtype < ORC_F64 || q_dtype > ORC_E5M2 || k_dtype < ORC_F64 || k_dtype > ORC_E5M2 ||
        v_dtype < ORC_F64 || v_dtype > ORC_E5M2)
        return 1;
    if (batch < 0 || heads < 1 || d < 1 || dv < 1) return 1;
    if (heads_k < 1 || heads % heads_k != 0) return 1;
    if (descale_stride_b < 0 || descale_stride_h < 0) return 1;
    const int group = heads / heads_k;  /* query heads per key/value head */
    if ((cu_seqlens_q == NULL) != (cu_seqlens_k == NULL)) return 1;
    int varlen = cu_seqlens_q != NULL;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= batch || h < 0 || h >= heads || i < 0) return 1;
        int64_t sq = varlen ? cu_seqlens_q[b + 1] - cu_seqlens_q[b] : seqlen_q;
        int64_t sk = varlen ? cu_seqlens_k[b + 1] - cu_seqlens_k[b] : seqlen_k;
        if (seqused_k) {
            if (seqused_k[b] < 0 || seqused_k[b] > sk) return 1;
            sk = seqused_k[b];
        }
        if (i >= sq || sk < 0) return 1;
        if (p_out && p_stride < sk) return 1;
    }

    #pragma omp parallel for schedule(dynamic, 16)
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        int64_t sq, sk, q_row, k_row0;
        if (varlen) {
            sq = cu_seqlens_q[b + 1] - cu_seqlens_q[b];
            sk = cu_seqlens_k[b + 1] - cu_seqlens_k[b];
            q_row = cu_seqlens_q[b] + i;
            k_row0 = cu_seqlens_k[b];
        } else {
            sq = seqlen_q;
            sk = seqlen_k;
            q_row = b * (int64_t)seqlen_q + i;
            k_row0 = b * (int64_t)seqlen_k;
        }
        if (seqused_k) sk = seqused_k[b];
        /* visible keys are j = 0 .. n_vis - 1 */
        int64_t n_vis = sk;
        if (causal) {
            int64_t last = i + sk - sq;          /* bottom-right aligned diagonal */
            n_vis = last < 0 ? 0 : (last + 1 < sk ? last + 1 : sk);
        }
        double* o_row = o_out + r * (int64_t)dv;
        double* p_row = p_out ? p_out + r * p_stride : NULL;
        if (p_row) for (int64_t j = 0; j < p_stride; ++j) p_row[j] = 0.0;
        if (n_vis == 0) {
            for (int c = 0; c < dv; ++c) o_row[c] = 0.0;
            lse_out[r] = -INFINITY;
            continue;
        }
        double* s = (double*)malloc(sizeof(double) * (size_t)n_vis);
        int64_t q_off = (q_row * heads + h) * (int64_t)d;
        const int64_t hk = h / group;  /* the key/value head this query head reads */
        const int64_t ds = b * descale_stride_b + hk * descale_stride_h;
        const double qd = q_descale ? q_descale[ds] : 1.0;
        const double kd = k_descale ? k_descale[ds] : 1.0;
        const double vd = v_descale ? v_descale[ds] : 1.0;
        /* scores */
        for (int64_t j = 0; j < n_vis; ++j) {
            int64_t k_off = ((k_row0 + j) * heads_k + hk) * (int64_t)d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += (orc_load(q, q_dtype, q_off + c) * qd) *
                       (orc_load(k, k_dtype, k_off + c) * kd);
            s[j] = softmax_scale * acc;
        }
        /* max, normaliser */
        double m = s[0];
        for (int64_t j = 1; j < n_vis; ++j) if (s[j] > m) m = s[j];
        double l = 0.0;
        for (int64_t j = 0; j < n_vis; ++j) l += exp(s[j] - m);
        /* output */
        for (int c = 0; c < dv; ++c) o_row[c] = 0.0;
        for (int64_t j = 0; j < n_vis; ++j) {
            double p = exp(s[j] - m) / l;
            if (p_row) p_row[j] = p;
            int64_t v_off = ((k_row0 + j) * heads_k + hk) * (int64_t)dv;
            for (int c = 0; c < dv; ++c)
                o_row[c] += p * (orc_load(v, v_dtype, v_off + c) * vd);
        }
        lse_out[r] = m + log(l);
        free(s);
    }
    return 0;
}

/*
 * Append new key/value rows to a fixed-capacity cache, in place:
 *   cache[b, seqlens[b] + i, hk, :] = new_rows[b, i, hk, :]   for i < n_new
 * cache    : [batch, capacity, heads_k, width] of the given storage type
 * new_rows : [batch, n_new, heads_k, width], same storage type
 * seqlens  : host int32 [batch], the filled length of each sequence before
 *            the append; seqlens[b] + n_new must not exceed the capacity.
 * Element bytes are copied unchanged (no conversion).  Returns 0, or 1 on a
 * bad argument (nothing written).
 */
int orc_append_kv(void* cache, const void* new_rows, int dtype, int batch, int capacity,
                  int heads_k, int width, const int32_t* seqlens, int n_new) {
    if (!cache || !seqlens || (n_new > 0 && !new_rows)) return 1;
    if (dtype < ORC_F64 || dtype > ORC_E5M2 || batch < 0 || capacity < 0 || heads_k < 1 ||
        width < 1 || n_new < 0)
        return 1;
    for (int b = 0; b < batch; ++b)
        if (seqlens[b] < 0 || (int64_t)seqlens[b] + n_new > capacity) return 1;
    const int64_t row_bytes = (int64_t)heads_k * width * orc_elem_bytes(dtype);
    for (int b = 0; b < batch; ++b)
        for (int i = 0; i < n_new; ++i)
            memcpy((char*)cache + ((int64_t)b * capacity + seqlens[b] + i) * row_bytes,
                   (const char*)new_rows + ((int64_t)b * n_new + i) * row_bytes, (size_t)row_bytes);
    return 0;
}
