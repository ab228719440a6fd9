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
 * the softmax scale and the output is scaled by the V descale.  Both are the
 * same as attending over the dequantised values x8 * descale, which is what
 * this oracle does: every input element is decoded exactly to fp64 and
 * multiplied by its tensor's descale in fp64.
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

enum { ORC_F64 = 0, ORC_BF16 = 1, ORC_E4M3 = 2 };

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

static double orc_load(const void* base, int dtype, int64_t idx) {
    switch (dtype) {
    case ORC_F64: return ((const double*)base)[idx];
    case ORC_BF16: return orc_bf16_to_f64(((const uint16_t*)base)[idx]);
    case ORC_E4M3: return orc_e4m3_to_f64(((const uint8_t*)base)[idx]);
    default: return NAN;
    }
}

/* Decode n elements of the given storage type to fp64 (exposed so the
 * decoders can be pinned against independent library conversions). */
int orc_decode(int dtype, const void* src, double* dst, int64_t n) {
    if (dtype < ORC_F64 || dtype > ORC_E4M3) return 1;
    for (int64_t i = 0; i < n; ++i) dst[i] = orc_load(src, dtype, i);
    return 0;
}

/*
 * Evaluate n_rows query rows.  rows[3r + 0..2] = (b, h, i).
 * o_out  : [n_rows, dv] fp64
 * lse_out: [n_rows]     fp64
 * p_out  : optional [n_rows, p_stride] fp64 softmax probabilities over key
 *          index j (masked keys get 0); p_stride >= the sequence's Sk.
 * Returns 0, or 1 on a bad argument (nothing written).
 */
int orc_attention_rows(const void* q, const void* k, const void* v, int dtype,
                       double q_descale, double k_descale, double v_descale,
                       int batch, int heads, int heads_k, int seqlen_q, int seqlen_k,
                       const int32_t* cu_seqlens_q, const int32_t* cu_seqlens_k,
                       int d, int dv, double softmax_scale, int causal,
                       const int64_t* rows, int64_t n_rows,
                       double* o_out, double* lse_out,
                       double* p_out, int64_t p_stride) {
    if (!q || !k || !v || !rows || !o_out || !lse_out) return 1;
    if (dtype < ORC_F64 || dtype > ORC_E4M3 || batch < 0 || heads < 1 || d < 1 || dv < 1) return 1;
    if (heads_k < 1 || heads % heads_k != 0) return 1;
    const int group = heads / heads_k;  /* query heads per key/value head */
    if ((cu_seqlens_q == NULL) != (cu_seqlens_k == NULL)) return 1;
    int varlen = cu_seqlens_q != NULL;
    for (int64_t r = 0; r < n_rows; ++r) {
        int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
        if (b < 0 || b >= batch || h < 0 || h >= heads || i < 0) return 1;
        int64_t sq = varlen ? cu_seqlens_q[b + 1] - cu_seqlens_q[b] : seqlen_q;
        int64_t sk = varlen ? cu_seqlens_k[b + 1] - cu_seqlens_k[b] : seqlen_k;
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
        /* scores */
        for (int64_t j = 0; j < n_vis; ++j) {
            int64_t k_off = ((k_row0 + j) * heads_k + hk) * (int64_t)d;
            double acc = 0.0;
            for (int c = 0; c < d; ++c)
                acc += (orc_load(q, dtype, q_off + c) * q_descale) *
                       (orc_load(k, dtype, k_off + c) * k_descale);
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
                o_row[c] += p * (orc_load(v, dtype, v_off + c) * v_descale);
        }
        lse_out[r] = m + log(l);
        free(s);
    }
    return 0;
}
