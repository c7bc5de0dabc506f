/*
 * CPU oracle for the routed Q4_0 x Q8_1 MoE expert matmul.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the CPU
 * baseline leg of the benchmark; never by the CUDA library.  See ft_oracle.h
 * for the byte layouts and the list of pins.
 *
 * Sources.  The pages describe one computation, the per-(token, top-k slot)
 * dot product of the routed expert's Q4_0 weight rows with the token's Q8_1
 * activation (FreeToken PR #185, "Problem": moe_vec_q4_0_q8_1 over the flat
 * (token, top-k) index), its quantizer quantize_row_q8_1 ("Fix"), and the
 * expert-grouped form built on expert_offsets with a leading 0 and a
 * searchsorted(right=True) slot-to-expert map (nvfp4-megamoe-kernel
 * CURRENT_BUG.md, Bugs 2 and 4).  The pages do not print the block formats;
 * they are the GGUF Q4_0 / Q8_1 formats restated in ft_oracle.h.
 *
 * Readings where the pages are silent:
 *   - "round" is round-half-away-from-zero (C roundf);
 *   - Q8_1 divides by the fp32 scale amax/127, not by its fp16 value;
 *   - s = fp16(d32 * (float)sum(q)) with d32 the fp32 scale;
 *   - the dot uses the exact integer sum of (q_w - 8) * q_a per block and
 *     never the rounded s;
 *   - for every weight type with an offset (the m of Q4_1 / Q5_1, the mins of
 *     the K-quants) the offset term is m * d_a * sum(q_a): the dequantized
 *     activation is d_a * q_a, so its block sum is d_a times the exact sum of
 *     the codes; the stored s, that sum rounded to fp16, is never used;
 *   - slots whose expert id is out of range are left out of the routing and
 *     produce zero output rows.
 *
 * Build: plain C99, -ffp-contract=off so that no multiply-add is fused.
 */
#include "ft_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

#define QK 32
#define Q4_0_BYTES 18
#define Q8_1_BYTES 36

/* ------------------------------------------------------------------ fp16 */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (exp == 0)
        v = ldexp((double)frac, -24);                    /* zero / subnormal */
    else if (exp == 31)
        v = frac ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + frac), exp - 25);      /* 1.frac * 2^(exp-15) */
    return sign ? -v : v;
}

/* Round a float to the nearest binary16, ties to even. */
uint16_t oracle_float_to_half(float f)
{
    double a = fabs((double)f);
    uint16_t sign = signbit(f) ? 0x8000 : 0;
    if (isnan(f))
        return sign | 0x7e00;
    if (a >= 65520.0)                                    /* past the max finite + half an ulp */
        return sign | 0x7c00;
    if (a < ldexp(1.0, -14)) {                           /* subnormal range: units of 2^-24 */
        double q = nearbyint(a * ldexp(1.0, 24));        /* default mode: to nearest, ties even */
        return sign | (uint16_t)q;                       /* q == 1024 encodes the smallest normal */
    }
    int e;
    double m = frexp(a, &e);                             /* a = m * 2^e, m in [0.5, 1) */
    double q = nearbyint(m * 2048.0);                    /* 11 significant bits */
    if (q == 2048.0) {
        q = 1024.0;
        e += 1;
    }
    int biased = e - 1 + 15;
    if (biased >= 31)
        return sign | 0x7c00;
    return sign | (uint16_t)(biased << 10) | (uint16_t)((int)q - 1024);
}

static uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
static void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)(v & 0xff); p[1] = (uint8_t)(v >> 8); }

/* ------------------------------------------------------------------ Q4_0 */

/* Q4_0 quantizer used for synthetic weights: d = m / -8 where m is the
 * block's element of largest magnitude (first on ties, sign kept),
 * q = clamp(round(w / d) + 8, 0, 15), value (q - 8) * d. */
void oracle_quantize_q4_0(const float* w, int64_t n_blocks, uint8_t* out)
{
    for (int64_t b = 0; b < n_blocks; ++b) {
        const float* x = w + b * QK;
        float m = 0.0f, amax = 0.0f;
        for (int i = 0; i < QK; ++i) {
            if (fabsf(x[i]) > amax) {
                amax = fabsf(x[i]);
                m = x[i];
            }
        }
        float d = m / -8.0f;
        uint8_t q[QK];
        for (int i = 0; i < QK; ++i) {
            int v = 8;
            if (d != 0.0f) {
                v = (int)roundf(x[i] / d) + 8;
                if (v < 0) v = 0;
                if (v > 15) v = 15;
            }
            q[i] = (uint8_t)v;
        }
        uint8_t* o = out + b * Q4_0_BYTES;
        wr16(o, oracle_float_to_half(d));
        for (int j = 0; j < 16; ++j)
            o[2 + j] = (uint8_t)(q[j] | (q[j + 16] << 4));
    }
}

static int q4_0_nibble(const uint8_t* block, int i)
{
    const uint8_t* qs = block + 2;
    return i < 16 ? (qs[i] & 0x0f) : (qs[i - 16] >> 4);
}

void oracle_dequantize_q4_0(const uint8_t* blocks, int64_t n_blocks, double* out)
{
    for (int64_t b = 0; b < n_blocks; ++b) {
        const uint8_t* blk = blocks + b * Q4_0_BYTES;
        double d = oracle_half_to_double(rd16(blk));
        for (int i = 0; i < QK; ++i)
            out[b * QK + i] = (double)(q4_0_nibble(blk, i) - 8) * d;
    }
}

/* ------------------------------------------------------------------ Q8_1 */

/* Activation quantizer (quantize_row_q8_1 on FreeToken PR #185, "Fix"),
 * per 32-block of an fp16 row, in fp32: amax = max |x|, d = amax / 127,
 * q = round(x / d) clamped to [-127, 127] (0 when amax == 0), s = d * sum q.
 * d and s are stored as fp16. */
/* One Q8_1 block from 32 fp32 values, in single precision as quantize_row_q8_1
 * defines it (FreeToken PR #185, "Fix"): d = amax / 127, q = round(x / d)
 * clamped to [-127, 127], s = d * sum(q); d and s stored as fp16. */
static void quantize_block_q8_1(const float* x, uint8_t* o)
{
    float amax = 0.0f;
    for (int i = 0; i < QK; ++i)
        if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    float d = amax / 127.0f;
    int sum = 0;
    for (int i = 0; i < QK; ++i) {
        int q = 0;
        if (amax != 0.0f) {
            q = (int)roundf(x[i] / d);
            if (q < -127) q = -127;
            if (q > 127) q = 127;
        }
        sum += q;
        o[4 + i] = (uint8_t)(int8_t)q;
    }
    float s = d * (float)sum;
    wr16(o, oracle_float_to_half(d));
    wr16(o + 2, oracle_float_to_half(s));
}

void oracle_quantize_q8_1(const uint16_t* x_fp16, int64_t tokens, int64_t ncols, uint8_t* out)
{
    int64_t nb = ncols / QK;
    for (int64_t t = 0; t < tokens; ++t) {
        for (int64_t b = 0; b < nb; ++b) {
            float x[QK];
            for (int i = 0; i < QK; ++i)
                x[i] = (float)oracle_half_to_double(x_fp16[t * ncols + b * QK + i]);
            quantize_block_q8_1(x, out + (t * nb + b) * Q8_1_BYTES);
        }
    }
}

void oracle_dequantize_q8_1(const uint8_t* blocks, int64_t n_blocks, double* out)
{
    for (int64_t b = 0; b < n_blocks; ++b) {
        const uint8_t* blk = blocks + b * Q8_1_BYTES;
        double d = oracle_half_to_double(rd16(blk));
        for (int i = 0; i < QK; ++i)
            out[b * QK + i] = (double)(int8_t)blk[4 + i] * d;
    }
}

/* ------------------------------------------ other 32-value GGUF weight types */

/* The other GGUF weight types whose blocks hold 32 weights, as matmul weights
 * against the same Q8_1 activations (the 19 per-type launchers of
 * moe_vec.cuh on FreeToken PR #185, "Notes"; the pages exercise only Q4_0 and
 * do not print the formats, restated in ft_oracle.h).  Each weight is
 * w_i = q_i * d + c with an integer level q_i and an offset c (0 or m), so a
 * block's contribution is
 *     d * d_a * sum_i q_i * q_a[i]  +  c * d_a * sum_i q_a[i],
 * and the second term takes d_a * sum(q_a) as the activation block's stored
 * fp16 s (the quantity Q8_1 stores s for).  The K-quants (below) are written
 * as w = d sc q - dmin m per 32-weight sub-block; their min term is taken with
 * the exact d_a * sum(q_a). */
int32_t oracle_gguf_block_bytes(int32_t type)
{
    switch (type) {
        case ORACLE_GGUF_Q4_0: return 18;
        case ORACLE_GGUF_Q4_1: return 20;
        case ORACLE_GGUF_Q5_0: return 22;
        case ORACLE_GGUF_Q5_1: return 24;
        case ORACLE_GGUF_Q8_0: return 34;
        case ORACLE_GGUF_Q4_K: return 144;
        case ORACLE_GGUF_Q5_K: return 176;
        case ORACLE_GGUF_Q6_K: return 210;
        case ORACLE_GGUF_Q2_K: return 84;
        case ORACLE_GGUF_Q3_K: return 110;
        default: return 0;
    }
}

/* Integer level q_i of weight i of a block. */
static int gguf_level(const uint8_t* blk, int32_t type, int i)
{
    int nib, hi5;
    uint32_t qh;
    switch (type) {
        case ORACLE_GGUF_Q4_0:
            return q4_0_nibble(blk, i) - 8;
        case ORACLE_GGUF_Q4_1:
            return i < 16 ? (blk[4 + i] & 0x0f) : (blk[4 + i - 16] >> 4);
        case ORACLE_GGUF_Q5_0:
        case ORACLE_GGUF_Q5_1: {
            const uint8_t* h = blk + (type == ORACLE_GGUF_Q5_0 ? 2 : 4);
            const uint8_t* qs = h + 4;
            qh = (uint32_t)h[0] | ((uint32_t)h[1] << 8) | ((uint32_t)h[2] << 16) | ((uint32_t)h[3] << 24);
            nib = i < 16 ? (qs[i] & 0x0f) : (qs[i - 16] >> 4);
            hi5 = (int)((qh >> i) & 1u);
            return (nib | (hi5 << 4)) - (type == ORACLE_GGUF_Q5_0 ? 16 : 0);
        }
        case ORACLE_GGUF_Q8_0:
            return (int)(int8_t)blk[2 + i];
        default:
            abort();
    }
}

/* Offset c of a block: the fp16 m of Q4_1 / Q5_1, else 0. */
static double gguf_offset(const uint8_t* blk, int32_t type)
{
    if (type == ORACLE_GGUF_Q4_1 || type == ORACLE_GGUF_Q5_1)
        return oracle_half_to_double(rd16(blk + 2));
    return 0.0;
}

/* K-quant super-blocks (Q4_K 144 B, Q5_K 176 B) hold 256 weights as eight
 * sub-blocks of 32: fp16 d, fp16 dmin, 12 bytes of packed 6-bit scale/min
 * pairs, then (Q5_K only) 32 bytes qh of 5th bits, then 128 bytes of
 * nibbles.  Sub-block j uses nibble byte 32 * (j / 2) + l, its low nibble for
 * even j and its high nibble for odd j, and (Q5_K) bit j of qh[l] as the 5th
 * bit; weight l = d * sc_j * q_l - dmin * m_j.  The pair (sc_j, m_j): for
 * j < 4 the low 6 bits of bytes j and j + 4; for j >= 4 the low nibble of byte
 * j + 4 with the top two bits of byte j - 4 above it, and the high nibble of
 * byte j + 4 with the top two bits of byte j above it. */
static int is_kquant(int32_t type)
{
    return type == ORACLE_GGUF_Q4_K || type == ORACLE_GGUF_Q5_K || type == ORACLE_GGUF_Q6_K ||
           type == ORACLE_GGUF_Q2_K || type == ORACLE_GGUF_Q3_K;
}

/* The two K-quants with 2-bit codes, 256 weights per super-block in two
 * halves of 128; sub-block j = 4 h + k (k < 4) of half h takes, for weight
 * l < 32, bits 2k, 2k + 1 of code byte 32 h + l, and its weights l < 16 use
 * scale group 2 j, weights l >= 16 group 2 j + 1.
 *   Q2_K  84 B: 16 scale bytes (low nibble scale, high nibble min, one per
 *         group), 64 code bytes, fp16 d, fp16 dmin;
 *         weight = d * scale * q - dmin * min, q = the 2-bit code.
 *   Q3_K 110 B: 32 bytes hmask, 64 code bytes, 12 bytes of sixteen packed
 *         6-bit scales, fp16 d; bit j of hmask[l] is the third bit of weight
 *         l of sub-block j, level q = (2-bit code | third bit << 2) - 4;
 *         weight = d * (scale - 32) * q.  The 6-bit scale of group g: its low
 *         four bits are the low (g < 8) or high (g >= 8) nibble of byte g % 8,
 *         its top two bits are bits 2 (g / 4 % 4) .. +1 of byte 8 + g % 4. */
static void q2k3k_sub(const uint8_t* sb, int32_t type, int j, int* lev, double* s_lo, double* s_hi,
                      double* m_lo, double* m_hi)
{
    const int h = j / 4, k = j % 4;
    const uint8_t* q = sb + (type == ORACLE_GGUF_Q2_K ? 16 : 32) + 32 * h;
    for (int l = 0; l < QK; ++l) {
        int v = (q[l] >> (2 * k)) & 3;
        if (type == ORACLE_GGUF_Q3_K)
            v = (v | (((sb[l] >> j) & 1) << 2)) - 4;
        lev[l] = v;
    }
    if (type == ORACLE_GGUF_Q2_K) {
        const double d = oracle_half_to_double(rd16(sb + 80)), dmin = oracle_half_to_double(rd16(sb + 82));
        *s_lo = d * (sb[2 * j] & 0x0f);
        *s_hi = d * (sb[2 * j + 1] & 0x0f);
        *m_lo = dmin * (sb[2 * j] >> 4);
        *m_hi = dmin * (sb[2 * j + 1] >> 4);
    } else {
        const double d = oracle_half_to_double(rd16(sb + 108));
        const uint8_t* sc = sb + 96;
        int g, v6[2];
        for (int i = 0; i < 2; ++i) {
            g = 2 * j + i;
            const int low4 = g < 8 ? (sc[g % 8] & 0x0f) : (sc[g % 8] >> 4);
            const int top2 = (sc[8 + g % 4] >> (2 * (g / 4))) & 3;
            v6[i] = (low4 | (top2 << 4)) - 32;
        }
        *s_lo = d * v6[0];
        *s_hi = d * v6[1];
        *m_lo = *m_hi = 0.0;
    }
}

/* Q6_K, 210 B per 256 weights: 128 B ql (low nibbles), 64 B qh (2-bit high
 * parts), 16 int8 scales, fp16 d last.  The super-block is two halves of 128
 * weights; sub-block j = 4 h + k (k < 4) of half h takes, for weight l < 32,
 * nibble byte 64 h + 32 (k % 2) + l (low nibble for k < 2, high for k >= 2),
 * bits 2k, 2k + 1 of byte 128 + 32 h + l as bits 4, 5, and level
 * q = that 6-bit value - 32; weights l < 16 use scale 8 h + 2 k, l >= 16 scale
 * 8 h + 2 k + 1: weight = d * scale * q. */
static void q6k_sub(const uint8_t* sb, int j, int* lev, double* dsc_lo, double* dsc_hi)
{
    const int h = j / 4, k = j % 4;
    const double d = oracle_half_to_double(rd16(sb + 208));
    *dsc_lo = d * (double)(int8_t)sb[192 + 8 * h + 2 * k];
    *dsc_hi = d * (double)(int8_t)sb[192 + 8 * h + 2 * k + 1];
    for (int l = 0; l < QK; ++l) {
        const uint8_t ql = sb[64 * h + 32 * (k % 2) + l];
        const int lo4 = k < 2 ? (ql & 0x0f) : (ql >> 4);
        const int hi2 = (sb[128 + 32 * h + l] >> (2 * k)) & 3;
        lev[l] = (lo4 | (hi2 << 4)) - 32;
    }
}

static void kquant_scale_min(const uint8_t* sc12, int j, int* sc, int* m)
{
    if (j < 4) {
        *sc = sc12[j] & 63;
        *m = sc12[j + 4] & 63;
    } else {
        *sc = (sc12[j + 4] & 0x0f) | ((sc12[j - 4] >> 6) << 4);
        *m = (sc12[j + 4] >> 4) | ((sc12[j] >> 6) << 4);
    }
}

/* Sub-block j of a K-quant super-block: its 32 levels, d * sc_j and dmin * m_j. */
static void kquant_sub(const uint8_t* sb, int32_t type, int j, int* lev, double* dsc, double* dmn)
{
    int sc, m;
    kquant_scale_min(sb + 4, j, &sc, &m);
    *dsc = oracle_half_to_double(rd16(sb)) * sc;
    *dmn = oracle_half_to_double(rd16(sb + 2)) * m;
    const uint8_t* qs = sb + (type == ORACLE_GGUF_Q5_K ? 48 : 16) + 32 * (j / 2);
    for (int l = 0; l < QK; ++l) {
        lev[l] = (j % 2 == 0) ? (qs[l] & 0x0f) : (qs[l] >> 4);
        if (type == ORACLE_GGUF_Q5_K)
            lev[l] |= ((sb[16 + l] >> j) & 1) << 4;
    }
}

void oracle_dequantize_gguf(int32_t type, const uint8_t* blocks, int64_t n_blocks, double* out)
{
    const int32_t bytes = oracle_gguf_block_bytes(type);
    if (type == ORACLE_GGUF_Q2_K || type == ORACLE_GGUF_Q3_K) {
        for (int64_t b = 0; b < n_blocks; ++b)
            for (int j = 0; j < 8; ++j) {
                int lev[QK];
                double slo, shi, mlo, mhi;
                q2k3k_sub(blocks + b * bytes, type, j, lev, &slo, &shi, &mlo, &mhi);
                for (int l = 0; l < QK; ++l)
                    out[b * 256 + j * QK + l] = l < 16 ? slo * lev[l] - mlo : shi * lev[l] - mhi;
            }
        return;
    }
    if (type == ORACLE_GGUF_Q6_K) {
        for (int64_t b = 0; b < n_blocks; ++b)
            for (int j = 0; j < 8; ++j) {
                int lev[QK];
                double dlo, dhi;
                q6k_sub(blocks + b * bytes, j, lev, &dlo, &dhi);
                for (int l = 0; l < QK; ++l)
                    out[b * 256 + j * QK + l] = (l < 16 ? dlo : dhi) * lev[l];
            }
        return;
    }
    if (is_kquant(type)) {
        for (int64_t b = 0; b < n_blocks; ++b)
            for (int j = 0; j < 8; ++j) {
                int lev[QK];
                double dsc, dmn;
                kquant_sub(blocks + b * bytes, type, j, lev, &dsc, &dmn);
                for (int l = 0; l < QK; ++l)
                    out[b * 256 + j * QK + l] = dsc * lev[l] - dmn;
            }
        return;
    }
    for (int64_t b = 0; b < n_blocks; ++b) {
        const uint8_t* blk = blocks + b * bytes;
        double d = oracle_half_to_double(rd16(blk));
        double c = gguf_offset(blk, type);
        for (int i = 0; i < QK; ++i)
            out[b * QK + i] = (double)gguf_level(blk, type, i) * d + c;
    }
}

int32_t oracle_gguf_block_dot(int32_t type, const uint8_t* w_block, const uint8_t* a_block)
{
    int32_t acc = 0;
    for (int i = 0; i < QK; ++i)
        acc += gguf_level(w_block, type, i) * (int32_t)(int8_t)a_block[4 + i];
    return acc;
}

void oracle_moe_gguf_q8_1(int32_t type, const uint8_t* weights, const uint8_t* act, const int32_t* topk_ids,
                          float* out, int64_t tokens, int32_t top_k, int32_t n_experts,
                          int64_t nrows, int64_t ncols)
{
    const int64_t nb = ncols / QK;
    const int32_t bytes = oracle_gguf_block_bytes(type);
    const int64_t n_slots = tokens * top_k;
    for (int64_t s = 0; s < n_slots; ++s) {
        const int32_t e = topk_ids[s];
        const int64_t t = s / top_k;
        for (int64_t r = 0; r < nrows; ++r) {
            double y = 0.0;
            if (e >= 0 && e < n_experts && is_kquant(type)) {
                /* sub-block b of the row = sub-block b % 8 of super-block b / 8:
                 * d sc d_a sum(q q_a) - dmin m d_a sum(q_a), the exact sum of q_a */
                const uint8_t* row = weights + ((int64_t)e * nrows + r) * (nb / 8) * bytes;
                for (int64_t b = 0; b < nb; ++b) {
                    int lev[QK];
                    double dsc, dmn;
                    if (type == ORACLE_GGUF_Q2_K || type == ORACLE_GGUF_Q3_K) {
                        /* two 16-weight groups per 32-block, each with its scale and
                         * (Q2_K) min: s_g d_a sum_g(q q_a) - m_g d_a sum_g(q_a) */
                        double slo, shi, mlo, mhi;
                        q2k3k_sub(row + (b / 8) * bytes, type, (int)(b % 8), lev, &slo, &shi, &mlo, &mhi);
                        const uint8_t* ab2 = act + (t * nb + b) * Q8_1_BYTES;
                        const double da2 = oracle_half_to_double(rd16(ab2));
                        int32_t dot_lo = 0, dot_hi = 0, sum_lo = 0, sum_hi = 0;
                        for (int l = 0; l < QK; ++l) {
                            const int32_t qa = (int32_t)(int8_t)ab2[4 + l];
                            if (l < 16) {
                                dot_lo += lev[l] * qa;
                                sum_lo += qa;
                            } else {
                                dot_hi += lev[l] * qa;
                                sum_hi += qa;
                            }
                        }
                        y += slo * da2 * (double)dot_lo + shi * da2 * (double)dot_hi -
                             mlo * da2 * (double)sum_lo - mhi * da2 * (double)sum_hi;
                        continue;
                    }
                    if (type == ORACLE_GGUF_Q6_K) {
                        /* two 16-weight scale groups per 32-block: d sc_lo d_a sum_lo + d sc_hi d_a sum_hi */
                        double dlo, dhi;
                        q6k_sub(row + (b / 8) * bytes, (int)(b % 8), lev, &dlo, &dhi);
                        const uint8_t* ab6 = act + (t * nb + b) * Q8_1_BYTES;
                        const double da6 = oracle_half_to_double(rd16(ab6));
                        int32_t dlo_i = 0, dhi_i = 0;
                        for (int l = 0; l < QK; ++l) {
                            if (l < 16) dlo_i += lev[l] * (int32_t)(int8_t)ab6[4 + l];
                            else dhi_i += lev[l] * (int32_t)(int8_t)ab6[4 + l];
                        }
                        y += dlo * da6 * (double)dlo_i + dhi * da6 * (double)dhi_i;
                        continue;
                    }
                    kquant_sub(row + (b / 8) * bytes, type, (int)(b % 8), lev, &dsc, &dmn);
                    const uint8_t* ab = act + (t * nb + b) * Q8_1_BYTES;
                    const double da = oracle_half_to_double(rd16(ab));
                    int32_t dot = 0, suma = 0;
                    for (int l = 0; l < QK; ++l) {
                        dot += lev[l] * (int32_t)(int8_t)ab[4 + l];
                        suma += (int32_t)(int8_t)ab[4 + l];
                    }
                    y += dsc * da * (double)dot - dmn * da * (double)suma;
                }
            } else if (e >= 0 && e < n_experts) {
                for (int64_t b = 0; b < nb; ++b) {
                    /* d_w d_a sum(q q_a) + m d_a sum(q_a), the exact sum of q_a */
                    const uint8_t* wb = weights + (((int64_t)e * nrows + r) * nb + b) * bytes;
                    const uint8_t* ab = act + (t * nb + b) * Q8_1_BYTES;
                    double dw = oracle_half_to_double(rd16(wb));
                    double da = oracle_half_to_double(rd16(ab));
                    int32_t suma = 0;
                    for (int l = 0; l < QK; ++l) suma += (int32_t)(int8_t)ab[4 + l];
                    y += dw * da * (double)oracle_gguf_block_dot(type, wb, ab) +
                         gguf_offset(wb, type) * da * (double)suma;
                }
            }
            out[s * nrows + r] = (float)y;
        }
    }
}

/* ----------------------------------------------- SoA repack of Q4_0 weights */

/* The one-time repack of Q4_0 weight blocks from their stored array of
 * 18-byte structures (fp16 d, 16 nibble bytes) into a structure of arrays:
 * all nibble bytes, 16 per block in block order, then all scales, one fp16
 * per block in block order.  Nothing is converted: the bytes move. */
void oracle_repack_q4_0_soa(const uint8_t* blocks, int64_t n_blocks, uint8_t* qs, uint16_t* d)
{
    for (int64_t b = 0; b < n_blocks; ++b) {
        d[b] = rd16(blocks + b * Q4_0_BYTES);
        memcpy(qs + b * 16, blocks + b * Q4_0_BYTES + 2, 16);
    }
}

/* ----------------------------------------------------- gated activation */

/* The two gated activations that sit between the expert layers: GELU in its
 * tanh form (flashinfer gelu_tanh_and_mul, called right after the routed
 * matmul on FreeToken PR #185, "Problem") and SiLU (the "SiLU*up" step between
 * the two expert layers on nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 6).
 *   silu(g)      = g / (1 + exp(-g))
 *   gelu_tanh(g) = g/2 * (1 + tanh(y)),  y = sqrt(2/pi) * (g + 0.044715 g^3)
 * Both in fp64.  gelu_tanh is evaluated as g / (1 + exp(-2 y)), the same
 * function since (1 + tanh(y)) / 2 = 1 / (1 + exp(-2 y)): written with tanh,
 * 1 + tanh(y) cancels to nothing (or to a few ulps of 1) for g below about -6,
 * where the exact value is tiny but not zero. */
static double act_fn(double g, int32_t kind)
{
    if (kind == ORACLE_ACT_SILU)
        return g / (1.0 + exp(-g));
    const double y = sqrt(2.0 / 3.14159265358979323846) * (g + 0.044715 * g * g * g);
    return g / (1.0 + exp(-2.0 * y));
}

/* a[r][i] = act(h[r][i]) * h[r][n_inter + i], computed in fp64 and rounded
 * once to fp32: the first half of each row of h is the gate, the second half
 * the up projection (the gate/up row order of the fused expert weight). */
void oracle_act_mul(const float* h, int64_t rows, int64_t n_inter, int32_t kind, float* a)
{
    for (int64_t r = 0; r < rows; ++r) {
        const float* hr = h + r * 2 * n_inter;
        for (int64_t i = 0; i < n_inter; ++i)
            a[r * n_inter + i] = (float)(act_fn((double)hr[i], kind) * (double)hr[n_inter + i]);
    }
}

/* oracle_act_mul followed by the Q8_1 quantizer on its fp32 result, one Q8_1
 * row of n_inter / 32 blocks per row of h. */
void oracle_act_mul_quantize_q8_1(const float* h, int64_t rows, int64_t n_inter, int32_t kind, uint8_t* out)
{
    int64_t nb = n_inter / QK;
    float* a = (float*)malloc((size_t)(n_inter > 0 ? n_inter : 1) * sizeof(float));
    if (!a) abort();
    for (int64_t r = 0; r < rows; ++r) {
        oracle_act_mul(h + r * 2 * n_inter, 1, n_inter, kind, a);
        for (int64_t b = 0; b < nb; ++b)
            quantize_block_q8_1(a + b * QK, out + (r * nb + b) * Q8_1_BYTES);
    }
    free(a);
}

/* ----------------------------------------------------------------- route */

/* Stable counting sort of the flat slots by expert id.
 * counts[e] = number of slots routed to e; offsets has E+1 entries with a
 * leading 0 (nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 4), offsets[e+1] =
 * offsets[e] + counts[e]; perm[offsets[e] + r] = the r-th slot, in ascending
 * slot order, whose id is e.  Positions p with offsets[e] <= p < offsets[e+1]
 * belong to expert e, which is the searchsorted(right=True) map of Bug 2.
 * Slots with ids outside [0, E) are left out; perm past offsets[E] is -1.
 * Returns the number of such slots. */
int64_t oracle_route(const int32_t* topk_ids, int64_t n_slots, int32_t n_experts,
                     int32_t* counts, int32_t* offsets, int32_t* perm)
{
    int64_t bad = 0;
    for (int32_t e = 0; e < n_experts; ++e) counts[e] = 0;
    for (int64_t s = 0; s < n_slots; ++s) {
        int32_t e = topk_ids[s];
        if (e < 0 || e >= n_experts) { ++bad; continue; }
        counts[e] += 1;
    }
    offsets[0] = 0;
    for (int32_t e = 0; e < n_experts; ++e) offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)calloc((size_t)n_experts + 1, sizeof(int32_t));
    for (int64_t s = 0; s < n_slots; ++s) {
        int32_t e = topk_ids[s];
        if (e < 0 || e >= n_experts) continue;
        perm[offsets[e] + cursor[e]] = (int32_t)s;
        cursor[e] += 1;
    }
    free(cursor);
    for (int64_t p = offsets[n_experts]; p < n_slots; ++p) perm[p] = -1;
    return bad;
}

/* ------------------------------------------------------------------- dot */

/* Exact integer dot of one Q4_0 block with one Q8_1 block:
 * sum_i (q_w[i] - 8) * q_a[i]; |result| <= 32 * 8 * 127 = 32512. */
int32_t oracle_block_dot(const uint8_t* w_block, const uint8_t* a_block)
{
    int32_t acc = 0;
    for (int i = 0; i < QK; ++i)
        acc += (q4_0_nibble(w_block, i) - 8) * (int32_t)(int8_t)a_block[4 + i];
    return acc;
}

/* y[s, r] = sum_b d_w[e(s), r, b] * d_a[t(s), b] * dot_b, t(s) = s / k,
 * e(s) = topk_ids[s]; fp64 sum in block order; 0 for a bad id. */
static double moe_one(const uint8_t* weights, const uint8_t* act, const int32_t* topk_ids,
                      int32_t top_k, int32_t n_experts, int64_t nrows, int64_t ncols,
                      int64_t s, int64_t r)
{
    int64_t nb = ncols / QK;
    int32_t e = topk_ids[s];
    if (e < 0 || e >= n_experts)
        return 0.0;
    int64_t t = s / top_k;
    const uint8_t* wrow = weights + ((int64_t)e * nrows + r) * nb * Q4_0_BYTES;
    const uint8_t* arow = act + t * nb * Q8_1_BYTES;
    double y = 0.0;
    for (int64_t b = 0; b < nb; ++b) {
        const uint8_t* wb = wrow + b * Q4_0_BYTES;
        const uint8_t* ab = arow + b * Q8_1_BYTES;
        double dw = oracle_half_to_double(rd16(wb));
        double da = oracle_half_to_double(rd16(ab));
        y += dw * da * (double)oracle_block_dot(wb, ab);
    }
    return y;
}

void oracle_moe_q4_0_q8_1(const uint8_t* weights, const uint8_t* act, const int32_t* topk_ids,
                          float* out, int64_t tokens, int32_t top_k, int32_t n_experts,
                          int64_t nrows, int64_t ncols)
{
    int64_t n_slots = tokens * top_k;
    for (int64_t s = 0; s < n_slots; ++s)
        for (int64_t r = 0; r < nrows; ++r)
            out[s * nrows + r] = (float)moe_one(weights, act, topk_ids, top_k, n_experts,
                                                nrows, ncols, s, r);
}

/* Per-slot activations (the second expert layer's input, one Q8_1 row per
 * routed slot, nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 6: L2 runs on the L1
 * output after SiLU*up): out[s][r] as above with activation row s instead of
 * row s / top_k. */
void oracle_moe_slots_q4_0_q8_1(const uint8_t* weights, const uint8_t* act_slots, const int32_t* topk_ids,
                                float* out, int64_t tokens, int32_t top_k, int32_t n_experts,
                                int64_t nrows, int64_t ncols)
{
    int64_t nb = ncols / QK;
    int64_t n_slots = tokens * top_k;
    for (int64_t s = 0; s < n_slots; ++s) {
        int32_t e = topk_ids[s];
        const uint8_t* arow = act_slots + s * nb * Q8_1_BYTES;
        for (int64_t r = 0; r < nrows; ++r) {
            double y = 0.0;
            if (e >= 0 && e < n_experts) {
                const uint8_t* wrow = weights + ((int64_t)e * nrows + r) * nb * Q4_0_BYTES;
                for (int64_t b = 0; b < nb; ++b) {
                    const uint8_t* wb = wrow + b * Q4_0_BYTES;
                    const uint8_t* ab = arow + b * Q8_1_BYTES;
                    double dw = oracle_half_to_double(rd16(wb));
                    double da = oracle_half_to_double(rd16(ab));
                    y += dw * da * (double)oracle_block_dot(wb, ab);
                }
            }
            out[s * nrows + r] = (float)y;
        }
    }
}

/* Expert-parallel shard (nvfp4-megamoe-kernel CURRENT_BUG.md, Bug 8: global
 * expert ids, remapped by the shard's first expert, non-local slots masked):
 * weights_local holds experts [expert_start, expert_start + n_local) of
 * n_global; a slot whose global id g lies in that range is computed with
 * local expert g - expert_start, every other slot's row is 0. */
void oracle_moe_ep_q4_0_q8_1(const uint8_t* weights_local, const uint8_t* act, const int32_t* topk_ids,
                             float* out, int64_t tokens, int32_t top_k, int32_t n_global,
                             int32_t expert_start, int32_t n_local, int64_t nrows, int64_t ncols)
{
    int64_t nb = ncols / QK;
    int64_t n_slots = tokens * top_k;
    (void)n_global;
    for (int64_t s = 0; s < n_slots; ++s) {
        int32_t g = topk_ids[s];
        int64_t t = s / top_k;
        const uint8_t* arow = act + t * nb * Q8_1_BYTES;
        for (int64_t r = 0; r < nrows; ++r) {
            double y = 0.0;
            if (g >= expert_start && g < expert_start + n_local) {
                int32_t e = g - expert_start;
                const uint8_t* wrow = weights_local + ((int64_t)e * nrows + r) * nb * Q4_0_BYTES;
                for (int64_t b = 0; b < nb; ++b) {
                    const uint8_t* wb = wrow + b * Q4_0_BYTES;
                    const uint8_t* ab = arow + b * Q8_1_BYTES;
                    double dw = oracle_half_to_double(rd16(wb));
                    double da = oracle_half_to_double(rd16(ab));
                    y += dw * da * (double)oracle_block_dot(wb, ab);
                }
            }
            out[s * nrows + r] = (float)y;
        }
    }
}

void oracle_moe_sample(const uint8_t* weights, const uint8_t* act, const int32_t* topk_ids,
                       int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows,
                       int64_t ncols, const int64_t* slots, const int64_t* rows, int64_t n,
                       double* out)
{
    (void)tokens;
    for (int64_t i = 0; i < n; ++i)
        out[i] = moe_one(weights, act, topk_ids, top_k, n_experts, nrows, ncols, slots[i], rows[i]);
}

/* dots[s][r][b] = the exact block dot; 0 for a bad id. */
void oracle_moe_block_dots(const uint8_t* weights, const uint8_t* act, const int32_t* topk_ids,
                           int64_t tokens, int32_t top_k, int32_t n_experts, int64_t nrows,
                           int64_t ncols, int32_t* dots)
{
    int64_t nb = ncols / QK;
    int64_t n_slots = tokens * top_k;
    for (int64_t s = 0; s < n_slots; ++s) {
        int32_t e = topk_ids[s];
        int64_t t = s / top_k;
        for (int64_t r = 0; r < nrows; ++r)
            for (int64_t b = 0; b < nb; ++b) {
                int32_t v = 0;
                if (e >= 0 && e < n_experts)
                    v = oracle_block_dot(weights + (((int64_t)e * nrows + r) * nb + b) * Q4_0_BYTES,
                                         act + (t * nb + b) * Q8_1_BYTES);
                dots[(s * nrows + r) * nb + b] = v;
            }
    }
}

/* Dequantize both operands to fp64 values and take the plain dot over K. */
void oracle_moe_dequant_bruteforce(const uint8_t* weights, const uint8_t* act,
                                   const int32_t* topk_ids, int64_t tokens, int32_t top_k,
                                   int32_t n_experts, int64_t nrows, int64_t ncols, double* out)
{
    int64_t nb = ncols / QK;
    int64_t n_slots = tokens * top_k;
    double* wv = (double*)malloc((size_t)ncols * sizeof(double));
    double* av = (double*)malloc((size_t)ncols * sizeof(double));
    for (int64_t s = 0; s < n_slots; ++s) {
        int32_t e = topk_ids[s];
        int64_t t = s / top_k;
        oracle_dequantize_q8_1(act + t * nb * Q8_1_BYTES, nb, av);
        for (int64_t r = 0; r < nrows; ++r) {
            double y = 0.0;
            if (e >= 0 && e < n_experts) {
                oracle_dequantize_q4_0(weights + ((int64_t)e * nrows + r) * nb * Q4_0_BYTES, nb, wv);
                for (int64_t i = 0; i < ncols; ++i)
                    y += wv[i] * av[i];
            }
            out[s * nrows + r] = y;
        }
    }
    free(wv);
    free(av);
}
