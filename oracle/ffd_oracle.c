/*
 * ffd_oracle.c -- CPU oracle for Faster Flash Decoding (FFD) sparse decode attention.
 *
 * TEST INFRASTRUCTURE ONLY. This is the plain, slow statement of what the FFD decode step
 * computes, used to check the CUDA library. Only the test-suite, the package smoke check and the
 * benchmark's CPU-baseline / reference leg load it. The product library never links, loads or
 * calls it, and the two share no code, header, table or constant.
 *
 * Source: "Faster Than Flash: Exploiting Attention Sparsity for Efficient Long-Context Decoding"
 * (technical summaries; the Japanese, Korean and German pages carry the same text), section
 * "Methodology":
 *   §1 "Content-aware scanning via low-bit quantization": K is split into a 2-bit thumbnail used
 *      to estimate scores and an 8-bit residual that rebuilds K close to fp16 precision.
 *   §2 "Top-delta selection": token j is kept when s_ij >= m~_i - delta; m~_i is a pseudo-max
 *      taken over the sink (initial) tokens and the local tokens only.
 *   §3 "Fused kernel": stage 1 pseudo-max from sink + local tokens; stage 2 streams the 2-bit
 *      keys, computes provisional scores and filters blocks against the threshold; stage 3
 *      loads the 8-bit residuals and V of the selected blocks and computes exact attention.
 *
 * The pages fix neither the thumbnail format nor the block size. The format used here (asymmetric
 * 2-bit codes per group of 32 channels with one fp16 scale and one fp16 zero; symmetric int8
 * residual K - dequant2(K) with one fp16 scale per group; 64-token blocks; score scale 1/sqrt(d))
 * is the library's stated format. Readings of points the pages leave open are listed where they
 * are used ("Reading:").
 *
 * Precision: the quantiser is fp32 with single-rounded IEEE operations, so its outputs are
 * bit-defined; everything in attention is fp64. Build with -ffp-contract=off: every fused
 * multiply-add below is written as fma()/fmaf() on purpose and no other may be formed.
 *
 * The oracle's own layout of the quantised cache (plain arrays; the tests unpack the library's
 * per-tile records, whose layout include/ffd.h states, into it):
 *   k, v      bf16 bits   [P][Hkv][64][128]
 *   thumb     u8          [P][Hkv][64][32]   channel c -> byte c/4, bits 2*(c%4)..2*(c%4)+1
 *   t_scale   f16 bits    [P][Hkv][64][4]    one per group of 32 channels
 *   t_zero    f16 bits    [P][Hkv][64][4]
 *   resid     i8          [P][Hkv][64][128]
 *   r_scale   f16 bits    [P][Hkv][64][4]
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define D 128
#define BLK 64
#define NGROUP 4
#define GSIZE 32

/* ------------------------------------------------------------------------------------------ */
/* Number formats (IEEE-754 binary16 and bfloat16), written from their definitions.            */
/* ------------------------------------------------------------------------------------------ */

/* bfloat16 is the upper half of a binary32: widening is exact. */
float ffdo_f32_from_bf16(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits; subnormal spacing 2^-24. */
float ffdo_f32_from_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int m = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return (float)(sign ? -v : v);
}

/* Round a binary32 to the nearest binary16, ties to even (IEEE default rounding).
 * The value is scaled so that one unit in the last place of its binade is 1.0, rounded with
 * nearbyint() (round-to-nearest-even in the default mode), and scaled back. */
uint16_t ffdo_f16_from_f32(float f) {
    uint16_t sign = signbit(f) ? 0x8000u : 0u;
    if (isnan(f)) return (uint16_t)(sign | 0x7E00u);
    double a = fabs((double)f);
    if (a == 0.0) return sign;
    if (isinf(f)) return (uint16_t)(sign | 0x7C00u);
    int e2;
    frexp(a, &e2);          /* a in [2^(e2-1), 2^e2) */
    int E = e2 - 1;         /* binade exponent */
    if (E < -14) E = -14;   /* below the normal range the spacing stays 2^-24 */
    double units = nearbyint(ldexp(a, 10 - E)); /* exact scaling, then RN-even */
    double val = ldexp(units, E - 10);
    if (val > 65504.0) return (uint16_t)(sign | 0x7C00u);
    if (val < ldexp(1.0, -14)) /* subnormal (or zero) */
        return (uint16_t)(sign | (uint16_t)ldexp(val, 24));
    int ve;
    double frac = frexp(val, &ve); /* val = frac * 2^ve, frac in [0.5, 1) */
    int biased = ve - 1 + 15;
    uint16_t mant = (uint16_t)(ldexp(frac, 11) - 1024.0);
    return (uint16_t)(sign | (uint16_t)(biased << 10) | mant);
}

/* ------------------------------------------------------------------------------------------ */
/* Methodology §1: 2-bit thumbnail + 8-bit residual of one group of 32 key channels.          */
/* ------------------------------------------------------------------------------------------ */

/* Quantise one group. x: 32 channel values of one token and one KV head (exact fp32 copies of
 * bf16 keys). Outputs: 2-bit codes c2, fp16 scale/zero of the thumbnail, int8 residual codes
 * c8 and the residual's fp16 scale.
 * Reading (the pages give only "2-bit thumbnail" and "8-bit residual"):
 *   zero  = f16(min x); scale = f16((max x - min x) / 3); codes use the stored fp16 values;
 *   c2    = clamp(rint((x - zero) / scale), 0, 3), 0 when the stored scale is 0;
 *   x^2   = fma(c2, scale, zero)   (the thumbnail's dequantised key, "dequant2");
 *   r     = x - x^2;  r_scale = f16(max|r| / 127);
 *   c8    = clamp(rint(r / r_scale), -127, 127), 0 when the stored r_scale is 0;
 *   rint  = round half to even. Every operation is one IEEE fp32 operation, rounded once.
 *   A signed-zero minimum or maximum counts as +0.
 * Returns 0, or 1 when an input lies outside the fp16 range (precondition |x| < 65504). */
int ffdo_quantize_group(const float *x, uint8_t *c2, uint16_t *t_scale, uint16_t *t_zero,
                        int8_t *c8, uint16_t *r_scale) {
    float mn = x[0], mx = x[0];
    int bad = 0;
    for (int c = 0; c < GSIZE; c++) {
        if (!(fabsf(x[c]) < 65504.0f)) bad = 1;
        if (x[c] < mn) mn = x[c];
        if (x[c] > mx) mx = x[c];
    }
    /* Reading: -0 and +0 compare equal, so which one is "the minimum" is not defined by the
     * comparison; a zero extreme is taken as +0. */
    if (mn == 0.0f) mn = 0.0f;
    if (mx == 0.0f) mx = 0.0f;
    uint16_t zf16 = ffdo_f16_from_f32(mn);
    float range = mx - mn;
    float step = range / 3.0f;
    uint16_t sf16 = ffdo_f16_from_f32(step);
    float zf = ffdo_f32_from_f16(zf16);
    float sf = ffdo_f32_from_f16(sf16);

    float r[GSIZE];
    float amax = 0.0f;
    for (int c = 0; c < GSIZE; c++) {
        int code = 0;
        if (sf != 0.0f) {
            float t = (x[c] - zf) / sf;
            float k = nearbyintf(t);
            if (k < 0.0f) k = 0.0f;
            if (k > 3.0f) k = 3.0f;
            code = (int)k;
        }
        c2[c] = (uint8_t)code;
        float xh = fmaf((float)code, sf, zf);
        r[c] = x[c] - xh;
        float ar = fabsf(r[c]);
        if (ar > amax) amax = ar;
    }
    uint16_t sr16 = ffdo_f16_from_f32(amax / 127.0f);
    float sr = ffdo_f32_from_f16(sr16);
    for (int c = 0; c < GSIZE; c++) {
        int code = 0;
        if (sr != 0.0f) {
            float k = nearbyintf(r[c] / sr);
            if (k < -127.0f) k = -127.0f;
            if (k > 127.0f) k = 127.0f;
            code = (int)k;
        }
        c8[c] = (int8_t)code;
    }
    *t_scale = sf16;
    *t_zero = zf16;
    *r_scale = sr16;
    return bad;
}

/* Quantise tiles [tile_begin, tile_end) of a cache laid out as [tiles][64][128] (a tile is one
 * page of one KV head, so tiles = P * Hkv). Writes the packed thumbnail, its scales and zeros,
 * the int8 residual and its scales in the layout given at the top of this file.
 * Returns the number of groups that violated the |x| < 65504 precondition. */
int64_t ffdo_quantize_tiles(int64_t tile_begin, int64_t tile_end, const uint16_t *k_bf16,
                            uint8_t *thumb, uint16_t *t_scale, uint16_t *t_zero, int8_t *resid,
                            uint16_t *r_scale) {
    int64_t bad = 0;
    for (int64_t t = tile_begin; t < tile_end; t++) {
        for (int j = 0; j < BLK; j++) {
            int64_t row = t * BLK + j;
            uint8_t *th = thumb + row * (D / 4);
            memset(th, 0, D / 4);
            for (int g = 0; g < NGROUP; g++) {
                float x[GSIZE];
                for (int c = 0; c < GSIZE; c++)
                    x[c] = ffdo_f32_from_bf16(k_bf16[row * D + g * GSIZE + c]);
                uint8_t c2[GSIZE];
                int8_t c8[GSIZE];
                bad += ffdo_quantize_group(x, c2, &t_scale[row * NGROUP + g],
                                           &t_zero[row * NGROUP + g], c8,
                                           &r_scale[row * NGROUP + g]);
                for (int c = 0; c < GSIZE; c++) {
                    int ch = g * GSIZE + c;
                    th[ch / 4] |= (uint8_t)(c2[c] << (2 * (ch % 4)));
                    resid[row * D + ch] = c8[c];
                }
            }
        }
    }
    return bad;
}

/* Dequantise one cached token from the stored format: x^2 (thumbnail only) and
 * K^ = fma(c8, r_scale, x^2) (thumbnail + residual), both fp32 per channel. */
void ffdo_dequant_token(const uint8_t *th, const uint16_t *ts, const uint16_t *tz, const int8_t *rs,
                        const uint16_t *rsc, float *xhat2, float *khat) {
    for (int c = 0; c < D; c++) {
        int g = c / GSIZE;
        int code = (th[c / 4] >> (2 * (c % 4))) & 3;
        float sf = ffdo_f32_from_f16(ts[g]);
        float zf = ffdo_f32_from_f16(tz[g]);
        float sr = ffdo_f32_from_f16(rsc[g]);
        float x2 = fmaf((float)code, sf, zf);
        xhat2[c] = x2;
        khat[c] = fmaf((float)rs[c], sr, x2);
    }
}

/* ------------------------------------------------------------------------------------------ */
/* Methodology §2-§3: one (sequence, KV head) decode step.                                     */
/* ------------------------------------------------------------------------------------------ */

/* Token j of a sequence of length n belongs to the sink set when j < S and to the local set
 * when j >= n - L (Methodology §2, pseudo-max approximation). */
static int in_sink_or_local(int j, int n, int S, int L) {
    return j < S || j >= n - L;
}

/* Locate the cache row of token j: logical block j/64 maps to a physical page through the
 * sequence's block-table row; the row inside the [P][Hkv][64] tile array follows. */
static int64_t token_row(const int32_t *pages, int num_kv_heads, int h, int j) {
    int64_t page = pages[j / BLK];
    return (page * num_kv_heads + h) * BLK + (j % BLK);
}

static double dot_q(const double *qrow, const float *k) {
    double s = 0.0;
    for (int c = 0; c < D; c++) s += qrow[c] * (double)k[c];
    return s;
}

/* FFD decode for one sequence and one KV head, i.e. its G query heads (GQA group).
 *   q        bf16 bits [G][128], the group's query rows
 *   pages    [ceil(n/64)] physical page of each logical block
 *   mask_in  optional [nb]: use this block mask instead of the Top-delta rule (stages 1 and 2
 *            are still computed and reported)
 * Outputs:
 *   out      [G][128] attention output, fp64
 *   m_tilde  [G] pseudo-max (-inf when the sink and local sets are empty)
 *   mask_out [nb] 1 = block kept
 *   margin   [nb] max over the block's tokens j < n and heads i of s^_ij - (m~_i - delta):
 *            the block passes the Top-delta rule iff margin >= 0. NaN marks forced blocks.
 *   s_hat    optional [G][n] provisional (thumbnail) scores
 *
 * Steps, in the pages' order (Methodology §3):
 *   stage 1  m~_i = max over j in sink U local of s_ij,  s_ij = sm * q_i . K^_j  (exact scores;
 *            Reading: the pages say only "sink and local tokens"; the exact reconstruction is
 *            used, and m~ is per query head i as the subscript in the keep rule shows).
 *   stage 2  s^_ij = sm * q_i . x^2_j for every token; block b (tokens 64b .. 64b+63, < n) is
 *            kept when it holds a sink or local token, or when some head i of the group and some
 *            token j of the block give s^_ij >= m~_i - delta.
 *            Reading: the rule is stated per token and applied per block ("filters blocks"); a
 *            block is kept if any token passes for any head of the group; the comparison is >=.
 *   stage 3  exact softmax over the kept tokens only (dropped tokens contribute nothing):
 *            out_i = sum_j e^(s_ij - M_i) V_j / sum_j e^(s_ij - M_i),  M_i = max_j s_ij.
 * n == 0 gives out = 0. Returns 0, or 2 when a page index is out of range. */
int ffdo_decode_unit(int G, int n, int S, int L, double delta, double sm_scale,
                     const uint16_t *q, const int32_t *pages, int num_pages, int num_kv_heads,
                     int h, const uint8_t *thumb, const uint16_t *t_scale, const uint16_t *t_zero,
                     const int8_t *resid, const uint16_t *r_scale, const uint16_t *v,
                     const uint8_t *mask_in, double *out, double *m_tilde, uint8_t *mask_out,
                     double *margin, double *s_hat) {
    int nb = (n + BLK - 1) / BLK;
    for (int b = 0; b < nb; b++)
        if (pages[b] < 0 || pages[b] >= num_pages) return 2;

    double *qd = (double *)malloc(sizeof(double) * (size_t)G * D);
    for (int i = 0; i < G * D; i++) qd[i] = (double)ffdo_f32_from_bf16(q[i]);
    float xh2[D], kh[D];

    /* Stage 1: pseudo-max over the sink and local tokens, exact scores. */
    for (int i = 0; i < G; i++) m_tilde[i] = -INFINITY;
    for (int j = 0; j < n; j++) {
        if (!in_sink_or_local(j, n, S, L)) continue;
        int64_t row = token_row(pages, num_kv_heads, h, j);
        ffdo_dequant_token(thumb + row * (D / 4), t_scale + row * NGROUP, t_zero + row * NGROUP,
                           resid + row * D, r_scale + row * NGROUP, xh2, kh);
        for (int i = 0; i < G; i++) {
            double s = sm_scale * dot_q(qd + i * D, kh);
            if (s > m_tilde[i]) m_tilde[i] = s;
        }
    }

    /* Stage 2: provisional scores from the 2-bit thumbnail; block filter. */
    for (int b = 0; b < nb; b++) {
        int forced = 0;
        double mg = -INFINITY;
        for (int j = b * BLK; j < (b + 1) * BLK && j < n; j++) {
            if (in_sink_or_local(j, n, S, L)) forced = 1;
            int64_t row = token_row(pages, num_kv_heads, h, j);
            ffdo_dequant_token(thumb + row * (D / 4), t_scale + row * NGROUP,
                               t_zero + row * NGROUP, resid + row * D, r_scale + row * NGROUP,
                               xh2, kh);
            for (int i = 0; i < G; i++) {
                double sh = sm_scale * dot_q(qd + i * D, xh2);
                if (s_hat) s_hat[(size_t)i * n + j] = sh;
                double thr = m_tilde[i] - delta;
                double d = sh - thr;
                if (d > mg) mg = d;
            }
        }
        margin[b] = forced ? NAN : mg;
        int keep = forced || mg >= 0.0;
        mask_out[b] = (uint8_t)(mask_in ? (mask_in[b] != 0) : keep);
    }

    /* Stage 3: exact attention over the kept tokens. */
    double *sc = (double *)malloc(sizeof(double) * (size_t)G * (n > 0 ? n : 1));
    double *M = (double *)malloc(sizeof(double) * (size_t)G);
    double *den = (double *)calloc((size_t)G, sizeof(double));
    double *num = (double *)calloc((size_t)G * D, sizeof(double));
    for (int i = 0; i < G; i++) M[i] = -INFINITY;
    for (int j = 0; j < n; j++) {
        if (!mask_out[j / BLK]) continue;
        int64_t row = token_row(pages, num_kv_heads, h, j);
        ffdo_dequant_token(thumb + row * (D / 4), t_scale + row * NGROUP, t_zero + row * NGROUP,
                           resid + row * D, r_scale + row * NGROUP, xh2, kh);
        for (int i = 0; i < G; i++) {
            double s = sm_scale * dot_q(qd + i * D, kh);
            sc[(size_t)i * n + j] = s;
            if (s > M[i]) M[i] = s;
        }
    }
    for (int j = 0; j < n; j++) {
        if (!mask_out[j / BLK]) continue;
        int64_t row = token_row(pages, num_kv_heads, h, j);
        for (int i = 0; i < G; i++) {
            double p = exp(sc[(size_t)i * n + j] - M[i]);
            den[i] += p;
            for (int c = 0; c < D; c++)
                num[i * D + c] += p * (double)ffdo_f32_from_bf16(v[row * D + c]);
        }
    }
    for (int i = 0; i < G; i++)
        for (int c = 0; c < D; c++)
            out[i * D + c] = den[i] > 0.0 ? num[i * D + c] / den[i] : 0.0;
    free(num);
    free(den);
    free(M);
    free(sc);
    free(qd);
    return 0;
}

/* Dense decode attention for one sequence and one KV head over the original bf16 keys (the
 * comparison kernel's definition: standard softmax attention over every token, no selection).
 *   out_i = sum_j e^(s_ij - M_i) V_j / sum_j e^(s_ij - M_i),  s_ij = sm * q_i . K_j.
 * Returns 0, or 2 when a page index is out of range. */
int ffdo_dense_unit(int G, int n, double sm_scale, const uint16_t *q, const int32_t *pages,
                    int num_pages, int num_kv_heads, int h, const uint16_t *k, const uint16_t *v,
                    double *out) {
    int nb = (n + BLK - 1) / BLK;
    for (int b = 0; b < nb; b++)
        if (pages[b] < 0 || pages[b] >= num_pages) return 2;
    double *sc = (double *)malloc(sizeof(double) * (n > 0 ? n : 1));
    float kf[D];
    for (int i = 0; i < G; i++) {
        double qd[D];
        for (int c = 0; c < D; c++) qd[c] = (double)ffdo_f32_from_bf16(q[i * D + c]);
        double M = -INFINITY;
        for (int j = 0; j < n; j++) {
            int64_t row = token_row(pages, num_kv_heads, h, j);
            for (int c = 0; c < D; c++) kf[c] = ffdo_f32_from_bf16(k[row * D + c]);
            sc[j] = sm_scale * dot_q(qd, kf);
            if (sc[j] > M) M = sc[j];
        }
        double den = 0.0, num[D];
        for (int c = 0; c < D; c++) num[c] = 0.0;
        for (int j = 0; j < n; j++) {
            int64_t row = token_row(pages, num_kv_heads, h, j);
            double p = exp(sc[j] - M);
            den += p;
            for (int c = 0; c < D; c++) num[c] += p * (double)ffdo_f32_from_bf16(v[row * D + c]);
        }
        for (int c = 0; c < D; c++) out[i * D + c] = den > 0.0 ? num[c] / den : 0.0;
    }
    free(sc);
    return 0;
}
