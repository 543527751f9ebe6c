/*
 * Oracle for block-quantized prefill GEMMs and the routed-MoE expert stage.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the library's product path may link,
 * load or call this file: only the tests, the smoke check and the bench's CPU
 * baseline do.  It shares no code, header, table or helper with the CUDA path.
 *
 * Plain, slow and literal: every weight is dequantised in fp32 (the products
 * e2m1 x E4M3 and E4M3 alone are exact there) and every dot product is summed
 * in fp64 in ascending k.  OpenMP only splits independent output elements.
 * Built with -ffp-contract=off so that no multiply-add is fused behind our back
 * (the pages warn that a compiler contracting a multiply into an FMA broke a
 * byte-exact quantiser: "AMD_HIP.md", gfx906 notes on the Q8_K quantiser).
 *
 * Sources of each step (page title, then section / commit):
 *  - W4 weights, e2m1 codes with one E4M3 scale per 16 K and an fp32 scale2
 *    applied once: "perf: strix-hip BF16 GEMMs via hipBLASLt", commit
 *    "f16a twins for the dense M128 and routed-MoE kernels".
 *  - FP8 weights with one fp32 scale per 128x128 block, each 128-K block summed
 *    unscaled and folded once (acc += blk * scale): same page, commit "FP8
 *    ... 128-K block scaling twin".
 *  - Expert stage: gate/up, SwiGLU, H rounded to q8_1 blocks of 32, down over
 *    IQ4_NL, weighted sum of the top-k experts: "Run Edge0-145B Q3_K on AMD HIP
 *    (Linux, gfx1100)", "Contents" (commit 4cb5224) and that commit's message.
 *  - Top-k routing with renormalised weights: "AMD_HIP.md", RDNA4 speed
 *    switches (router_top10).
 *  - Dense Q8_0 x q8_1 projections re-quantised to q8_1: "Run Edge0-145B Q3_K on
 *    AMD HIP (Linux, gfx1100)", commit 17c02cd's message (lat_dense_w11).
 * Format details the pages leave open (nibble order, codebook, q8_1 rounding)
 * follow the workload statement; each reading is named where it is used.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------ */
/* Scalar formats                                                           */
/* ------------------------------------------------------------------------ */

/* e2m1 (4-bit float, 1 sign, 2 exponent, 1 mantissa bit): bit 3 is the sign,
 * bits 0..2 index the magnitudes {0, 0.5, 1, 1.5, 2, 3, 4, 6}. */
float orc_e2m1(unsigned code)
{
    static const float mag[8] = {0.0f, 0.5f, 1.0f, 1.5f, 2.0f, 3.0f, 4.0f, 6.0f};
    float v = mag[code & 7u];
    return (code & 8u) ? -v : v;
}

/* OCP FP8 E4M3: bias 7, subnormals m/8 * 2^-6, no infinities, NaN only for
 * S.1111.111, largest finite 448. */
float orc_e4m3(unsigned byte)
{
    unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
    double v;
    if (e == 15u && m == 7u)
        return NAN;
    if (e == 0u)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, (int)e - 7);
    return (float)(s ? -v : v);
}

/* IEEE-754 binary16 -> double. */
double orc_f16(uint16_t h)
{
    unsigned s = (h >> 15) & 1u, e = (h >> 10) & 31u, m = h & 1023u;
    double v;
    if (e == 0u)
        v = ldexp((double)m, -24);
    else if (e == 31u)
        v = m ? NAN : INFINITY;
    else
        v = ldexp(1.0 + (double)m / 1024.0, (int)e - 15);
    return s ? -v : v;
}

/* bfloat16 -> float: the top half of a binary32. */
float orc_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* float -> binary16, round to nearest even, overflow to infinity. */
uint16_t orc_f16_rne(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint16_t sign = (uint16_t)((u >> 16) & 0x8000u);
    int e = (int)((u >> 23) & 255u);
    uint32_t m = u & 0x7FFFFFu;
    if (e == 255)                              /* inf / nan */
        return (uint16_t)(sign | 0x7C00u | (m ? 0x200u : 0u));
    if (e == 0 && m == 0)
        return sign;
    /* value = (1.m) * 2^(e-127), or m * 2^-149 for binary32 subnormals */
    uint64_t sig;                              /* integer significand */
    int exp2;                                  /* value = sig * 2^exp2 */
    if (e == 0) { sig = m; exp2 = -149; }
    else        { sig = m | 0x800000u; exp2 = e - 150; }
    /* binary16 keeps 11 significant bits for normals (exponent >= -14) and a
     * fixed quantum 2^-24 for subnormals. Find the quantum q of the result. */
    int msb = 63;
    while (!((sig >> msb) & 1u)) msb--;
    int top = msb + exp2;                      /* floor(log2(value)) */
    int q = (top >= -14) ? top - 10 : -24;     /* quantum exponent */
    uint64_t r;                                /* result in units of 2^q */
    if (exp2 >= q) {
        r = sig << (exp2 - q);
    } else {
        int sh = q - exp2;
        if (sh > 62) {
            r = 0;                             /* far below half the smallest subnormal */
        } else {
            uint64_t keep = sig >> sh, rem = sig & ((1ull << sh) - 1), half = 1ull << (sh - 1);
            r = keep + ((rem > half) || (rem == half && (keep & 1u)));
        }
    }
    /* assemble: r may have carried into the next binade */
    if (q == -24 && r < 1024u)                 /* subnormal (or zero) */
        return (uint16_t)(sign | r);
    if (r >= 2048u) { r >>= 1; q += 1; }       /* carry out of 11 bits (exact: r was 2048) */
    int ebits = q + 10 + 15;                   /* biased exponent of 1.xxx * 2^(q+10) */
    if (ebits >= 31)
        return (uint16_t)(sign | 0x7C00u);
    return (uint16_t)(sign | ((unsigned)ebits << 10) | (unsigned)(r & 1023u));
}

/* ------------------------------------------------------------------------ */
/* Dense W4A16: Y[m,n] = scale2 * sum_k X[m,k] * e2m1(code[n,k]) * e4m3(s[n,k/16]) */
/* ------------------------------------------------------------------------ */

/* Weight element (n, k) of a W4 matrix with K columns: element 2j of a row is
 * the low nibble of byte j, element 2j+1 the high nibble. */
static float w4_weight(const uint8_t *Wc, const uint8_t *Ws, int K, long n, int k)
{
    uint8_t byte = Wc[n * (long)(K / 2) + k / 2];
    unsigned code = (k & 1) ? (byte >> 4) : (byte & 15u);
    float scale = orc_e4m3(Ws[n * (long)(K / 16) + k / 16]);
    return orc_e2m1(code) * scale;                     /* exact in fp32 */
}

/* rows/cols select the output elements computed (NULL: all); Y is
 * [nrows][ncols] in fp64, not rounded to the output type. */
void orc_w4a16(const uint16_t *X, int M, int K, int N,
               const uint8_t *Wc, const uint8_t *Ws, float scale2,
               const int32_t *rows, int nrows, const int32_t *cols, int ncols,
               double *Y)
{
    if (!rows) nrows = M;
    if (!cols) ncols = N;
#pragma omp parallel for collapse(2) schedule(static)
    for (int i = 0; i < nrows; i++) {
        for (int j = 0; j < ncols; j++) {
            long m = rows ? rows[i] : i, n = cols ? cols[j] : j;
            double acc = 0.0;
            for (int k = 0; k < K; k++)
                acc += (double)orc_bf16(X[m * K + k]) * (double)w4_weight(Wc, Ws, K, n, k);
            Y[(long)i * ncols + j] = (double)scale2 * acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Dense FP8, 128x128 block scales:                                          */
/*   Y[m,n] = sum_kb S[n/128, kb] * sum_{k in kb} X[m,k] * e4m3(W[n,k])       */
/* ------------------------------------------------------------------------ */
void orc_fp8_blk128(const uint16_t *X, int M, int K, int N,
                    const uint8_t *W, const float *S,
                    const int32_t *rows, int nrows, const int32_t *cols, int ncols,
                    double *Y)
{
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    int KB = K / 128;
#pragma omp parallel for collapse(2) schedule(static)
    for (int i = 0; i < nrows; i++) {
        for (int j = 0; j < ncols; j++) {
            long m = rows ? rows[i] : i, n = cols ? cols[j] : j;
            double acc = 0.0;
            for (int kb = 0; kb < KB; kb++) {
                double blk = 0.0;
                for (int k = kb * 128; k < kb * 128 + 128; k++)
                    blk += (double)orc_bf16(X[m * K + k]) * (double)orc_e4m3(W[n * (long)K + k]);
                acc += (double)S[(n / 128) * KB + kb] * blk;
            }
            Y[(long)i * ncols + j] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Routing: top-k, renormalised weights, per-expert grouping                 */
/* ------------------------------------------------------------------------ */

/* For each token: the k largest logits (a tie goes to the lower expert index),
 * w_j = exp(l_j - l_max) / sum over the k chosen of exp(l_i - l_max).  Softmax
 * over all E followed by renormalising the k chosen weights gives the same
 * numbers: softmax keeps the order and its normaliser cancels.
 * Grouping: counts[e] pairs chose e; offsets is their exclusive prefix sum
 * (offsets[E] = T*k); the pairs of expert e occupy rows offsets[e].. in
 * ascending (token, slot) order; row[t*k+j] is the row of pair (t, j) and
 * src[row] its token. */
void orc_route(const float *logits, int T, int E, int k,
               int32_t *ids, float *w, int32_t *counts, int32_t *offsets,
               int32_t *src, int32_t *row)
{
#pragma omp parallel for schedule(static)
    for (int t = 0; t < T; t++) {
        const float *l = logits + (long)t * E;
        unsigned char *taken = (unsigned char *)calloc((size_t)E, 1);
        for (int j = 0; j < k; j++) {
            int best = -1;
            for (int e = 0; e < E; e++)
                if (!taken[e] && (best < 0 || l[e] > l[best]))
                    best = e;
            taken[best] = 1;
            ids[(long)t * k + j] = best;
        }
        free(taken);
        double lmax = (double)l[ids[(long)t * k]];
        double den = 0.0;
        for (int j = 0; j < k; j++)
            den += exp((double)l[ids[(long)t * k + j]] - lmax);
        for (int j = 0; j < k; j++)
            w[(long)t * k + j] = (float)(exp((double)l[ids[(long)t * k + j]] - lmax) / den);
    }
    for (int e = 0; e < E; e++)
        counts[e] = 0;
    for (long p = 0; p < (long)T * k; p++)
        counts[ids[p]]++;
    offsets[0] = 0;
    for (int e = 0; e < E; e++)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t *cursor = (int32_t *)malloc(sizeof(int32_t) * (size_t)E);
    memcpy(cursor, offsets, sizeof(int32_t) * (size_t)E);
    for (int t = 0; t < T; t++)
        for (int j = 0; j < k; j++) {
            int e = ids[(long)t * k + j];
            int r = cursor[e]++;
            row[(long)t * k + j] = r;
            src[r] = t;
        }
    free(cursor);
}

/* Expert of a grouped row: the e with offsets[e] <= r < offsets[e+1]. */
static int expert_of_row(const int32_t *offsets, int E, int r)
{
    int e = 0;
    while (e + 1 < E && offsets[e + 1] <= r)
        e++;
    return e;
}

/* ------------------------------------------------------------------------ */
/* Gate/up (W4), SwiGLU, q8_1 rounding of H                                 */
/* ------------------------------------------------------------------------ */

/* One q8_1 block of 32 values: d = max|h| / 127 (fp32 division), q =
 * round-half-away-from-zero(h / d) clamped to +-127, d16 = fp16(d),
 * s16 = fp16(d * sum q).  A block of zeros gets d = q = s = 0. */
void orc_q8_1_block(const float *h, int8_t *q, uint16_t *d16, uint16_t *s16)
{
    float amax = 0.0f;
    for (int i = 0; i < 32; i++)
        if (fabsf(h[i]) > amax)
            amax = fabsf(h[i]);
    if (amax == 0.0f) {
        for (int i = 0; i < 32; i++)
            q[i] = 0;
        *d16 = 0;
        *s16 = 0;
        return;
    }
    float d = amax / 127.0f;
    int sum = 0;
    for (int i = 0; i < 32; i++) {
        float v = roundf(h[i] / d);                    /* roundf: halves away from zero */
        if (v > 127.0f) v = 127.0f;
        if (v < -127.0f) v = -127.0f;
        q[i] = (int8_t)v;
        sum += q[i];
    }
    *d16 = orc_f16_rne(d);
    *s16 = orc_f16_rne(d * (float)sum);
}

/* SwiGLU on fp32 gate/up values: silu(g) * u = g / (1 + e^-g) * u, in fp64,
 * rounded once to fp32. */
float orc_swiglu(float g, float u)
{
    return (float)((double)g / (1.0 + exp(-(double)g)) * (double)u);
}

/* For each selected grouped row r (token src[r], expert e of the row):
 *   g[n] = scale2[e] * sum_k X[t,k] * Wgu[e, n, k],   u[n] = same with row F+n,
 * both rounded to fp32; h = swiglu(g, u); H rounded to q8_1 per 32 columns.
 * Outputs per selected row: Hq [F] int8, Hd/Hs [F/32] fp16 bits, and h [F]
 * (fp32, before rounding) if h_out is not NULL. */
void orc_moe_gate_up_q8_1(const uint16_t *X, int D, int F, int E,
                          const int32_t *offsets, const int32_t *src,
                          const uint8_t *Wgu_c, const uint8_t *Wgu_s, const float *gu_scale2,
                          const int32_t *rows, int nrows,
                          int8_t *Hq, uint16_t *Hd, uint16_t *Hs, float *h_out)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int i = 0; i < nrows; i++) {
        int r = rows[i];
        int e = expert_of_row(offsets, E, r);
        long t = src[r];
        const uint8_t *Wc = Wgu_c + (long)e * 2 * F * (D / 2);
        const uint8_t *Ws = Wgu_s + (long)e * 2 * F * (D / 16);
        float *h = (float *)malloc(sizeof(float) * (size_t)F);
        for (int n = 0; n < F; n++) {
            double g = 0.0, u = 0.0;
            for (int k = 0; k < D; k++) {
                double x = (double)orc_bf16(X[t * D + k]);
                g += x * (double)w4_weight(Wc, Ws, D, n, k);
                u += x * (double)w4_weight(Wc, Ws, D, (long)F + n, k);
            }
            float g32 = (float)((double)gu_scale2[e] * g);
            float u32 = (float)((double)gu_scale2[e] * u);
            h[n] = orc_swiglu(g32, u32);
        }
        for (int b = 0; b < F / 32; b++)
            orc_q8_1_block(h + b * 32, Hq + (long)i * F + b * 32,
                           Hd + (long)i * (F / 32) + b, Hs + (long)i * (F / 32) + b);
        if (h_out)
            memcpy(h_out + (long)i * F, h, sizeof(float) * (size_t)F);
        free(h);
    }
}

/* ------------------------------------------------------------------------ */
/* Down: IQ4_NL weights x q8_1 H, one exact integer dot per 32-block        */
/* ------------------------------------------------------------------------ */

/* IQ4_NL: a 4-bit index into this non-uniform int8 codebook, one fp16 scale
 * per 32 elements. */
static const int orc_iq4nl_codebook[16] = {
    -127, -104, -83, -65, -49, -35, -22, -10, 1, 13, 25, 38, 53, 69, 89, 113};

int orc_iq4nl_value(unsigned idx) { return orc_iq4nl_codebook[idx & 15u]; }

/* For each selected grouped row (its q8_1 codes Hq[i], scales Hd[i] given in
 * selection order, expert from offsets):
 *   y[n] = sum_b fp16(Hd[b]) * fp16(Wd[e,n,b]) * I_b,
 *   I_b  = sum_{k in block b} Hq[k] * codebook[idx[e,n,k]]   (exact integer).
 * Y is [nrows][D] in fp64. */
void orc_moe_down_iq4(const int8_t *Hq, const uint16_t *Hd, int F, int D, int E,
                      const int32_t *offsets, const uint8_t *Wd_idx, const uint16_t *Wd_s,
                      const int32_t *rows, int nrows, double *Y)
{
#pragma omp parallel for collapse(2) schedule(static)
    for (int i = 0; i < nrows; i++) {
        for (int n = 0; n < D; n++) {
            int e = expert_of_row(offsets, E, rows[i]);
            const uint8_t *idx = Wd_idx + ((long)e * D + n) * (F / 2);
            const uint16_t *ws = Wd_s + ((long)e * D + n) * (F / 32);
            double acc = 0.0;
            for (int b = 0; b < F / 32; b++) {
                long long I = 0;
                for (int k = b * 32; k < b * 32 + 32; k++) {
                    uint8_t byte = idx[k / 2];
                    unsigned c = (k & 1) ? (byte >> 4) : (byte & 15u);
                    I += (long long)Hq[(long)i * F + k] * orc_iq4nl_value(c);
                }
                acc += orc_f16(Hd[(long)i * (F / 32) + b]) * orc_f16(ws[b]) * (double)I;
            }
            Y[(long)i * D + n] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Dense Q8_0 weights x q8_1 activations, one exact integer dot per 32-block */
/* ------------------------------------------------------------------------ */

/* The dense latent projections of "Run Edge0-145B Q3_K on AMD HIP (Linux,
 * gfx1100)" (commit 17c02cd's message: Q8_0 x q8_1 integer dots; D re-quantises
 * its products to q8_1 blocks).  Q8_0 is read as 32 int8 codes with one fp16
 * scale per block; the q8_1 activations carry their fp16 d (s is not needed by
 * a symmetric weight format).
 *   y[m,n] = sum_b fp16(Xd[m,b]) * fp16(Wd[n,b]) * I_b,
 *   I_b    = sum_{k in block b} Xq[m,k] * Wq[n,k]      (exact integer).
 * Selected rows / columns (NULL: all); Y is [nrows][ncols] in fp64. */
void orc_q8_0_q8_1(const int8_t *Xq, const uint16_t *Xd, int M, int K, int N,
                   const int8_t *Wq, const uint16_t *Wd,
                   const int32_t *rows, int nrows, const int32_t *cols, int ncols, double *Y)
{
    (void)M;
    (void)N;
#pragma omp parallel for collapse(2) schedule(static)
    for (int i = 0; i < nrows; i++) {
        for (int j = 0; j < ncols; j++) {
            long m = rows ? rows[i] : i;
            long n = cols ? cols[j] : j;
            double acc = 0.0;
            for (int b = 0; b < K / 32; b++) {
                long long I = 0;
                for (int k = b * 32; k < b * 32 + 32; k++)
                    I += (long long)Xq[m * K + k] * (long long)Wq[n * K + k];
                acc += orc_f16(Xd[m * (K / 32) + b]) * orc_f16(Wd[n * (K / 32) + b]) * (double)I;
            }
            Y[(long)i * ncols + j] = acc;
        }
    }
}

/* ------------------------------------------------------------------------ */
/* Weighted combine: Y[t,:] = sum_j w[t,j] * Yslot[row(t,j), :], j ascending  */
/* ------------------------------------------------------------------------ */

/* slot[i*k + j] is the index, in Ys, of the down output of pair (token i, j). */
void orc_moe_combine(const float *w, const int32_t *slot, const double *Ys,
                     int ntok, int k, int D, double *Y)
{
#pragma omp parallel for schedule(static)
    for (int i = 0; i < ntok; i++)
        for (int n = 0; n < D; n++) {
            double acc = 0.0;
            for (int j = 0; j < k; j++)
                acc += (double)w[(long)i * k + j] * Ys[(long)slot[(long)i * k + j] * D + n];
            Y[(long)i * D + n] = acc;
        }
}
