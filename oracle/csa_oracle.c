/*
 * CPU oracle for the CSA2 decode step over an FP4 global KV cache.
 *
 * TEST INFRASTRUCTURE.  Only the test-suite, the smoke check and the timed CPU
 * baseline of the benchmark may load this library.  It shares no code, table
 * or header with the CUDA path; it is plain, slow C in double precision, written
 * so that each function can be checked against its source passage by eye.
 *
 * Sources (web pages on DeepSeek-V4.1-Flash):
 *  [G2C]  "G2C Brief - DeepSeek V4.1-Flash: a model designed around its KV cache",
 *         sections "FP4 cache entries, and why they're safe",
 *         "The global branch: compress, index, select",
 *         "CSA2: most layers don't keep their own cache",
 *         "The hierarchical indexer: making later indexers context-independent".
 *  [FPR]  "DeepSeek V4.1 Flash: Pushing the Limits" (talk write-up), section
 *         "The Paper" (Full / Reindex / Reuse modes).
 *  [MET]  "DeepSeek Retires Its 1.6T Model for a 552B One" (the three modes).
 * The indexer score formula sum_h w_h * ReLU(q_h . k) is not printed on any page;
 * it is the workload statement's formula, used as given.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* Number formats                                                            */
/* ------------------------------------------------------------------------- */

/* bf16: the top 16 bits of an IEEE binary32. */
double oracle_bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP FP8 E4M3 ("fn": no infinities, bias 7, S.1111.111 is NaN, max 448).
 * [G2C] "FP4 cache entries": one 8-bit E4M3 scale per 16 channels. */
double oracle_e4m3_value(uint8_t byte)
{
    int sign = byte >> 7;
    int e = (byte >> 3) & 0xF;
    int m = byte & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);                    /* subnormal: m/8 * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* OCP FP4 E2M1 (bias 1, no inf/NaN): sign bit 3, exponent bits 2..1, mantissa bit 0.
 * [G2C] "FP4 cache entries": main cache entries are 4-bit floats (E2M1). */
double oracle_e2m1_value(uint8_t code)
{
    int sign = (code >> 3) & 1;
    int e = (code >> 1) & 0x3;
    int m = code & 0x1;
    double v;
    if (e == 0)
        v = 0.5 * (double)m;                         /* subnormal: m/2 * 2^(1-1) */
    else
        v = ldexp(1.0 + 0.5 * (double)m, e - 1);
    return sign ? -v : v;
}

/* Round a non-negative real v to the nearest finite non-negative E4M3 value,
 * ties to the even code (= even mantissa), values beyond 448 clamp to 448.
 * The target is num/den (callers pass amax and 6, so no division is made).
 * Below the saturation point the 127 candidates are enumerated and their
 * distances |num - den*value| compared; these are exact in double because num
 * is a bf16 and den*value has at most 7 significant bits of similar size. */
uint8_t oracle_e4m3_round_ratio(double num, double den)
{
    uint8_t best = 0;
    double best_d = INFINITY;
    if (num >= den * 448.0)
        return 0x7E;                                 /* saturate; keeps the distances below exact */
    for (int c = 0; c <= 0x7E; ++c) {
        double d = fabs(num - den * oracle_e4m3_value((uint8_t)c));
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = (uint8_t)c;
            best_d = d;
        }
    }
    return best;
}

/* Nearest E2M1 magnitude code (0..7) to |x|/s for s > 0, ties to the even code,
 * magnitudes at or beyond 6 clamp to 6.  Below that, the distances |x| - grid*s
 * are exact in double (bf16 minus a product with at most 6 significant bits). */
uint8_t oracle_e2m1_round_ratio(double ax, double s)
{
    uint8_t best = 0;
    double best_d = INFINITY;
    if (ax >= 6.0 * s)
        return 7;                                    /* saturate; keeps the distances below exact */
    for (int c = 0; c <= 7; ++c) {
        double d = fabs(ax - s * oracle_e2m1_value((uint8_t)c));
        if (d < best_d || (d == best_d && (c & 1) == 0 && (best & 1) == 1)) {
            best = (uint8_t)c;
            best_d = d;
        }
    }
    return best;
}

/* ------------------------------------------------------------------------- */
/* a1: quantise latent rows ([G2C] "FP4 cache entries, and why they're safe") */
/* ------------------------------------------------------------------------- */
/*
 * Each group of 16 consecutive channels gets one E4M3 scale s = RNE(amax / 6)
 * (6 is the largest E2M1 magnitude, so the largest element lands on the top
 * code), saturating at 448; each channel gets the E2M1 code nearest to x / s
 * with its sign kept (so -0 and small negatives give 0x8).  A group whose scale
 * rounds to zero stores all-zero codes.  Codes are packed two per byte, the
 * even channel in the low nibble; scales are stored apart from codes.
 *
 * x      : [n_rows][D] bf16 bits
 * codes  : [n_rows][D/2]
 * scales : [n_rows][D/16]
 */
void oracle_quantize_rows(const uint16_t *x, int64_t n_rows, int D, uint8_t *codes, uint8_t *scales)
{
    for (int64_t r = 0; r < n_rows; ++r) {
        const uint16_t *xr = x + r * D;
        for (int g = 0; g < D / 16; ++g) {
            double amax = 0.0;
            for (int i = 0; i < 16; ++i) {
                double a = fabs(oracle_bf16_value(xr[g * 16 + i]));
                if (a > amax)
                    amax = a;
            }
            uint8_t sbyte = oracle_e4m3_round_ratio(amax, 6.0);
            double s = oracle_e4m3_value(sbyte);
            scales[r * (D / 16) + g] = sbyte;
            for (int i = 0; i < 16; ++i) {
                int ch = g * 16 + i;
                uint16_t bits = xr[ch];
                uint8_t code = 0;
                if (s > 0.0) {
                    double v = oracle_bf16_value(bits);
                    code = oracle_e2m1_round_ratio(fabs(v), s);
                    if (bits & 0x8000)
                        code |= 0x8;
                }
                uint8_t *dst = codes + r * (D / 2) + ch / 2;
                if ((ch & 1) == 0)
                    *dst = (uint8_t)((*dst & 0xF0) | code);
                else
                    *dst = (uint8_t)((*dst & 0x0F) | (code << 4));
            }
        }
    }
}

/* Dequantise rows back to doubles: v = E2M1(code) * E4M3(scale). */
void oracle_dequantize_rows(const uint8_t *codes, const uint8_t *scales, int64_t n_rows, int D, double *out)
{
    for (int64_t r = 0; r < n_rows; ++r)
        for (int ch = 0; ch < D; ++ch) {
            uint8_t byte = codes[r * (D / 2) + ch / 2];
            uint8_t code = (ch & 1) ? (byte >> 4) : (byte & 0xF);
            out[r * D + ch] = oracle_e2m1_value(code) * oracle_e4m3_value(scales[r * (D / 16) + ch / 16]);
        }
}

/* Signed E4M3 of a real x: the magnitude rounded as oracle_e4m3_round_ratio
 * (nearest, ties to the even code, 448 beyond the largest value), the sign of
 * x kept (a zero result of a negative x keeps its sign bit). */
uint8_t oracle_e4m3_round(double x)
{
    uint8_t m = oracle_e4m3_round_ratio(fabs(x), 1.0);
    return (uint8_t)(x < 0.0 ? (m | 0x80) : m);
}

/* ------------------------------------------------------------------------- */
/* Indexer keys projected from the main cache entries ([G2C] "The global     */
/* branch: compress, index, select": the indexer's keys are a projection of  */
/* the main cache entries rather than a separately computed cache)           */
/* ------------------------------------------------------------------------- */
/*
 * For each stored row (FP4 codes + E4M3 scales, dequantised exactly):
 *     ik[j] = E4M3( sum_c v[c] * w[c][j] ),   j < DI
 * with w a [D][DI] matrix of bf16 values.  Every product has at most 8 + 6
 * significant bits and the sum over c is taken in double; it is exact while
 * the products' exponents span at most 30 binades (53 bits less 14
 * significant bits less 9 carry bits for up to 512 terms), which holds for
 * weights and rows of ordinary size (the workloads' w is N(0, 1/D) in bf16).
 *
 * codes  : [n_rows][D/2]      scales : [n_rows][D/16]
 * w      : [D][DI] bf16 bits  ik     : [n_rows][DI] E4M3 bytes (out)
 */
void oracle_project_ikeys(const uint8_t *codes, const uint8_t *scales, int64_t n_rows, int D,
                          const uint16_t *w, int DI, uint8_t *ik)
{
    double *v = (double *)malloc(sizeof(double) * (size_t)D);
    for (int64_t r = 0; r < n_rows; ++r) {
        oracle_dequantize_rows(codes + r * (D / 2), scales + r * (D / 16), 1, D, v);
        for (int j = 0; j < DI; ++j) {
            double acc = 0.0;
            for (int c = 0; c < D; ++c)
                acc += v[c] * oracle_bf16_value(w[(int64_t)c * DI + j]);
            ik[r * DI + j] = oracle_e4m3_round(acc);
        }
    }
    free(v);
}

/* ------------------------------------------------------------------------- */
/* a2/a4: indexer score ([G2C] "The global branch", item 3; [FPR] Full mode)  */
/* ------------------------------------------------------------------------- */
/*
 * For one query (one sequence, one position) and each candidate row t:
 *     score(t) = sum_h w[h] * ReLU( sum_d iq[h][d] * ik[t][d] )
 * Products of two E4M3 values are exact in double, and so is every sum over
 * d (at most 2^35 dynamic range plus 7 carry bits).  The weighted head sum is
 * accumulated in double and rounded once to fp32.
 *
 * iq   : [HI][DI] E4M3 bytes        w : [HI] fp32
 * ik   : key table, row t at ik + rows[j]*DI (E4M3 bytes)
 * rows : candidate row ids, n of them
 * out  : [n] fp32
 */
void oracle_index_score(const uint8_t *iq, const float *w, int HI, int DI,
                        const uint8_t *ik, const int64_t *rows, int64_t n, float *out)
{
    double *q = (double *)malloc(sizeof(double) * (size_t)HI * DI);
    for (int i = 0; i < HI * DI; ++i)
        q[i] = oracle_e4m3_value(iq[i]);
    double *k = (double *)malloc(sizeof(double) * (size_t)DI);
    for (int64_t j = 0; j < n; ++j) {
        const uint8_t *kr = ik + rows[j] * (int64_t)DI;
        for (int d = 0; d < DI; ++d)
            k[d] = oracle_e4m3_value(kr[d]);
        double acc = 0.0;
        for (int h = 0; h < HI; ++h) {
            double dot = 0.0;
            for (int d = 0; d < DI; ++d)
                dot += q[h * DI + d] * k[d];
            double relu = dot > 0.0 ? dot : 0.0;
            acc += (double)w[h] * relu;
        }
        out[j] = (float)acc;
    }
    free(k);
    free(q);
}

/* ------------------------------------------------------------------------- */
/* MXFP4 indexer keys ([G2C] "FP4 cache entries, and why they're safe": the   */
/* indexer K entry of 128 values x 4 bits plus one 8-bit scale per 32 values, */
/* 68 B, the OCP MXFP4 format the report says V4 adopted)                    */
/* ------------------------------------------------------------------------- */
/*
 * Per block of 32 consecutive channels with largest magnitude amax:
 *   X = floor(log2(amax)) - 2     (2 is the exponent of E2M1's largest value, 6)
 *   clamped to [-8, 6], and X = -8 for an all-zero block;
 *   scale byte = X + 127 (UE8M0: the value 2^X);
 *   code = sign(x) | E2M1 magnitude nearest to |x| / 2^X (ties to the even
 *   code, 6 beyond), packed two per byte, the even channel in the low nibble.
 * The clamp is this library's addition to the OCP rule: with X in [-8, 6] every
 * stored value 2^X * E2M1 is exactly an E4M3 value (6 * 2^6 = 384 <= 448, and
 * 0.5 * 2^-8 = 2^-9 is E4M3's smallest step), so a key decodes exactly.
 */
int oracle_mx_exponent(double amax)
{
    if (!(amax > 0.0))
        return -8;
    int e;
    frexp(amax, &e);                 /* amax = f * 2^e, f in [0.5, 1): floor(log2 amax) = e - 1 */
    int X = (e - 1) - 2;
    if (X < -8)
        X = -8;
    if (X > 6)
        X = 6;
    return X;
}

/* Quantise rows of reals x [n][DI] (DI a multiple of 32) to MXFP4:
 * codes [n][DI/2], scales [n][DI/32]. */
void oracle_mx_quantize(const double *x, int64_t n, int DI, uint8_t *codes, uint8_t *scales)
{
    for (int64_t r = 0; r < n; ++r)
        for (int blk = 0; blk < DI / 32; ++blk) {
            const double *xb = x + r * DI + blk * 32;
            double amax = 0.0;
            for (int i = 0; i < 32; ++i)
                if (fabs(xb[i]) > amax)
                    amax = fabs(xb[i]);
            const int X = oracle_mx_exponent(amax);
            const double s = ldexp(1.0, X);
            scales[r * (DI / 32) + blk] = (uint8_t)(X + 127);
            for (int i = 0; i < 32; ++i) {
                uint8_t code = oracle_e2m1_round_ratio(fabs(xb[i]), s);
                if (signbit(xb[i]))
                    code |= 0x8;
                const int ch = blk * 32 + i;
                uint8_t *dst = codes + r * (DI / 2) + ch / 2;
                if ((ch & 1) == 0)
                    *dst = (uint8_t)((*dst & 0xF0) | code);
                else
                    *dst = (uint8_t)((*dst & 0x0F) | (code << 4));
            }
        }
}

/* MXFP4 decode: 2^(scale - 127) * E2M1(code). */
double oracle_mx_value(uint8_t code, uint8_t scale)
{
    return ldexp(oracle_e2m1_value(code), (int)scale - 127);
}

void oracle_mx_dequantize(const uint8_t *codes, const uint8_t *scales, int64_t n, int DI, double *out)
{
    for (int64_t r = 0; r < n; ++r)
        for (int ch = 0; ch < DI; ++ch) {
            uint8_t byte = codes[r * (DI / 2) + ch / 2];
            uint8_t code = (ch & 1) ? (byte >> 4) : (byte & 0xF);
            out[r * DI + ch] = oracle_mx_value(code, scales[r * (DI / 32) + ch / 32]);
        }
}

/* Indexer scores with MXFP4 keys: the score formula of oracle_index_score,
 * with each key decoded from its codes and block scales (products exact in
 * double, as there). */
void oracle_index_score_mx(const uint8_t *iq, const float *w, int HI, int DI, const uint8_t *kcodes,
                           const uint8_t *kscales, const int64_t *rows, int64_t n, float *out)
{
    double *q = (double *)malloc(sizeof(double) * (size_t)HI * DI);
    for (int i = 0; i < HI * DI; ++i)
        q[i] = oracle_e4m3_value(iq[i]);
    double *k = (double *)malloc(sizeof(double) * (size_t)DI);
    for (int64_t j = 0; j < n; ++j) {
        oracle_mx_dequantize(kcodes + rows[j] * (int64_t)(DI / 2), kscales + rows[j] * (int64_t)(DI / 32), 1, DI, k);
        double acc = 0.0;
        for (int h = 0; h < HI; ++h) {
            double dot = 0.0;
            for (int d = 0; d < DI; ++d)
                dot += q[h * DI + d] * k[d];
            double relu = dot > 0.0 ? dot : 0.0;
            acc += (double)w[h] * relu;
        }
        out[j] = (float)acc;
    }
    free(k);
    free(q);
}

/* Projected indexer keys in MXFP4: the exact products of oracle_project_ikeys,
 * quantised per block of 32 key channels by oracle_mx_quantize. */
void oracle_project_ikeys_mx(const uint8_t *codes, const uint8_t *scales, int64_t n_rows, int D, const uint16_t *w,
                             int DI, uint8_t *kcodes, uint8_t *kscales)
{
    double *v = (double *)malloc(sizeof(double) * (size_t)D);
    double *ik = (double *)malloc(sizeof(double) * (size_t)DI);
    for (int64_t r = 0; r < n_rows; ++r) {
        oracle_dequantize_rows(codes + r * (D / 2), scales + r * (D / 16), 1, D, v);
        for (int j = 0; j < DI; ++j) {
            double acc = 0.0;
            for (int c = 0; c < D; ++c)
                acc += v[c] * oracle_bf16_value(w[(int64_t)c * DI + j]);
            ik[j] = acc;
        }
        oracle_mx_quantize(ik, 1, DI, kcodes + r * (DI / 2), kscales + r * (DI / 32));
    }
    free(ik);
    free(v);
}

/* ------------------------------------------------------------------------- */
/* a3: top-K selection ([FPR] "keep the best 512"; [G2C] "The global branch") */
/* ------------------------------------------------------------------------- */

typedef struct {
    float score;
    int64_t index;
} scored;

/* Larger score first; equal scores: lower index first.  -0 and +0 compare equal. */
static int by_score_desc_index_asc(const void *pa, const void *pb)
{
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    if (a->score > b->score)
        return -1;
    if (a->score < b->score)
        return 1;
    return (a->index < b->index) ? -1 : (a->index > b->index);
}

/*
 * Indices (0..n-1) of the K largest scores, ties to the lower index, taken
 * only among entries with valid[i] != 0 (valid == NULL: all).  Writes
 * min(K, #valid) indices in rank order, then -1 up to K.
 */
void oracle_topk(const float *scores, const uint8_t *valid, int64_t n, int64_t K, int64_t *out)
{
    scored *s = (scored *)malloc(sizeof(scored) * (size_t)(n > 0 ? n : 1));
    int64_t m = 0;
    for (int64_t i = 0; i < n; ++i)
        if (valid == NULL || valid[i]) {
            s[m].score = scores[i];
            s[m].index = i;
            ++m;
        }
    qsort(s, (size_t)m, sizeof(scored), by_score_desc_index_asc);
    for (int64_t j = 0; j < K; ++j)
        out[j] = j < m ? s[j].index : -1;
    free(s);
}

/*
 * [G2C] "The hierarchical indexer": positions are grouped into blocks of
 * `block` consecutive rows (block j = rows [j*block, (j+1)*block)), each block
 * is scored by its best member, and the best n_keep blocks are kept.  Rows at
 * or past n are not members (the last block may be partial).
 * blockscore : [ceil(n/block)] out
 */
void oracle_block_max(const float *scores, int64_t n, int block, float *blockscore)
{
    int64_t nb = (n + block - 1) / block;
    for (int64_t j = 0; j < nb; ++j) {
        float best = -INFINITY;
        for (int64_t t = j * block; t < (j + 1) * block && t < n; ++t)
            if (scores[t] > best)
                best = scores[t];
        blockscore[j] = best;
    }
}

/* ------------------------------------------------------------------------- */
/* a5/a6: sparse attention over the selected FP4 rows                        */
/* ([G2C] "The global branch", item 3; [FPR] Full mode: one W_KV so K = V)   */
/* ------------------------------------------------------------------------- */
/*
 * For each head h: z_j = scale * q_h . v_{idx_j} over the selected entries j
 * (idx_j < 0 is padding and is skipped), out_h = sum_j softmax(z)_j v_{idx_j},
 * lse_h = log sum_j exp(z_j).  The cached latent serves as both key and value.
 * Everything is accumulated in double and rounded once.  No valid entry:
 * out_h = 0 and lse_h = -inf.
 *
 * q      : [H][D] bf16 bits
 * codes  : row r at codes + r*(D/2);  scales: row r at scales + r*(D/16)
 * idx    : [K] row ids
 * out    : [H][D] fp32,  lse : [H] fp32 (may be NULL)
 */
void oracle_attend(const uint16_t *q, int H, int D, double scale,
                   const uint8_t *codes, const uint8_t *scales,
                   const int64_t *idx, int64_t K, float *out, float *lse)
{
    int64_t nv = 0;
    for (int64_t j = 0; j < K; ++j)
        if (idx[j] >= 0)
            ++nv;
    double *v = (double *)malloc(sizeof(double) * (size_t)(nv > 0 ? nv : 1) * D);
    int64_t r = 0;
    for (int64_t j = 0; j < K; ++j)
        if (idx[j] >= 0) {
            oracle_dequantize_rows(codes + idx[j] * (int64_t)(D / 2), scales + idx[j] * (int64_t)(D / 16),
                                   1, D, v + r * D);
            ++r;
        }
    double *z = (double *)malloc(sizeof(double) * (size_t)(nv > 0 ? nv : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    for (int h = 0; h < H; ++h) {
        if (nv == 0) {
            for (int d = 0; d < D; ++d)
                out[h * D + d] = 0.0f;
            if (lse)
                lse[h] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < nv; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += oracle_bf16_value(q[h * D + d]) * v[j * D + d];
            z[j] = scale * dot;
            if (z[j] > m)
                m = z[j];
        }
        double l = 0.0;
        for (int d = 0; d < D; ++d)
            acc[d] = 0.0;
        for (int64_t j = 0; j < nv; ++j) {
            double p = exp(z[j] - m);
            l += p;
            for (int d = 0; d < D; ++d)
                acc[d] += p * v[j * D + d];
        }
        for (int d = 0; d < D; ++d)
            out[h * D + d] = (float)(acc[d] / l);
        if (lse)
            lse[h] = (float)(m + log(l));
    }
    free(acc);
    free(z);
    free(v);
}

/* Joint attention of the sparse global branch and the local sliding window.
 * [FPR] "The Paper": the selected entries are glued onto the sliding-window
 * KV and the query attends to both with one softmax; [G2C] "Two attention
 * paths in every layer": the local branch is exact attention over the most
 * recent 128 tokens; "FP4 cache entries, and why they're safe": the local
 * cache stays in FP8.  Window rows are FP8 E4M3 vectors of D channels (no
 * scale), one shared latent per token (K = V, as for the global entries).
 * swa holds the sequence's local rows; rows [lo, hi) are the window.  The
 * softmax runs over the selected dequantised FP4 rows and the window rows
 * together, in double precision. */
void oracle_attend_swa(const uint16_t *q, int H, int D, double scale,
                       const uint8_t *codes, const uint8_t *scales,
                       const int64_t *idx, int64_t K,
                       const uint8_t *swa, int64_t lo, int64_t hi,
                       float *out, float *lse)
{
    int64_t nv = 0;
    for (int64_t j = 0; j < K; ++j)
        if (idx[j] >= 0)
            ++nv;
    const int64_t nw = hi > lo ? hi - lo : 0;
    const int64_t n = nv + nw;
    double *v = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * D);
    int64_t r = 0;
    for (int64_t j = 0; j < K; ++j)
        if (idx[j] >= 0) {
            oracle_dequantize_rows(codes + idx[j] * (int64_t)(D / 2), scales + idx[j] * (int64_t)(D / 16),
                                   1, D, v + r * D);
            ++r;
        }
    for (int64_t t = lo; t < hi; ++t, ++r)
        for (int d = 0; d < D; ++d)
            v[r * D + d] = oracle_e4m3_value(swa[t * (int64_t)D + d]);
    double *z = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    double *acc = (double *)malloc(sizeof(double) * (size_t)D);
    for (int h = 0; h < H; ++h) {
        if (n == 0) {
            for (int d = 0; d < D; ++d)
                out[h * D + d] = 0.0f;
            if (lse)
                lse[h] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t j = 0; j < n; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += oracle_bf16_value(q[h * D + d]) * v[j * D + d];
            z[j] = scale * dot;
            if (z[j] > m)
                m = z[j];
        }
        double l = 0.0;
        for (int d = 0; d < D; ++d)
            acc[d] = 0.0;
        for (int64_t j = 0; j < n; ++j) {
            double p = exp(z[j] - m);
            l += p;
            for (int d = 0; d < D; ++d)
                acc[d] += p * v[j * D + d];
        }
        for (int d = 0; d < D; ++d)
            out[h * D + d] = (float)(acc[d] / l);
        if (lse)
            lse[h] = (float)(m + log(l));
    }
    free(acc);
    free(z);
    free(v);
}

/* ---------------------------------------------------------------------------
 * Persistent cache records.  "G2C Brief - DeepSeek V4.1-Flash", section "FP4
 * cache entries, and why they're safe", the derivation of the 890 bytes per
 * token: a cache entry is its main entry (512 four-bit values and 32 scale
 * bytes, 288 B) and its indexer entry (128 four-bit values and 4 scale bytes
 * in MXFP4, 68 B), 356 B; a layer that keeps a cache with compression m stores
 * one entry per m tokens.  A record keeps the table's order: the main entry's
 * code bytes, its scale bytes, then the indexer entry's bytes (E4M3: DI value
 * bytes; MXFP4: DI/2 code bytes, then DI/32 scale bytes).
 * ------------------------------------------------------------------------- */
int64_t oracle_record_bytes(int D, int DI, int mx)
{
    return (int64_t)(D / 2) + D / 16 + (mx ? DI / 2 + DI / 32 : DI);
}

/* Bytes per token of the caches of n_layers layers, layer i storing one record
 * of record_bytes[i] bytes per m[i] tokens. */
double oracle_bytes_per_token(const int64_t *record_bytes, const int32_t *m, int n_layers)
{
    double t = 0.0;
    for (int i = 0; i < n_layers; ++i)
        t += (double)record_bytes[i] / (double)m[i];
    return t;
}

/* Rows [row0, row0 + n) of each of B sequences as records, out [B][n][record];
 * a row at or past lengths[b] gives a record of zeros.  keys holds each row's
 * indexer entry as the record stores it ([B][cap][key bytes]). */
void oracle_cache_spill(const uint8_t *codes, const uint8_t *scales, const uint8_t *keys, int B, int64_t cap, int D,
                        int DI, int mx, const int64_t *lengths, int64_t row0, int64_t n, uint8_t *out)
{
    const int64_t cb = D / 2, sb = D / 16, kb = oracle_record_bytes(D, DI, mx) - cb - sb;
    const int64_t rb = cb + sb + kb;
    for (int b = 0; b < B; ++b)
        for (int64_t i = 0; i < n; ++i) {
            const int64_t r = row0 + i;
            uint8_t *rec = out + ((int64_t)b * n + i) * rb;
            if (r >= lengths[b]) {
                memset(rec, 0, (size_t)rb);
                continue;
            }
            const int64_t row = (int64_t)b * cap + r;
            memcpy(rec, codes + row * cb, (size_t)cb);
            memcpy(rec + cb, scales + row * sb, (size_t)sb);
            memcpy(rec + cb + sb, keys + row * kb, (size_t)kb);
        }
}

/* Appends n records per sequence (in [B][n][record]) at rows lengths[b] ..
 * lengths[b] + n - 1, then lengths[b] += n; a sequence whose rows would pass
 * cap is left unchanged.  Returns how many sequences were left unchanged. */
int oracle_cache_reload(uint8_t *codes, uint8_t *scales, uint8_t *keys, int B, int64_t cap, int D, int DI, int mx,
                        int64_t *lengths, const uint8_t *in, int64_t n)
{
    const int64_t cb = D / 2, sb = D / 16, kb = oracle_record_bytes(D, DI, mx) - cb - sb;
    const int64_t rb = cb + sb + kb;
    int skipped = 0;
    for (int b = 0; b < B; ++b) {
        if (lengths[b] + n > cap) {
            ++skipped;
            continue;
        }
        for (int64_t i = 0; i < n; ++i) {
            const uint8_t *rec = in + ((int64_t)b * n + i) * rb;
            const int64_t row = (int64_t)b * cap + lengths[b] + i;
            memcpy(codes + row * cb, rec, (size_t)cb);
            memcpy(scales + row * sb, rec + cb, (size_t)sb);
            memcpy(keys + row * kb, rec + cb + sb, (size_t)kb);
        }
        lengths[b] += n;
    }
    return skipped;
}
