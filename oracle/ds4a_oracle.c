/*
 * ds4a oracle: a plain, slow, fp64 CPU statement of the three-tier
 * compressed-attention step of the DeepSeek V4 Flash engine (DwarfStar, ds4).
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the checker, not the product: only
 * the test suite, the smoke check and the benchmark's CPU-baseline leg may load
 * it.  It shares no code, header, table or helper with the CUDA library, and
 * the CUDA library never calls it.
 *
 * Sources (the pages this restates):
 *   [ARCH]  "Redis 作者が DeepSeek V4 専用の推論エンジンを C で書いた ―
 *            DwarfStar(ds4.c) のアーキテクチャを読む【第1回/全8回】" (Qiita):
 *            §2 (DS4_SHAPE_FLASH: 64 heads, 1 KV head, head dim 512, n_swa 128,
 *            indexer 64 heads x 128 dims, top_k 512), §3 (three tiers: raw
 *            window + compressed rows + indexer), §3-1 (raw window rounded
 *            through f16), §3-2 (compressor pooling), §3-3 (indexer picks the
 *            top-k compressed rows for the main attention).
 *   [NOTES] "antirez/ds4 深度阅读笔记", section 固定模型形状 (fixed shapes).
 *
 * The pages print no indexer scoring formula.  This library specifies it as
 *     s_r = sum_h w_h * max(0, sum_d iq[h,d] * ik[r,d])
 * and the attention as one joint softmax over (selected compressed rows) U
 * (raw-window rows), each cached row serving as both key and value (one KV
 * head, [ARCH] §2 n_head_kv = 1).
 *
 * Everything is computed in double precision, summed sequentially in the
 * order the definition states (d inner, then h; rows in list order).  Inputs
 * are decoded exactly from their storage formats (bf16, fp16, fp32).
 *
 * Every function here is pinned by tests that do not re-type its formula
 * (hand-worked cases, closed forms, invariants, library special cases).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

int oracle_abi_version(void) { return 1; }

/* ------------------------------------------------------------------------ */
/* Storage-format decoding (IEEE 754 binary16; bfloat16 = the top half of   */
/* an IEEE binary32).  Written from the format definitions.                 */
/* ------------------------------------------------------------------------ */

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int m = h & 0x7F;
    double v;
    if (e == 0xFF)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, 1 - 127 - 7);          /* subnormal */
    else
        v = ldexp((double)(m | 0x80), e - 127 - 7); /* normal: 1.m * 2^(e-127) */
    return sign ? -v : v;
}

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0x1F)
        v = m ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)m, 1 - 15 - 10);
    else
        v = ldexp((double)(m | 0x400), e - 15 - 10);
    return sign ? -v : v;
}

/* Round a double to the nearest binary16 value (ties to even), returned as
 * its bit pattern.  Overflow goes to infinity.  Used by the raw-window push,
 * which stores every row "rounded to f16" ([ARCH] §3-1). */
uint16_t oracle_double_to_f16(double x)
{
    uint16_t sign = 0;
    if (isnan(x))
        return 0x7E00;
    if (signbit(x)) {
        sign = 0x8000;
        x = -x;
    }
    if (isinf(x))
        return sign | 0x7C00;
    /* Spacing of binary16 values around x: 2^(E-10) for normal exponent E,
     * 2^-24 for subnormals.  Round x to a multiple of that spacing. */
    int E;
    if (x == 0.0)
        return sign;
    frexp(x, &E);      /* x = f * 2^E with f in [0.5, 1) -> unbiased exp E-1 */
    int ue = E - 1;
    if (ue < -14)
        ue = -14;      /* subnormal range shares the spacing of 2^-14 */
    double ulp = ldexp(1.0, ue - 10);
    double q = x / ulp;               /* exact: scaling by a power of two */
    double fl = floor(q);
    double rem = q - fl;
    double n;
    if (rem > 0.5)
        n = fl + 1.0;
    else if (rem < 0.5)
        n = fl;
    else
        n = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double r = n * ulp;
    if (r > 65504.0)
        return sign | 0x7C00;         /* beyond the largest finite half */
    /* Encode r. */
    if (r < ldexp(1.0, -14)) {
        int mant = (int)(r / ldexp(1.0, -24));
        return sign | (uint16_t)mant;
    }
    int e2;
    double f = frexp(r, &e2);         /* r = f * 2^e2, f in [0.5,1) */
    int be = e2 - 1 + 15;
    int mant = (int)((f * 2.0 - 1.0) * 1024.0);
    return sign | (uint16_t)(be << 10) | (uint16_t)mant;
}

/* ------------------------------------------------------------------------ */
/* A1. Indexer score                                                        */
/* ------------------------------------------------------------------------ */

/*
 * Scores every compressed row of one unit (one sequence x layer) for n_q
 * queries.  [ARCH] §3-3: the indexer has its own light query system (64
 * heads x 128 dims, [ARCH] §2) and one 128-d key per compressed row; its
 * score ranks the rows.  Formula (this library's specification):
 *     s[q,r] = sum_h w[q,h] * max(0, sum_d iq[q,h,d] * ik[r,d])
 *
 * Visibility: row r exists iff r < n_rows.  With positions given (a prefill
 * chunk), query q also needs row_pos[r] <= q_pos[q] (it may not look at rows
 * finalised after its own position).  Rows that are not visible get -inf.
 *
 * iq:  bf16 [n_q][n_head][dim]       w: fp32 [n_q][n_head]
 * ik:  bf16 [n_cap][dim]             scores: double [n_q][n_cap]
 */
void oracle_indexer_score(const uint16_t *iq, const float *w, const uint16_t *ik,
                          int64_t n_rows, int64_t n_cap, int n_q, int n_head, int dim,
                          const int32_t *q_pos, const int32_t *row_pos, double *scores)
{
    double *qd = (double *)malloc(sizeof(double) * (size_t)n_head * (size_t)dim);
    double *kd = (double *)malloc(sizeof(double) * (size_t)dim);
    for (int q = 0; q < n_q; q++) {
        for (int64_t i = 0; i < (int64_t)n_head * dim; i++)
            qd[i] = oracle_bf16_to_double(iq[(int64_t)q * n_head * dim + i]);
        for (int64_t r = 0; r < n_cap; r++) {
            int visible = r < n_rows;
            if (visible && q_pos != NULL && row_pos != NULL)
                visible = row_pos[r] <= q_pos[q];
            if (!visible) {
                scores[(int64_t)q * n_cap + r] = -INFINITY;
                continue;
            }
            for (int d = 0; d < dim; d++)
                kd[d] = oracle_bf16_to_double(ik[r * dim + d]);
            double s = 0.0;
            for (int h = 0; h < n_head; h++) {
                double dot = 0.0;
                for (int d = 0; d < dim; d++)
                    dot += qd[(int64_t)h * dim + d] * kd[d];
                double relu = dot > 0.0 ? dot : 0.0;
                s += (double)w[(int64_t)q * n_head + h] * relu;
            }
            scores[(int64_t)q * n_cap + r] = s;
        }
    }
    free(qd);
    free(kd);
}

/* ------------------------------------------------------------------------ */
/* A2. Top-k selection                                                      */
/* ------------------------------------------------------------------------ */

typedef struct {
    double s;
    int32_t r;
} oracle_scored_row;

/* Highest score first; equal scores: lower row index first. */
static int by_score_desc_then_row(const void *a, const void *b)
{
    const oracle_scored_row *x = (const oracle_scored_row *)a;
    const oracle_scored_row *y = (const oracle_scored_row *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->r > y->r) - (x->r < y->r);
}

static int int32_ascending(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * [ARCH] §3-3: the indexer passes only the n_indexer_top_k (512 on Flash,
 * 1024 on Pro) highest-scoring compressed rows to the main attention.
 * Visible rows are those with a score that is not -inf and not NaN.
 * Result: m = min(top_k, n_visible) row indices in ascending order in idx,
 * the m-th highest score in *kth (-inf when m == 0).  Returns m.
 */
int oracle_topk_select(const double *scores, int64_t n, int top_k, int32_t *idx, double *kth)
{
    oracle_scored_row *v = (oracle_scored_row *)malloc(sizeof(oracle_scored_row) * (size_t)(n > 0 ? n : 1));
    int64_t nv = 0;
    for (int64_t r = 0; r < n; r++) {
        double s = scores[r];
        if (isnan(s) || s == -INFINITY)
            continue;
        v[nv].s = s;
        v[nv].r = (int32_t)r;
        nv++;
    }
    qsort(v, (size_t)nv, sizeof(oracle_scored_row), by_score_desc_then_row);
    int m = (int)(nv < top_k ? nv : top_k);
    for (int i = 0; i < m; i++)
        idx[i] = v[i].r;
    qsort(idx, (size_t)m, sizeof(int32_t), int32_ascending);
    if (kth)
        *kth = m > 0 ? v[m - 1].s : -INFINITY;
    free(v);
    return m;
}

/* ------------------------------------------------------------------------ */
/* A4. Sparse attention over selected compressed rows U raw-window rows      */
/* ------------------------------------------------------------------------ */

/*
 * One query (n_head heads of width dim) attends over one joint row set:
 *   - n_sel compressed rows comp[sel[j]] (bf16), then
 *   - n_raw raw-window rows raw[raw_sel[j]] (fp16: the raw tier is kept
 *     "rounded to f16", [ARCH] §3-1).
 * Each row is used as both key and value (one KV head, [ARCH] §2).  For each
 * head h:
 *     l_j = scale * sum_d q[h,d] * x_j[d]
 *     a_j = exp(l_j - max l) / sum_i exp(l_i - max l)
 *     out[h,:] = sum_j a_j * x_j[:]
 *     lse[h] = max l + log(sum_j exp(l_j - max l))
 * An empty row set gives out = 0 and lse = -inf.
 * q: bf16 [n_head][dim]; out: double [n_head][dim]; lse: double [n_head] or NULL.
 * Returns 0, or -1 when a row index is negative.
 */
/* The definition above on rows already decoded to double: x [n][dim] holds
 * the selected compressed rows followed by the raw rows.  Frees nothing. */
static void attention_on_rows(const uint16_t *q, int n_head, int dim, const double *x, int n, double scale,
                              double *out, double *lse)
{
    if (n == 0) {
        for (int64_t i = 0; i < (int64_t)n_head * dim; i++)
            out[i] = 0.0;
        if (lse)
            for (int h = 0; h < n_head; h++)
                lse[h] = -INFINITY;
        return;
    }
    double *qd = (double *)malloc(sizeof(double) * (size_t)dim);
    double *l = (double *)malloc(sizeof(double) * (size_t)n);
    double *a = (double *)malloc(sizeof(double) * (size_t)n);
    for (int h = 0; h < n_head; h++) {
        for (int d = 0; d < dim; d++)
            qd[d] = oracle_bf16_to_double(q[(int64_t)h * dim + d]);
        double mx = -INFINITY;
        for (int j = 0; j < n; j++) {
            double dot = 0.0;
            for (int d = 0; d < dim; d++)
                dot += qd[d] * x[(int64_t)j * dim + d];
            l[j] = scale * dot;
            if (l[j] > mx) mx = l[j];
        }
        double z = 0.0;
        for (int j = 0; j < n; j++)
            z += exp(l[j] - mx);
        for (int j = 0; j < n; j++)
            a[j] = exp(l[j] - mx) / z;
        for (int d = 0; d < dim; d++) {
            double acc = 0.0;
            for (int j = 0; j < n; j++)
                acc += a[j] * x[(int64_t)j * dim + d];
            out[(int64_t)h * dim + d] = acc;
        }
        if (lse)
            lse[h] = mx + log(z);
    }
    free(qd);
    free(l);
    free(a);
}

/* Decodes the raw rows raw_sel[0..n_raw) (fp16) into x after n_sel rows. */
static void decode_raw_rows(const uint16_t *raw, const int32_t *raw_sel, int n_raw, int n_sel, int dim, double *x)
{
    for (int j = 0; j < n_raw; j++)
        for (int d = 0; d < dim; d++)
            x[(int64_t)(n_sel + j) * dim + d] = oracle_f16_to_double(raw[(int64_t)raw_sel[j] * dim + d]);
}

int oracle_sparse_attention(const uint16_t *q, int n_head, int dim,
                            const uint16_t *comp, const int32_t *sel, int n_sel,
                            const uint16_t *raw, const int32_t *raw_sel, int n_raw,
                            double scale, double *out, double *lse)
{
    int n = n_sel + n_raw;
    for (int j = 0; j < n_sel; j++)
        if (sel[j] < 0) return -1;
    for (int j = 0; j < n_raw; j++)
        if (raw_sel[j] < 0) return -1;
    double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)dim);
    for (int j = 0; j < n_sel; j++)
        for (int d = 0; d < dim; d++)
            x[(int64_t)j * dim + d] = oracle_bf16_to_double(comp[(int64_t)sel[j] * dim + d]);
    decode_raw_rows(raw, raw_sel, n_raw, n_sel, dim, x);
    attention_on_rows(q, n_head, dim, x, n, scale, out, lse);
    free(x);
    return 0;
}

/*
 * Compressor pooling ([ARCH] §3-2, the pooling inside the compressor's
 * decode step): `ratio` frontier rows of (kv, score) become one compressed
 * row.  Each column j is pooled on its own: the scores of that column over
 * the frontier rows are logits of a softmax whose weights average the kv
 * values of the column,
 *     m_j = max_r score[r][j]
 *     out[j] = sum_r exp(score[r][j] - m_j) * kv[r][j] / sum_r exp(score[r][j] - m_j)
 * and a column whose weights sum to zero (every score -inf) gives 0, as the
 * pages' guard on the denominator does.  kv and score: fp32 [ratio][width],
 * out: [width].
 */
void oracle_compressor_pool(const float *kv, const float *score, int ratio, int width, double *out)
{
    for (int j = 0; j < width; j++) {
        double m = -INFINITY;
        for (int r = 0; r < ratio; r++) {
            const double s = (double)score[(int64_t)r * width + j];
            if (s > m) m = s;
        }
        double num = 0.0, den = 0.0;
        if (m > -INFINITY) {
            for (int r = 0; r < ratio; r++) {
                const double e = exp((double)score[(int64_t)r * width + j] - m);
                den += e;
                num += e * (double)kv[(int64_t)r * width + j];
            }
        }
        out[j] = den > 0.0 ? num / den : 0.0;
    }
}

/*
 * Raw-window push ([ARCH] §3-1): the raw tier keeps the last `cap` (128)
 * tokens' rows, each rounded through f16.  The window is kept oldest first:
 * while it holds fewer than cap rows the new row is appended; a full window
 * first drops its oldest row (the others move down one slot).  ring: f16 bits
 * [cap][dim]; *n_raw: rows held (updated); kv: the new fp32 row.
 */
void oracle_push_raw(uint16_t *ring, int *n_raw, int cap, int dim, const float *kv)
{
    if (*n_raw >= cap) {
        for (int s = 1; s < cap; s++)
            for (int d = 0; d < dim; d++) ring[(int64_t)(s - 1) * dim + d] = ring[(int64_t)s * dim + d];
        *n_raw = cap - 1;
    }
    for (int d = 0; d < dim; d++) ring[(int64_t)(*n_raw) * dim + d] = oracle_double_to_f16((double)kv[d]);
    *n_raw += 1;
}

/* ------------------------------------------------------------------------ */
/* FP8 row store.  [ARCH] §3-2: a new compressed row is RMS-normalised, its */
/* tail rotated, and then put through an FP8 quantisation round trip before */
/* it is stored.  The pages name neither the FP8 format nor its scaling.    */
/* This library reads the round trip as: E4M3 codes with one power-of-two   */
/* scale per row, so that storing the codes and the scale keeps exactly the */
/* values the round trip produces.                                          */
/* ------------------------------------------------------------------------ */

/* E4M3 ("FN" variant of the 8-bit floating-point formats): 1 sign bit, 4
 * exponent bits (bias 7), 3 fraction bits.  Exponent field 15 with fraction 7
 * is NaN; there are no infinities.  Normal values 2^(e-7) * (1 + m/8), largest
 * 448; subnormals (exponent field 0) m * 2^-9. */
double oracle_e4m3_to_double(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xF;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp((double)(8 + m), e - 7 - 3);
    return sign ? -v : v;
}

/* The E4M3 value nearest to x (ties to the even code), saturating: |x| >= 448
 * (infinities included) gives +-448.  NaN gives the NaN code 0x7F. */
uint8_t oracle_double_to_e4m3(double x)
{
    if (isnan(x))
        return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    x = fabs(x);
    if (x >= 448.0)
        return sign | 0x7E;
    if (x == 0.0)
        return sign;
    /* Grid spacing at x: 2^(E-3) in the binade [2^E, 2^(E+1)), E >= -6; the
     * subnormal range below 2^-6 shares the spacing 2^-9. */
    int E;
    frexp(x, &E);
    int ue = E - 1;
    if (ue < -6)
        ue = -6;
    double ulp = ldexp(1.0, ue - 3);
    double q = x / ulp;
    double fl = floor(q);
    double rem = q - fl;
    double n;
    if (rem > 0.5)
        n = fl + 1.0;
    else if (rem < 0.5)
        n = fl;
    else
        n = fmod(fl, 2.0) == 0.0 ? fl : fl + 1.0;   /* tie: the even multiple */
    double r = n * ulp;                 /* <= 448: x < 448 and 448 is on the grid */
    if (r == 0.0)
        return sign;
    if (r < ldexp(1.0, -6))
        return sign | (uint8_t)(r / ldexp(1.0, -9));
    int e2;
    double f = frexp(r, &e2);           /* r = f * 2^e2, f in [0.5, 1) */
    int be = e2 - 1 + 7;
    int mant = (int)((f * 2.0 - 1.0) * 8.0);
    return sign | (uint8_t)(be << 3) | (uint8_t)mant;
}

/* The row's scale exponent: the smallest integer e with amax <= 448 * 2^e,
 * kept within [-126, 127] (the scale 2^e is then a normal fp32).  amax 0, or
 * not finite, gives 0. */
int oracle_fp8_row_exponent(double amax)
{
    if (!(amax > 0.0) || isinf(amax))
        return 0;
    int e = 0;
    while (amax > 448.0 * ldexp(1.0, e) && e < 127)
        e++;
    while (e > -126 && amax <= 448.0 * ldexp(1.0, e - 1))
        e--;
    return e;
}

/* The FP8 round trip's stored form for n_rows rows of dim fp32 values: per
 * row, amax = max |x| over its elements (NaN elements do not count), scale =
 * 2^oracle_fp8_row_exponent(amax), code[d] = nearest E4M3 of x[d] / scale.
 * The stored value of element d is e4m3(code[d]) * scale. */
void oracle_quantize_rows_fp8(const float *x, int64_t n_rows, int dim, uint8_t *codes, float *row_scale)
{
    for (int64_t r = 0; r < n_rows; r++) {
        const float *xr = x + r * dim;
        double amax = 0.0;
        for (int d = 0; d < dim; d++) {
            double v = fabs((double)xr[d]);
            if (v > amax)
                amax = v;              /* NaN compares false: skipped */
        }
        double s = ldexp(1.0, oracle_fp8_row_exponent(amax));
        row_scale[r] = (float)s;
        for (int d = 0; d < dim; d++)
            codes[r * dim + d] = oracle_double_to_e4m3((double)xr[d] / s);
    }
}

/* oracle_sparse_attention with the compressed rows in the FP8 store: row i
 * holds codes[i][0..dim) and row_scale[i]; element d of row i is
 * e4m3(codes[i][d]) * row_scale[i].  Raw rows stay fp16. */
int oracle_sparse_attention_fp8(const uint16_t *q, int n_head, int dim,
                                const uint8_t *codes, const float *row_scale, const int32_t *sel, int n_sel,
                                const uint16_t *raw, const int32_t *raw_sel, int n_raw,
                                double scale, double *out, double *lse)
{
    int n = n_sel + n_raw;
    for (int j = 0; j < n_sel; j++)
        if (sel[j] < 0) return -1;
    for (int j = 0; j < n_raw; j++)
        if (raw_sel[j] < 0) return -1;
    double *x = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * (size_t)dim);
    for (int j = 0; j < n_sel; j++) {
        const double s = (double)row_scale[sel[j]];
        for (int d = 0; d < dim; d++)
            x[(int64_t)j * dim + d] = oracle_e4m3_to_double(codes[(int64_t)sel[j] * dim + d]) * s;
    }
    decode_raw_rows(raw, raw_sel, n_raw, n_sel, dim, x);
    attention_on_rows(q, n_head, dim, x, n, scale, out, lse);
    free(x);
    return 0;
}
