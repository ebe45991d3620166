/*
 * si_oracle.c -- plain, slow CPU oracle for the indexer -> Top-K -> sparse
 * attention path.  TEST INFRASTRUCTURE ONLY: it is built by build() and used by
 * the tests, the smoke check and the CPU-baseline leg of the benchmark; the
 * product library never links or calls it, and it shares no code, header or
 * table with the CUDA sources.
 *
 * Every value is computed in double precision straight from the definitions
 * on the page "Day0 Inference Support and Performance Optimization for New
 * Architecture LLMs" (Baidu Cloud), section 2.2 "Sparse Attention: Indexer
 * Filtering Top-K Historical Positions" and section 4 ("4.1 Overall Indexer
 * Fusion", "4.2 Index-Based Reading for Sparse Attention"):
 *
 *   1. the indexer scores each query against every earlier position,
 *      score(t,s) = sum_h w[t,h] * ReLU(q_idx[t,h,:] . k_idx[s,:])
 *      (head-weighted aggregation of per-head relevance; ReLU per head);
 *   2. the Top-K positions by score are selected (ties -> lower position);
 *   3. attention reads only the selected K/V rows and returns the
 *      softmax-weighted sum of their values.
 *
 * Keys live in a paged cache, which the fused indexer of section 4.1 scores
 * in place: logical position s of sequence q is physical row
 * block_table[q][s / page] * page + s % page.
 *
 * Storage codes: 0 = float32, 1 = bfloat16 bit patterns, 2 = FP8 e4m3 codes
 * (OCP definition: 1 sign, 4 exponent bits with bias 7, 3 mantissa bits; code
 * S.1111.111 is NaN, there are no infinities), 3 = FP4 e2m1 codes, two per
 * byte with the even element in the low nibble (OCP definition: 1 sign, 2
 * exponent bits with bias 1, 1 mantissa bit; no NaN or infinity), 4 = MXFP8:
 * e4m3 codes in groups of 32 consecutive entries of a row, each group with
 * one E8M0 scale byte (section 5.1; see "MXFP8" below).
 *
 * No blocking, fusion or reordering: loops run in the order of the
 * definitions; a library sort (qsort) orders the candidates.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_BF16 = 1, ORC_E4M3 = 2, ORC_E2M1 = 3, ORC_MXE4M3 = 4 };

typedef struct {
    int32_t n_seq;
    int32_t max_blocks;
    int32_t page;
    int32_t n_q;
    const int32_t *block_table; /* [n_seq, max_blocks] */
    const int32_t *ctx_len;     /* [n_seq] */
    const int32_t *q_seq;       /* [n_q] */
    const int32_t *q_pos;       /* [n_q] */
} orc_batch;

/* ---------------------------------------------------------------- decoding */

double orc_bf16_to_f64(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16; /* bf16 is the top half of an IEEE float32 */
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

double orc_e4m3_to_f64(uint8_t c)
{
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 15;
    int m = c & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);            /* subnormal: 0.m * 2^(1-7) */
    else
        v = ldexp(1.0 + m / 8.0, e - 7);     /* normal: 1.m * 2^(e-7) */
    return sign ? -v : v;
}

double orc_e2m1_to_f64(uint8_t c)
{
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 3;
    int m = c & 1;
    double v;
    if (e == 0)
        v = 0.5 * m;                          /* subnormal: 0.m * 2^(1-1) */
    else
        v = ldexp(1.0 + m / 2.0, e - 1);      /* normal: 1.m * 2^(e-1) */
    return sign ? -v : v;
}

/* element i of a buffer (for e2m1, i counts 4-bit elements; an MXFP8 buffer
 * gives the bare e4m3 code value, without its group scale) */
static double elem(const void *base, int type, int64_t i)
{
    switch (type) {
    case ORC_F32: return (double)((const float *)base)[i];
    case ORC_BF16: return orc_bf16_to_f64(((const uint16_t *)base)[i]);
    case ORC_E2M1: {
        uint8_t byte = ((const uint8_t *)base)[i >> 1];
        return orc_e2m1_to_f64((i & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15));
    }
    default: return orc_e4m3_to_f64(((const uint8_t *)base)[i]);
    }
}

/* ------------------------------------------------------------------- MXFP8 */

/* Section 5.1 of the page quantises the indexer's Q and K to MXFP8 with one
 * scaling factor per group of 32 entries, computed from the data ("dynamic
 * per-group").  MXFP8 is the OCP Microscaling (MX) v1.0 format: a group
 * holds 32 e4m3 codes P_i and one E8M0 scale byte e, X = 2^(e - 127) (e = 255
 * is NaN); entry i is X * P_i.  The page states no conversion rule, so the
 * MX specification's own is taken:
 *   shared exponent E = floor(log2(max_i |V_i|)) - 8 (8 is the exponent of
 *   e4m3's largest normal, 448 = 1.75 * 2^8), clamped to [-127, 127]; an
 *   all-zero group takes E = -127;
 *   P_i = V_i / 2^E rounded to the nearest e4m3 value, ties to the even code,
 *   magnitudes above 448 clamped to 448, the sign kept (a negative value that
 *   rounds to zero gives -0).
 * A group holding a NaN or an infinity gets e = 255 and NaN codes. */

double orc_e8m0_to_f64(uint8_t e)
{
    return e == 255 ? NAN : ldexp(1.0, (int)e - 127);
}

/* Nearest e4m3 code to x: the finite non-negative codes 0..126 are tried one
 * by one; at equal distance the even code (mantissa bit 0 clear) wins; above
 * 448 the largest code is taken; the sign bit is copied. */
uint8_t orc_f64_to_e4m3_sat(double x)
{
    if (isnan(x))
        return 0x7F;
    double a = fabs(x);
    int best = 0;
    double bd = INFINITY;
    for (int c = 0; c <= 126; c++) {
        double d = fabs(a - orc_e4m3_to_f64((uint8_t)c));
        if (d < bd || (d == bd && (c & 1) == 0 && (best & 1) == 1)) {
            bd = d;
            best = c;
        }
    }
    if (a > 448.0)
        best = 126;
    return (uint8_t)(signbit(x) ? (best | 0x80) : best);
}

/* One group of 32 values: writes the 32 codes and returns the scale byte. */
uint8_t orc_mx_group(const double *v, uint8_t *codes)
{
    double amax = 0.0;
    int finite = 1;
    for (int i = 0; i < 32; i++) {
        if (!isfinite(v[i]))
            finite = 0;
        else if (fabs(v[i]) > amax)
            amax = fabs(v[i]);
    }
    if (!finite) {
        for (int i = 0; i < 32; i++)
            codes[i] = 0x7F;
        return 255;
    }
    int E = -127;
    if (amax > 0.0) {
        int ex;
        frexp(amax, &ex);          /* amax = m * 2^ex, m in [0.5, 1): floor(log2) = ex - 1 */
        E = ex - 1 - 8;
        if (E < -127) E = -127;
        if (E > 127) E = 127;
    }
    for (int i = 0; i < 32; i++)
        codes[i] = orc_f64_to_e4m3_sat(ldexp(v[i], -E));
    return (uint8_t)(E + 127);
}

/* Rows of `dim` entries (dim a multiple of 32) of a float32 or bf16 buffer
 * to MXFP8 codes [n_rows, dim] and scale bytes [n_rows, dim / 32]. */
void oracle_mx_quantize(const void *x, int type, int64_t n_rows, int32_t dim, uint8_t *codes,
                        uint8_t *scales)
{
    double v[32];
    for (int64_t r = 0; r < n_rows; r++)
        for (int32_t g = 0; g < dim / 32; g++) {
            for (int i = 0; i < 32; i++)
                v[i] = elem(x, type, r * dim + g * 32 + i);
            scales[r * (dim / 32) + g] = orc_mx_group(v, codes + r * dim + g * 32);
        }
}

/* physical row of logical position s of sequence q */
static int64_t page_row(const orc_batch *b, int32_t q, int64_t s)
{
    int32_t blk = b->block_table[(int64_t)q * b->max_blocks + s / b->page];
    return (int64_t)blk * b->page + s % b->page;
}

/* ------------------------------------------------------------ thread pool */

typedef struct {
    void (*fn)(void *ctx, int64_t i);
    void *ctx;
    int64_t n;
    int tid, nthreads;
} orc_job;

static void *orc_worker(void *p)
{
    orc_job *j = (orc_job *)p;
    for (int64_t i = j->tid; i < j->n; i += j->nthreads)
        j->fn(j->ctx, i);
    return NULL;
}

static void orc_parallel(void (*fn)(void *, int64_t), void *ctx, int64_t n, int nthreads)
{
    if (nthreads < 1)
        nthreads = 1;
    if (nthreads > 256)
        nthreads = 256;
    pthread_t th[256];
    orc_job jobs[256];
    for (int t = 0; t < nthreads; t++) {
        jobs[t].fn = fn; jobs[t].ctx = ctx; jobs[t].n = n;
        jobs[t].tid = t; jobs[t].nthreads = nthreads;
        if (t > 0)
            pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
    }
    orc_worker(&jobs[0]);
    for (int t = 1; t < nthreads; t++)
        pthread_join(th[t], NULL);
}

/* --------------------------------------------------------------- indexer */

typedef struct {
    const orc_batch *b;
    const int32_t *rows; /* which query rows (NULL = 0..n_rows-1) */
    int32_t Hi, Di;
    const void *q_idx; int q_type;      /* [n_q, Hi, Di] */
    const float *q_scale;               /* [n_q, Hi] or NULL: q = code * q_scale */
    const float *w;                     /* [n_q, Hi] */
    const void *k; int k_type;          /* paged [n_blocks, page, k_stride] */
    const float *k_scale;               /* [n_blocks, page] or NULL */
    int64_t k_stride;
    double *scores; int64_t ld;         /* [n_rows, ld] */
} idx_ctx;

/* score(r, s) for the key at physical row `row` of the paged cache */
static double score_one(const idx_ctx *c, int32_t r, int64_t row)
{
    double kscale = c->k_scale ? (double)c->k_scale[row] : 1.0;
    double score = 0.0;
    for (int32_t h = 0; h < c->Hi; h++) {
        double qscale = c->q_scale ? (double)c->q_scale[(int64_t)r * c->Hi + h] : 1.0;
        double dot = 0.0;
        for (int32_t d = 0; d < c->Di; d++) {
            double qv = elem(c->q_idx, c->q_type, ((int64_t)r * c->Hi + h) * c->Di + d) * qscale;
            double kv = elem(c->k, c->k_type, row * c->k_stride + d) * kscale;
            dot += qv * kv;
        }
        double relu = dot > 0.0 ? dot : 0.0;
        score += (double)c->w[(int64_t)r * c->Hi + h] * relu;
    }
    return score + 0.0; /* -0.0 -> +0.0 */
}

static void idx_row(void *p, int64_t i)
{
    const idx_ctx *c = (const idx_ctx *)p;
    const orc_batch *b = c->b;
    int32_t r = c->rows ? c->rows[i] : (int32_t)i;
    int32_t seq = b->q_seq[r];
    int64_t pos = b->q_pos[r];
    double *out = c->scores + i * c->ld;
    for (int64_t s = 0; s < c->ld; s++) {
        if (s > pos) {            /* causal: only positions s <= pos are scored */
            out[s] = -INFINITY;
            continue;
        }
        out[s] = score_one(c, r, page_row(b, seq, s));
    }
}

void oracle_indexer_scores(const orc_batch *b, const int32_t *rows, int32_t n_rows,
                           int32_t Hi, int32_t Di, const void *q_idx, int q_type,
                           const float *q_scale, const float *w, const void *k, int k_type,
                           const float *k_scale, int64_t k_stride, double *scores, int64_t ld,
                           int nthreads)
{
    idx_ctx c = { b, rows, Hi, Di, q_idx, q_type, q_scale, w, k, k_type, k_scale, k_stride,
                  scores, ld };
    orc_parallel(idx_row, &c, n_rows, nthreads);
}

/* ------------------------------------------------------- indexer, MXFP8 */

/* Section 5.1's indexer: Q and K in MXFP8, one E8M0 scale per group of 32
 * entries.  Section 4.3's prolog quantises the query per group before the
 * fused scoring; a query given in float32 or
 * bf16 is converted here by the MX rule above, one (row, head) group at a
 * time.  Each entry is then X * P (scale times code) and the score is the
 * definition of section 2.2 over those values:
 *   score(t,s) = sum_h w[t,h] * ReLU(sum_d q[t,h,d] * k[s,d]). */
typedef struct {
    const orc_batch *b;
    const int32_t *rows;
    int32_t Hi, Di;
    const void *q_idx; int q_type;      /* [n_q, Hi, Di]: f32, bf16 or MX codes */
    const uint8_t *q_mx;                /* [n_q, Hi, Di / 32] scale bytes (MX q) */
    const float *w;                     /* [n_q, Hi] */
    const uint8_t *k;                   /* paged MX codes [n_blocks, page, k_stride] */
    const uint8_t *k_mx;                /* [n_blocks, page, k_stride / 32] scale bytes */
    int64_t k_stride;
    double *scores; int64_t ld;         /* [n_rows, ld] */
} mx_ctx;

/* The query of row r as MXFP8 values, [Hi * Di] doubles. */
static void mx_query(const mx_ctx *c, int32_t r, double *q)
{
    int32_t G = c->Di / 32;
    for (int32_t h = 0; h < c->Hi; h++)
        for (int32_t g = 0; g < G; g++) {
            int64_t off = ((int64_t)r * c->Hi + h) * c->Di + g * 32;
            uint8_t codes[32], sb;
            if (c->q_type == ORC_MXE4M3) {
                memcpy(codes, (const uint8_t *)c->q_idx + off, 32);
                sb = c->q_mx[((int64_t)r * c->Hi + h) * G + g];
            } else {
                double v[32];
                for (int i = 0; i < 32; i++)
                    v[i] = elem(c->q_idx, c->q_type, off + i);
                sb = orc_mx_group(v, codes);
            }
            for (int i = 0; i < 32; i++)
                q[(int64_t)h * c->Di + g * 32 + i] = orc_e4m3_to_f64(codes[i]) * orc_e8m0_to_f64(sb);
        }
}

static double mx_score(const mx_ctx *c, int32_t r, const double *q, int64_t row)
{
    int32_t G = (int32_t)(c->k_stride / 32);
    double score = 0.0;
    for (int32_t h = 0; h < c->Hi; h++) {
        double dot = 0.0;
        for (int32_t d = 0; d < c->Di; d++) {
            double kv = orc_e4m3_to_f64(c->k[row * c->k_stride + d]) *
                        orc_e8m0_to_f64(c->k_mx[row * G + d / 32]);
            dot += q[(int64_t)h * c->Di + d] * kv;
        }
        double relu = dot > 0.0 ? dot : 0.0;
        score += (double)c->w[(int64_t)r * c->Hi + h] * relu;
    }
    return score + 0.0; /* -0.0 -> +0.0 */
}

static void mx_row(void *p, int64_t i)
{
    const mx_ctx *c = (const mx_ctx *)p;
    const orc_batch *b = c->b;
    int32_t r = c->rows ? c->rows[i] : (int32_t)i;
    int32_t seq = b->q_seq[r];
    int64_t pos = b->q_pos[r];
    double *q = (double *)malloc(sizeof(double) * (size_t)c->Hi * (size_t)c->Di);
    mx_query(c, r, q);
    double *out = c->scores + i * c->ld;
    for (int64_t s = 0; s < c->ld; s++)    /* causal: positions s <= pos only */
        out[s] = s > pos ? -INFINITY : mx_score(c, r, q, page_row(b, seq, s));
    free(q);
}

/* Scores of MXFP8 keys (codes `k`, scale bytes `k_mx`) against a query that is
 * MXFP8 (q_type 4, scale bytes q_mx) or float32 / bf16 (converted per group),
 * -inf past each row's position. */
void oracle_indexer_scores_mx(const orc_batch *b, const int32_t *rows, int32_t n_rows, int32_t Hi,
                              int32_t Di, const void *q_idx, int q_type, const uint8_t *q_mx,
                              const float *w, const uint8_t *k, const uint8_t *k_mx,
                              int64_t k_stride, double *scores, int64_t ld, int nthreads)
{
    mx_ctx c = { b, rows, Hi, Di, q_idx, q_type, q_mx, w, k, k_mx, k_stride, scores, ld };
    orc_parallel(mx_row, &c, n_rows, nthreads);
}

/* ------------------------------------------------------------------ top-k */

typedef struct { double score; int64_t pos; } orc_cand;

/* descending score; equal scores -> ascending position */
static int cand_cmp(const void *x, const void *y)
{
    const orc_cand *a = (const orc_cand *)x, *b = (const orc_cand *)y;
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->pos > b->pos) - (a->pos < b->pos);
}

static int i32_cmp(const void *x, const void *y)
{
    int32_t a = *(const int32_t *)x, b = *(const int32_t *)y;
    return (a > b) - (a < b);
}

typedef struct {
    const orc_batch *b;
    const int32_t *rows;
    const double *scores; int64_t ld;
    int32_t K;
    int32_t *idx;         /* [n_rows, K] */
    double *kth;          /* [n_rows, 2]: K-th and (K+1)-th score, or NaN */
} topk_ctx;

static void topk_row(void *p, int64_t i)
{
    const topk_ctx *c = (const topk_ctx *)p;
    int32_t r = c->rows ? c->rows[i] : (int32_t)i;
    int64_t n = (int64_t)c->b->q_pos[r] + 1;   /* candidates: positions 0..pos */
    int32_t *out = c->idx + i * c->K;
    orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(n > 0 ? n : 1));
    for (int64_t s = 0; s < n; s++) {
        cand[s].score = c->scores[i * c->ld + s];
        cand[s].pos = s;
    }
    qsort(cand, (size_t)n, sizeof(orc_cand), cand_cmp);
    int64_t m = n < c->K ? n : c->K;          /* all of them if pos + 1 <= K */
    for (int64_t j = 0; j < m; j++)
        out[j] = (int32_t)cand[j].pos;
    qsort(out, (size_t)m, sizeof(int32_t), i32_cmp);   /* ascending positions */
    for (int64_t j = m; j < c->K; j++)
        out[j] = -1;
    if (c->kth) {
        c->kth[2 * i] = (n >= c->K) ? cand[c->K - 1].score : NAN;
        c->kth[2 * i + 1] = (n > c->K) ? cand[c->K].score : NAN;
    }
    free(cand);
}

void oracle_topk(const orc_batch *b, const int32_t *rows, int32_t n_rows, const double *scores,
                 int64_t ld, int32_t K, int32_t *idx, double *kth, int nthreads)
{
    topk_ctx c = { b, rows, scores, ld, K, idx, kth };
    orc_parallel(topk_row, &c, n_rows, nthreads);
}

/* ------------------------------------------- candidate-restricted selection */

/* The vLLM article on DeepSeek-V4.1 ("Kernels"): the indexer logits are
 * computed only for a fixed set of candidate positions per query instead of
 * the whole context.  Row r's candidates are the entries s of its list with
 * 0 <= s <= pos (other entries, -1 included, are not candidates).  Each is
 * scored with the same definition as above; the Top-K is taken among the
 * candidates only (score descending, equal scores -> lower position), and
 * written as ascending positions, -1 padded when there are fewer than K. */
typedef struct {
    idx_ctx ic;
    const int32_t *cand; int64_t ld_cand; int32_t n_cand;   /* [n_q, ld_cand] */
    int32_t K;
    int32_t *idx;          /* [n_rows, K] */
    double *scores;        /* [n_rows, n_cand]: score of list entry j, -inf if none */
    double *kth;           /* [n_rows, 2] or NULL */
} cand_ctx;

static void cand_row(void *p, int64_t i)
{
    const cand_ctx *c = (const cand_ctx *)p;
    const orc_batch *b = c->ic.b;
    int32_t r = c->ic.rows ? c->ic.rows[i] : (int32_t)i;
    int32_t seq = b->q_seq[r];
    int64_t pos = b->q_pos[r];
    double *sc = c->scores + i * c->n_cand;
    int32_t *out = c->idx + i * c->K;
    orc_cand *cand = (orc_cand *)malloc(sizeof(orc_cand) * (size_t)(c->n_cand > 0 ? c->n_cand : 1));
    int64_t n = 0;
    for (int32_t j = 0; j < c->n_cand; j++) {
        int64_t s = c->cand[(int64_t)r * c->ld_cand + j];
        if (s < 0 || s > pos) {   /* not a candidate of this row */
            sc[j] = -INFINITY;
            continue;
        }
        sc[j] = score_one(&c->ic, r, page_row(b, seq, s));
        cand[n].score = sc[j];
        cand[n].pos = s;
        n++;
    }
    qsort(cand, (size_t)n, sizeof(orc_cand), cand_cmp);
    int64_t m = n < c->K ? n : c->K;
    for (int64_t j = 0; j < m; j++)
        out[j] = (int32_t)cand[j].pos;
    qsort(out, (size_t)m, sizeof(int32_t), i32_cmp);
    for (int64_t j = m; j < c->K; j++)
        out[j] = -1;
    if (c->kth) {
        c->kth[2 * i] = (n >= c->K) ? cand[c->K - 1].score : NAN;
        c->kth[2 * i + 1] = (n > c->K) ? cand[c->K].score : NAN;
    }
    free(cand);
}

void oracle_topk_cand(const orc_batch *b, const int32_t *rows, int32_t n_rows, int32_t Hi,
                      int32_t Di, const void *q_idx, int q_type, const float *q_scale,
                      const float *w, const void *k, int k_type, const float *k_scale,
                      int64_t k_stride, const int32_t *cand, int64_t ld_cand, int32_t n_cand,
                      int32_t K, int32_t *idx, double *scores, double *kth, int nthreads)
{
    cand_ctx c = { { b, rows, Hi, Di, q_idx, q_type, q_scale, w, k, k_type, k_scale, k_stride,
                     NULL, 0 },
                   cand, ld_cand, n_cand, K, idx, scores, kth };
    orc_parallel(cand_row, &c, n_rows, nthreads);
}

/* --------------------------------------------------------- sparse attention */

typedef struct {
    const orc_batch *b;
    const int32_t *rows;
    int32_t Hq, Dqk, Dv;
    const void *q; int q_type;          /* [n_q, Hq, Dqk] */
    const void *k; const void *v; int kv_type;
    int64_t k_stride, v_stride;         /* V row = first Dv entries of its row */
    const float *k_scale, *v_scale;     /* dequantisation scales or NULL (= 1) */
    int32_t scale_tile;                 /* 0: one scale per row; else entries per scale */
    int32_t k_nscale, v_nscale;         /* scales per row */
    const int32_t *idx; int32_t K;      /* [n_rows, K], -1 = unused */
    double scale;
    double *out;                        /* [n_rows, Hq, Dv] */
    double *lse;                        /* [n_rows, Hq] or NULL */
} attn_ctx;

/* Entry d of physical row `row` of a cache, dequantised: code * scale, the
 * scale per row or per tile of scale_tile entries (section 5.2 "KV Cache: FP8
 * with Token-Head-Tile Granularity"). */
static double kv_entry(const void *data, int type, int64_t stride, const float *scale,
                       int32_t tile, int32_t nscale, int64_t row, int32_t d)
{
    double x = elem(data, type, row * stride + d);
    if (scale)
        x *= (double)scale[row * nscale + (tile > 0 ? d / tile : 0)];
    return x;
}

static void attn_row(void *p, int64_t i)
{
    const attn_ctx *c = (const attn_ctx *)p;
    const orc_batch *b = c->b;
    int32_t r = c->rows ? c->rows[i] : (int32_t)i;
    int32_t seq = b->q_seq[r];
    const int32_t *sel = c->idx + i * c->K;
    double *z = (double *)malloc(sizeof(double) * (size_t)c->K);
    int64_t *prow = (int64_t *)malloc(sizeof(int64_t) * (size_t)c->K);
    int32_t n = 0;
    for (int32_t j = 0; j < c->K; j++)
        if (sel[j] >= 0)
            prow[n++] = page_row(b, seq, sel[j]);
    for (int32_t h = 0; h < c->Hq; h++) {
        double *o = c->out + ((int64_t)i * c->Hq + h) * c->Dv;
        int64_t qoff = ((int64_t)r * c->Hq + h) * c->Dqk;
        double zmax = -INFINITY;
        for (int32_t j = 0; j < n; j++) {       /* logits over the selected rows */
            double dot = 0.0;
            for (int32_t d = 0; d < c->Dqk; d++)
                dot += elem(c->q, c->q_type, qoff + d) *
                       kv_entry(c->k, c->kv_type, c->k_stride, c->k_scale, c->scale_tile,
                                c->k_nscale, prow[j], d);
            z[j] = c->scale * dot;
            if (z[j] > zmax) zmax = z[j];
        }
        double l = 0.0;
        for (int32_t j = 0; j < n; j++) {       /* softmax weights */
            z[j] = exp(z[j] - zmax);
            l += z[j];
        }
        for (int32_t d = 0; d < c->Dv; d++) {   /* weighted sum of values */
            double acc = 0.0;
            for (int32_t j = 0; j < n; j++)
                acc += z[j] * kv_entry(c->v, c->kv_type, c->v_stride, c->v_scale, c->scale_tile,
                                       c->v_nscale, prow[j], d);
            o[d] = n > 0 ? acc / l : 0.0;
        }
        if (c->lse)
            c->lse[(int64_t)i * c->Hq + h] = n > 0 ? zmax + log(l) : -INFINITY;
    }
    free(z);
    free(prow);
}

void oracle_sparse_attn(const orc_batch *b, const int32_t *rows, int32_t n_rows, int32_t Hq,
                        int32_t Dqk, int32_t Dv, const void *q, int q_type, const void *k,
                        const void *v, int kv_type, int64_t k_stride, int64_t v_stride,
                        const float *k_scale, const float *v_scale, int32_t scale_tile,
                        int32_t k_nscale, int32_t v_nscale, const int32_t *idx, int32_t K,
                        double scale, double *out, double *lse, int nthreads)
{
    attn_ctx c = { b, rows, Hq, Dqk, Dv, q, q_type, k, v, kv_type, k_stride, v_stride,
                   k_scale, v_scale, scale_tile, k_nscale, v_nscale, idx, K, scale, out, lse };
    orc_parallel(attn_row, &c, n_rows, nthreads);
}
