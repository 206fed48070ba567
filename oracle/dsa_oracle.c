/*
 * CPU oracle for DeepSeek-V4 indexed sparse attention in a chunked prefill.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow statement of what the
 * hot path computes. Only the tests, the smoke check and the benchmark's CPU
 * baseline leg may load it; the library's own path never does, and this file
 * shares no code, header or table with the CUDA sources.
 *
 * Arithmetic: every sum is accumulated in IEEE double (fp64) in the plain
 * index order and rounded once to the output type. Inputs arrive as raw bf16
 * bit patterns (uint16_t) or fp32.
 *
 * What each function follows (page title, section):
 *  - pooling: "perf(deepseek-v4): skip redundant all-pooled indexer scoring",
 *    Summary and Correctness -- every ratio raw rows compress into one pooled
 *    row; 10 tokens at ratio 4 give two pooled rows and a two-token remainder.
 *    The excerpt names the compressor but prints no formula; the reading taken
 *    is the mean of the ratio consecutive raw rows.
 *  - index scores and the pooled-ratio causal mask: "perf(deepseek_v4): faster
 *    exact DeepSeek-V4 prefill", Summary item 5 (mask folded into the indexer
 *    score epilogue with the same sentinel semantics) and Performance (the
 *    indexer scores every causally visible pooled row). Score reading:
 *    s[t,j] = sum_h w[t,h] * ReLU(q[t,h,:] . k[j,:]); masked entries -inf.
 *  - top-k: the first page, Summary (top-k selection down to index_topk,
 *    skipped when all pooled rows fit, selection = sequential indices).
 *    Order: score descending, index ascending; the kept set is emitted in
 *    ascending index order, padded with -1.
 *  - attention: the second page, Summary item 1 (exact attention over the raw
 *    sliding window plus the pooled rows, B=1, H=64, D=512), with one shared
 *    512-wide row serving as key and value for every head.
 *
 * Parity pins live in the test suite: brute force, closed forms and library
 * special cases (numpy einsum/lexsort, torch CPU scaled_dot_product_attention).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value, ties to even (IEEE 754
 * roundTiesToEven onto a format with 8 significant bits and fp32's exponent
 * range), and return its bit pattern. */
uint16_t dsa_oracle_round_bf16(double x)
{
    if (isnan(x))
        return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (ax == 0.0)
        return sign;
    if (isinf(ax))
        return sign | 0x7F80;
    int e;
    frexp(ax, &e);              /* ax = m * 2^e with 0.5 <= m < 1 */
    int qexp = e - 8;           /* spacing of 8-significant-bit values near ax */
    if (qexp < -133)
        qexp = -133;            /* subnormal spacing of the bf16 format */
    double r = nearbyint(ldexp(ax, -qexp));  /* default mode: nearest, ties to even */
    double y = ldexp(r, qexp);
    if (y >= 0x1p128)
        return sign | 0x7F80;   /* rounds past the largest finite value */
    float f = (float)y;         /* exact: y lies on the bf16 grid */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* Mean pooling: out[g, d] = bf16( (sum_{i<ratio} src[g*ratio + i, d]) / ratio ).
 * src holds groups*ratio consecutive raw rows of width dim. */
void dsa_oracle_pool_rows(const uint16_t *src, int64_t groups, int32_t dim,
                          int32_t ratio, uint16_t *out)
{
    for (int64_t g = 0; g < groups; ++g)
        for (int32_t d = 0; d < dim; ++d) {
            double s = 0.0;
            for (int32_t i = 0; i < ratio; ++i)
                s += bf16_bits_to_double(src[(g * ratio + i) * (int64_t)dim + d]);
            out[g * (int64_t)dim + d] = dsa_oracle_round_bf16(s / (double)ratio);
        }
}

/* Number of pooled rows visible to absolute token position t: pooled row j
 * covers raw tokens j*ratio .. j*ratio+ratio-1 and is visible once its last
 * raw token is at or before t. Capped by the rows that exist. */
static int64_t n_visible(int64_t t, int32_t ratio, int64_t n)
{
    int64_t v = (t + 1) / ratio;
    return v < n ? v : n;
}

/* Indexer scores for R query rows at absolute positions pos[r]:
 *   scores[r, j] = fp32( sum_h w[r,h] * max(0, sum_d q[r,h,d] * k[j,d]) )  for j < n_vis
 *   scores[r, j] = -inf                                                     for n_vis <= j < n
 * mag[r, j] (optional) = sum_h |w[r,h]| * max(0, dot), the size of the terms
 * that were summed, used to state tolerances near cancellation. */
void dsa_oracle_index_scores(const uint16_t *q_idx, const float *w,
                             const int64_t *pos, int64_t R,
                             const uint16_t *pooled_ik, int64_t n,
                             int32_t heads, int32_t dim, int32_t ratio,
                             float *scores, double *mag)
{
    double *kd = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1) * dim);
    for (int64_t i = 0; i < n * dim; ++i)
        kd[i] = bf16_bits_to_double(pooled_ik[i]);

#pragma omp parallel
    {
        /* q of one row, stored [d][h] so the per-head sums below run side by side */
        double *qt = (double *)malloc(sizeof(double) * (size_t)dim * heads);
        double *dot = (double *)malloc(sizeof(double) * (size_t)heads);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < R; ++r) {
            for (int32_t h = 0; h < heads; ++h)
                for (int32_t d = 0; d < dim; ++d)
                    qt[(int64_t)d * heads + h] =
                        bf16_bits_to_double(q_idx[(r * heads + h) * (int64_t)dim + d]);
            int64_t nv = n_visible(pos[r], ratio, n);
            for (int64_t j = 0; j < n; ++j) {
                float *so = &scores[r * n + j];
                if (j >= nv) {
                    *so = -INFINITY;
                    if (mag)
                        mag[r * n + j] = 0.0;
                    continue;
                }
                const double *k = &kd[j * dim];
                for (int32_t h = 0; h < heads; ++h)
                    dot[h] = 0.0;
                /* dot[h] = sum over d in increasing order of q[h,d]*k[d] */
                for (int32_t d = 0; d < dim; ++d) {
                    const double kv = k[d];
                    const double *qd = &qt[(int64_t)d * heads];
                    for (int32_t h = 0; h < heads; ++h)
                        dot[h] += qd[h] * kv;
                }
                double s = 0.0, a = 0.0;
                for (int32_t h = 0; h < heads; ++h) {
                    double rl = dot[h] > 0.0 ? dot[h] : 0.0;
                    double wh = (double)w[r * heads + h];
                    s += wh * rl;
                    a += fabs(wh) * rl;
                }
                *so = (float)s;
                if (mag)
                    mag[r * n + j] = a;
            }
        }
        free(qt);
        free(dot);
    }
    free(kd);
}

typedef struct {
    float s;
    int32_t j;
} cand_t;

/* total order: larger score first; equal scores: lower index first */
static int cand_cmp(const void *pa, const void *pb)
{
    const cand_t *a = (const cand_t *)pa, *b = (const cand_t *)pb;
    if (a->s > b->s)
        return -1;
    if (a->s < b->s)
        return 1;
    return (a->j > b->j) - (a->j < b->j);
}

static int idx_cmp(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/* Per-row top-k over the visible scores. Rows with n_vis <= k keep every
 * visible row (the sequential indices 0..n_vis-1); otherwise the k best under
 * (score desc, index asc). Output: ascending indices, -1 padded, [R, k]. */
void dsa_oracle_topk(const float *scores, const int64_t *pos, int64_t R,
                     int64_t n, int32_t ratio, int32_t k, int32_t *sel)
{
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < R; ++r) {
        int32_t *out = &sel[r * k];
        int64_t nv = n_visible(pos[r], ratio, n);
        if (nv <= k) {
            for (int32_t i = 0; i < k; ++i)
                out[i] = i < nv ? i : -1;
            continue;
        }
        cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)nv);
        for (int64_t j = 0; j < nv; ++j) {
            c[j].s = scores[r * n + j];
            c[j].j = (int32_t)j;
        }
        qsort(c, (size_t)nv, sizeof(cand_t), cand_cmp);
        for (int32_t i = 0; i < k; ++i)
            out[i] = c[i].j;
        qsort(out, (size_t)k, sizeof(int32_t), idx_cmp);
        free(c);
    }
}

/* Exact attention of R query rows (absolute positions pos[r]) over
 *   (i)  raw rows u = max(0, t-window+1) .. t  (raw_kv row u - raw_start), then
 *   (ii) pooled rows sel[r, 0..k-1] that are >= 0,
 * with one shared row serving as key and value for every head:
 *   out[r,h,:] = sum_i softmax_i(scale * q[r,h,:] . kv_i) * kv_i     (fp64)
 * A row with no key at all is impossible (the window always holds t itself).
 * Returns 0, or -1 when a raw row falls outside raw_kv or a pooled index is
 * out of range. */
int dsa_oracle_attention(const uint16_t *q, const int64_t *pos, int64_t R,
                         const uint16_t *raw_kv, int64_t raw_start, int64_t raw_rows,
                         const uint16_t *pooled_kv, int64_t n,
                         const int32_t *sel, int32_t k, int32_t window,
                         int32_t heads, int32_t dim, double scale, double *out)
{
    int bad = 0;
#pragma omp parallel
    {
        int64_t maxkeys = (int64_t)window + k;
        double *keys = (double *)malloc(sizeof(double) * (size_t)maxkeys * dim);
        double *logit = (double *)malloc(sizeof(double) * (size_t)maxkeys);
        double *qh = (double *)malloc(sizeof(double) * (size_t)dim);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < R; ++r) {
            int64_t t = pos[r];
            int64_t u0 = t - window + 1 < 0 ? 0 : t - window + 1;
            int64_t nk = 0;
            int ok = 1;
            for (int64_t u = u0; u <= t; ++u, ++nk) {
                int64_t row = u - raw_start;
                if (row < 0 || row >= raw_rows) {
                    ok = 0;
                    break;
                }
                for (int32_t d = 0; d < dim; ++d)
                    keys[nk * dim + d] = bf16_bits_to_double(raw_kv[row * dim + d]);
            }
            for (int32_t i = 0; ok && i < k; ++i) {
                int32_t j = sel[r * k + i];
                if (j < 0)
                    continue;
                if (j >= n) {
                    ok = 0;
                    break;
                }
                for (int32_t d = 0; d < dim; ++d)
                    keys[nk * dim + d] = bf16_bits_to_double(pooled_kv[(int64_t)j * dim + d]);
                ++nk;
            }
            if (!ok) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            for (int32_t h = 0; h < heads; ++h) {
                for (int32_t d = 0; d < dim; ++d)
                    qh[d] = bf16_bits_to_double(q[(r * heads + h) * (int64_t)dim + d]);
                double m = -INFINITY;
                for (int64_t i = 0; i < nk; ++i) {
                    double s = 0.0;
                    for (int32_t d = 0; d < dim; ++d)
                        s += qh[d] * keys[i * dim + d];
                    logit[i] = scale * s;
                    if (logit[i] > m)
                        m = logit[i];
                }
                double z = 0.0;
                for (int64_t i = 0; i < nk; ++i) {
                    logit[i] = exp(logit[i] - m);
                    z += logit[i];
                }
                double *o = &out[(r * heads + h) * (int64_t)dim];
                for (int32_t d = 0; d < dim; ++d)
                    o[d] = 0.0;
                for (int64_t i = 0; i < nk; ++i) {
                    double p = logit[i] / z;
                    for (int32_t d = 0; d < dim; ++d)
                        o[d] += p * keys[i * dim + d];
                }
            }
        }
        free(keys);
        free(logit);
        free(qh);
    }
    return bad ? -1 : 0;
}

/* Round an fp64 array to bf16 bit patterns, element by element. */
void dsa_oracle_round_bf16_array(const double *x, int64_t count, uint16_t *out)
{
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < count; ++i)
        out[i] = dsa_oracle_round_bf16(x[i]);
}

/* Threads the OpenMP runtime will use for the parallel loops above. */
int dsa_oracle_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
