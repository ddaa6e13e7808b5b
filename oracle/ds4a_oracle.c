/*
 * ds4a_oracle.c -- plain, slow, fp64 CPU oracle of the compressed sparse MQA
 * attention path of DeepSeek-V4-Flash as the DS4 engine pages describe it.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load or call this code.  It shares no code,
 * header, table or helper with the CUDA path, and it never reads anything the
 * CUDA path produced.
 *
 * Sources (page title, section):
 *   [KVC]  "DS4 (DwarfStar 4)", Key Techniques, "KV attention compression":
 *          layers 0-1 raw sliding window only; even layers from 2 compress at
 *          ratio 4 with a learned indexer keeping the top 512 compressed rows;
 *          odd layers compress at ratio 128 with no indexer; the compressor
 *          keeps a rolling score/KV state and appends a pooled row at every
 *          ratio boundary.
 *   [ARCH] "DS4 (DwarfStar 4)", Architecture, fixed model shape: 64 attention
 *          heads, multi-query (1 KV head), 128-token sliding window.
 *   [TIER] "DS4 (DwarfStar 4)", Key Techniques, "KV cache with disk as
 *          first-class citizen": raw sliding-window tier (128 tokens per
 *          layer), compressed rows pooled at ratio boundaries.
 * Readings where the pages are silent (each is listed in the design notes):
 *   R1 pooled row = softmax over the block of s_t = w . k_t, weights applied
 *      to both k_t and v_t (same weights);
 *   R3 one caller-supplied indexer key per compressed row;
 *   R4 indexer score = plain dot product q_idx . kidx_j, no scale or bias;
 *   R5 row j is visible to the query at position p iff (j+1)*r <= p+1;
 *   R7 append-then-attend (a block completed by the current token is visible);
 *   R9 window = positions max(0, p-W+1) .. p, current token included;
 *   R10 ranking by score (highest first) then by lower index;
 *   R11 k > visible rows selects every visible row;
 *   R12 no sink, softcap or bias in the softmax.
 * Precision: every step in double.  The one place where floating point decides
 * an integer -- which rows the indexer keeps -- ranks the scores after rounding
 * them to binary32, the precision the CUDA kernels decide in.
 *
 * Pins (tests/test_oracle_pins.py): ratio-1 pooling is the identity, w = 0
 * gives the block mean, score shifts cancel, a two-token block has the closed
 * form sigma(s1-s0), pooling equals a library softmax-weighted sum, top-k
 * equals brute force over all subsets and a library lexicographic sort,
 * attention equals a library scaled-dot-product attention, identical keys give
 * the mean of V, any split of the key set merges back by log-sum-exp, union
 * order does not matter, row counts are floor(prefix/r), prefill of one token
 * equals the decode step, and prefill is causal.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>

/* ---- [KVC] layer schedule ------------------------------------------------ */

/* compression ratio of a layer: 0 = raw window only */
int orc_layer_ratio(int layer)
{
    if (layer < 2) return 0;
    return (layer % 2 == 0) ? 4 : 128;
}

/* indexer top-k of a layer: 0 = no indexer (all visible rows attended) */
int orc_layer_topk(int layer)
{
    return (layer >= 2 && layer % 2 == 0) ? 512 : 0;
}

/* R5: number of compressed rows visible to the query at position p */
long orc_rows_visible(long p, int r)
{
    if (r <= 0) return 0;
    return (p + 1) / r;
}

/* ---- [KVC] + R1: the compressor ------------------------------------------ */

/* Pool one block of n tokens: s_t = w . k_t, alpha = softmax(s),
 * out_k = sum_t alpha_t k_t, out_v = sum_t alpha_t v_t. */
void orc_pool_block(const double *k, const double *v, int n, int D,
                    const double *w, double *out_k, double *out_v)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double smax = -INFINITY;
    for (int t = 0; t < n; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += w[d] * k[(size_t)t * D + d];
        s[t] = acc;
        if (acc > smax) smax = acc;
    }
    double z = 0.0;
    for (int t = 0; t < n; ++t) z += exp(s[t] - smax);
    for (int d = 0; d < D; ++d) { out_k[d] = 0.0; out_v[d] = 0.0; }
    for (int t = 0; t < n; ++t) {
        double a = exp(s[t] - smax) / z;
        for (int d = 0; d < D; ++d) {
            out_k[d] += a * k[(size_t)t * D + d];
            out_v[d] += a * v[(size_t)t * D + d];
        }
    }
    free(s);
}

/* Pool blocks b0 .. b1-1 of ratio r.  raw_k/raw_v hold the tokens at positions
 * raw_pos0 .. raw_pos0+n_raw-1.  Block b covers positions b*r .. b*r+r-1.
 * Writes row b-b0 of out_k/out_v.  Returns the number of rows, or -1 if a
 * block reaches outside the raw rows given. */
long orc_compress_range(const double *raw_k, const double *raw_v, long raw_pos0, long n_raw,
                        int D, const double *w, int r, long b0, long b1,
                        double *out_k, double *out_v)
{
    if (r <= 0 || b1 < b0) return -1;
    for (long b = b0; b < b1; ++b) {
        long first = b * r - raw_pos0;
        if (first < 0 || first + r > n_raw) return -1;
        orc_pool_block(raw_k + (size_t)first * D, raw_v + (size_t)first * D, r, D, w,
                       out_k + (size_t)(b - b0) * D, out_v + (size_t)(b - b0) * D);
    }
    return b1 - b0;
}

/* ---- [KVC], the pooled-key reading of R3 ----------------------------------
 * In the alternative reading of where an indexer key comes from, the compressor
 * pools per-token indexer keys with the block's own weights: the key of block b
 * is sum_t alpha_t ki_t with alpha = softmax over the block of w . k_t (the
 * same alpha as orc_pool_block). */
void orc_pool_block_keys(const double *k, const double *ki, int n, int D, int DI,
                         const double *w, double *out_ki)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)n);
    double smax = -INFINITY;
    for (int t = 0; t < n; ++t) {
        double acc = 0.0;
        for (int d = 0; d < D; ++d) acc += w[d] * k[(size_t)t * D + d];
        s[t] = acc;
        if (acc > smax) smax = acc;
    }
    double z = 0.0;
    for (int t = 0; t < n; ++t) z += exp(s[t] - smax);
    for (int c = 0; c < DI; ++c) out_ki[c] = 0.0;
    for (int t = 0; t < n; ++t) {
        double a = exp(s[t] - smax) / z;
        for (int c = 0; c < DI; ++c) out_ki[c] += a * ki[(size_t)t * DI + c];
    }
    free(s);
}

/* Pooled keys of blocks b0 .. b1-1 (rows as orc_compress_range); -1 if a block
 * reaches outside the raw rows given. */
long orc_compress_range_keys(const double *raw_k, const double *raw_ki, long raw_pos0, long n_raw,
                             int D, int DI, const double *w, int r, long b0, long b1, double *out_ki)
{
    if (r <= 0 || b1 < b0) return -1;
    for (long b = b0; b < b1; ++b) {
        long first = b * r - raw_pos0;
        if (first < 0 || first + r > n_raw) return -1;
        orc_pool_block_keys(raw_k + (size_t)first * D, raw_ki + (size_t)first * DI, r, D, DI, w,
                            out_ki + (size_t)(b - b0) * DI);
    }
    return b1 - b0;
}

/* ---- [KVC] + R3/R4/R10/R11: the indexer ----------------------------------- */

/* score_j = q . kidx_j in double, for j = 0 .. n-1 */
void orc_index_scores(const double *q, const double *kidx, long n, int d, double *out)
{
    for (long j = 0; j < n; ++j) {
        double acc = 0.0;
        for (int c = 0; c < d; ++c) acc += q[c] * kidx[(size_t)j * d + c];
        out[j] = acc;
    }
}

typedef struct { float s; int j; } orc_ranked;

static int orc_rank_cmp(const void *a, const void *b)
{
    const orc_ranked *x = (const orc_ranked *)a, *y = (const orc_ranked *)b;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    return (x->j < y->j) ? -1 : (x->j > y->j);
}

static int orc_int_cmp(const void *a, const void *b)
{
    int x = *(const int *)a, y = *(const int *)b;
    return (x > y) - (x < y);
}

/* The k highest scores (ranked in binary32, ties to the lower index).
 * Writes min(k, n) indices in ascending order and returns that count. */
int orc_topk(const double *score, long n, int k, int *out_idx)
{
    orc_ranked *r = (orc_ranked *)malloc(sizeof(orc_ranked) * (size_t)(n > 0 ? n : 1));
    for (long j = 0; j < n; ++j) { r[j].s = (float)score[j]; r[j].j = (int)j; }
    qsort(r, (size_t)n, sizeof(orc_ranked), orc_rank_cmp);
    int m = (n < k) ? (int)n : k;
    for (int i = 0; i < m; ++i) out_idx[i] = r[i].j;
    qsort(out_idx, (size_t)m, sizeof(int), orc_int_cmp);
    free(r);
    return m;
}

/* Indexer for n_q queries at positions q_pos0 .. q_pos0+n_q-1.  Query i sees
 * rows j < min(n_rows, floor((q_pos0+i+1)/ratio)).  out_idx is [n_q, k]
 * (ascending, padded with -1), out_n [n_q] the count kept. */
void orc_indexer(const double *q_idx, int n_q, const double *kidx, long n_rows, int d,
                 long q_pos0, int ratio, int k, int *out_idx, int *out_n)
{
    double *s = (double *)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
    for (int i = 0; i < n_q; ++i) {
        long n_vis = orc_rows_visible(q_pos0 + i, ratio);
        if (n_vis > n_rows) n_vis = n_rows;
        orc_index_scores(q_idx + (size_t)i * d, kidx, n_vis, d, s);
        int *row = out_idx + (size_t)i * k;
        int m = orc_topk(s, n_vis, k, row);
        for (int t = m; t < k; ++t) row[t] = -1;
        out_n[i] = m;
    }
    free(s);
}

/* ---- [ARCH] + R12: multi-query attention ---------------------------------- */

/* For each head h: o_h = sum_j softmax_j(scale * q_h . K_j) V_j over the n rows
 * given; one KV head shared by all H query heads. */
void orc_attend(const double *q, int H, int D, double scale,
                const double *K, const double *V, long n, double *out)
{
    double *z = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int h = 0; h < H; ++h) {
        const double *qh = q + (size_t)h * D;
        double zmax = -INFINITY;
        for (long j = 0; j < n; ++j) {
            double acc = 0.0;
            for (int d = 0; d < D; ++d) acc += qh[d] * K[(size_t)j * D + d];
            z[j] = scale * acc;
            if (z[j] > zmax) zmax = z[j];
        }
        double den = 0.0;
        for (long j = 0; j < n; ++j) den += exp(z[j] - zmax);
        double *oh = out + (size_t)h * D;
        for (int d = 0; d < D; ++d) oh[d] = 0.0;
        for (long j = 0; j < n; ++j) {
            double a = exp(z[j] - zmax) / den;
            for (int d = 0; d < D; ++d) oh[d] += a * V[(size_t)j * D + d];
        }
    }
    free(z);
}

/* The key set of one query at position p: the window rows (R9), then the
 * compressed rows -- sel[0..n_sel-1] when sel is given (negative entries are
 * padding and skipped), else rows 0 .. n_sel-1.  raw rows hold positions
 * raw_pos0 .. raw_pos0+n_raw-1.  Returns the number of rows gathered, or -1
 * if a window position is missing from the raw rows. */
static long orc_gather_union(int D, long p, int window,
                             const double *raw_k, const double *raw_v, long raw_pos0, long n_raw,
                             const double *comp_k, const double *comp_v,
                             const int *sel, long n_sel, double *K, double *V)
{
    long first = p - window + 1;
    if (first < 0) first = 0;
    long n = 0;
    for (long t = first; t <= p; ++t) {
        long i = t - raw_pos0;
        if (i < 0 || i >= n_raw) return -1;
        memcpy(K + (size_t)n * D, raw_k + (size_t)i * D, sizeof(double) * (size_t)D);
        memcpy(V + (size_t)n * D, raw_v + (size_t)i * D, sizeof(double) * (size_t)D);
        ++n;
    }
    for (long s = 0; s < n_sel; ++s) {
        long j = sel ? sel[s] : s;
        if (j < 0) continue;
        memcpy(K + (size_t)n * D, comp_k + (size_t)j * D, sizeof(double) * (size_t)D);
        memcpy(V + (size_t)n * D, comp_v + (size_t)j * D, sizeof(double) * (size_t)D);
        ++n;
    }
    return n;
}

/* One decode step's attention at position p (one query, H heads).
 * Returns 0, or -1 if the raw rows do not cover the window. */
int orc_decode_attend(int H, int D, double scale, const double *q, long p, int window,
                      const double *raw_k, const double *raw_v, long raw_pos0, long n_raw,
                      const double *comp_k, const double *comp_v, const int *sel, long n_sel,
                      double *out)
{
    size_t cap = (size_t)window + (size_t)(n_sel > 0 ? n_sel : 0);
    double *K = (double *)malloc(sizeof(double) * cap * D + 8);
    double *V = (double *)malloc(sizeof(double) * cap * D + 8);
    long n = orc_gather_union(D, p, window, raw_k, raw_v, raw_pos0, n_raw,
                              comp_k, comp_v, sel, n_sel, K, V);
    if (n >= 0) orc_attend(q, H, D, scale, K, V, n, out);
    free(K);
    free(V);
    return n < 0 ? -1 : 0;
}

/* Prefill attention for T queries at positions q_pos0 .. q_pos0+T-1.
 * raw rows hold positions q_pos0-n_prior .. q_pos0+T-1.  With ratio == 0 no
 * compressed row is attended; with sel (shape [T, k_stride]) query i attends
 * the rows listed in its sel row; without sel it attends every visible row.
 * q and out are [T, H, D].  Returns 0, or -1 on a missing window row. */
int orc_prefill_attend(int T, int H, int D, double scale, const double *q,
                       const double *raw_k, const double *raw_v, long n_prior, int window,
                       const double *comp_k, const double *comp_v,
                       const int *sel, int k_stride, long q_pos0, int ratio, double *out)
{
    int rc = 0;
    for (int i = 0; i < T; ++i) {
        long p = q_pos0 + i;
        const int *srow = NULL;
        long n_sel = 0;
        if (ratio > 0) {
            if (sel) { srow = sel + (size_t)i * k_stride; n_sel = k_stride; }
            else n_sel = orc_rows_visible(p, ratio);
        }
        if (orc_decode_attend(H, D, scale, q + (size_t)i * H * D, p, window,
                              raw_k, raw_v, q_pos0 - n_prior, n_prior + T,
                              comp_k, comp_v, srow, n_sel, out + (size_t)i * H * D) != 0)
            rc = -1;
    }
    return rc;
}
