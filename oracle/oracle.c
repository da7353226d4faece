/*
 * oracle.c -- plain, slow, CPU reference for the paged key scoring and the
 * exact top-k selection of a sparse-attention decode step.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library.  The GPU library never
 * includes, links or calls it, and this file includes nothing from it.
 *
 * What it follows:
 *  - The score is the indexer's: for query row r and key position j
 *        s[r,j] = sum_h w[r,h] * ReLU( q[r,h,:] . (k[j,:] * scale[j]) )
 *    with k stored as FP8 E4M3 and one f32 scale per key.  The reference check
 *    of "sgl-amd-mono-upstream PR 18" (GLM-5.3 indexer launch), section
 *    "Modifications / 0. An exact top-k check", recomputes launch scores in
 *    f64 from the launch's own bf16 query, head weights and cached keys; this
 *    file does the same, literally, in double precision.
 *  - The selection list: the keys strictly above the k-th largest score in
 *    ascending position, then the keys tied with it in ascending position
 *    until the list holds k; rows with n <= k keep every key and pad with -1.
 *    The same page's "missed" count defines the exact top-k set as the first
 *    k keys by (score descending, position ascending); the list here is built
 *    from that set by a full sort.
 *
 * Nothing here is blocked, fused or reordered beyond the definitions above.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- formats */

/* FP8 E4M3 (the OCP "fn" variant used by FP8 KV caches): 1 sign bit, 4
 * exponent bits with bias 7, 3 mantissa bits.  Exponent field 0 holds the
 * subnormals m/8 * 2^-6; S.1111.111 is NaN; there are no infinities, so the
 * largest finite value is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_f64(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* Nearest E4M3 code of an f32 value, ties to the even mantissa, magnitudes
 * beyond the largest finite value (448) saturated to +-448, NaN to the NaN
 * code.  Written from the format definition: the magnitude is compared with
 * every finite non-negative code (0x00 .. 0x7E, increasing with the code), and
 * of two equally near codes the one with an even mantissa (even code) wins. */
uint8_t oracle_f32_to_e4m3(float x)
{
    const uint8_t sign = signbit(x) ? 0x80 : 0x00;
    if (isnan(x))
        return 0x7F;
    const double a = fabs((double)x);
    if (a >= 448.0)
        return (uint8_t)(sign | 0x7E);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        const double err = fabs(oracle_e4m3_to_f64((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

/* bf16 is the upper half of an IEEE-754 binary32. */
double oracle_bf16_to_f64(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* ReLU that lets NaN through (a NaN dot product must not turn into 0). */
static double relu(double x)
{
    if (isnan(x))
        return x;
    return x > 0.0 ? x : 0.0;
}

/* ------------------------------------------------------------------ scores */

/* Error codes shared by the entry points below. */
enum { OR_OK = 0, OR_ERR_ARG = -1, OR_ERR_BOUNDS = -6 };

typedef struct {
    int q_is_e4m3;               /* 0: q holds bf16 bits, 1: q holds E4M3 codes */
    const void *q;               /* [R][H][D] */
    const float *head_w;         /* [R][H] */
    const uint8_t *k_cache;      /* [pool_pages][P][D] E4M3 codes */
    const float *k_scale;        /* [pool_pages][P] */
    int64_t pool_pages;
    const int32_t *block_table;  /* [n_req][max_pages] */
    int max_pages;
    const int32_t *seq_lens;     /* [R] keys visible to each row */
    const int32_t *row_req;      /* [R] request of each row */
    int R, H, D, P;
} oracle_problem;

static double q_value(const oracle_problem *pb, int r, int h, int d)
{
    size_t i = ((size_t)r * pb->H + h) * pb->D + d;
    if (pb->q_is_e4m3)
        return oracle_e4m3_to_f64(((const uint8_t *)pb->q)[i]);
    return oracle_bf16_to_f64(((const uint16_t *)pb->q)[i]);
}

/* s[r, j] by the literal formula.  Key j of row r lives in page
 * block_table[row_req[r]][j / P], slot j % P. */
static int score_one(const oracle_problem *pb, int r, int64_t j, double *out)
{
    int req = pb->row_req[r];
    int64_t page_idx = j / pb->P;
    int slot = (int)(j % pb->P);
    int32_t page;
    double *kf;
    double s = 0.0;
    int h, d;

    if (j < 0 || j >= pb->seq_lens[r] || page_idx >= pb->max_pages)
        return OR_ERR_BOUNDS;
    page = pb->block_table[(int64_t)req * pb->max_pages + page_idx];
    if (page < 0 || page >= pb->pool_pages)
        return OR_ERR_BOUNDS;

    /* k[j,:] * scale[j], each element decoded from its E4M3 code. */
    kf = (double *)malloc(sizeof(double) * (size_t)pb->D);
    if (!kf)
        return OR_ERR_ARG;
    for (d = 0; d < pb->D; ++d) {
        size_t ki = ((size_t)page * pb->P + slot) * pb->D + d;
        kf[d] = oracle_e4m3_to_f64(pb->k_cache[ki]) *
                (double)pb->k_scale[(size_t)page * pb->P + slot];
    }
    for (h = 0; h < pb->H; ++h) {
        double dot = 0.0;
        for (d = 0; d < pb->D; ++d)
            dot += q_value(pb, r, h, d) * kf[d];
        s += (double)pb->head_w[(size_t)r * pb->H + h] * relu(dot);
    }
    free(kf);
    *out = s;
    return OR_OK;
}

static int check_problem(const oracle_problem *pb)
{
    int r;
    if (!pb->q || !pb->head_w || !pb->k_cache || !pb->k_scale || !pb->block_table ||
        !pb->seq_lens || !pb->row_req)
        return OR_ERR_ARG;
    if (pb->R < 0 || pb->H <= 0 || pb->D <= 0 || pb->P <= 0 || pb->max_pages < 0)
        return OR_ERR_ARG;
    for (r = 0; r < pb->R; ++r) {
        if (pb->seq_lens[r] < 0 || (int64_t)pb->seq_lens[r] > (int64_t)pb->max_pages * pb->P)
            return OR_ERR_BOUNDS;
        if (pb->row_req[r] < 0)
            return OR_ERR_ARG;
    }
    return OR_OK;
}

/* Every score of every row: out[r * out_stride + j] for j < seq_lens[r].
 * Entries at j >= seq_lens[r] are not written. */
int oracle_scores(int q_is_e4m3, const void *q, const float *head_w,
                  const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                  const int32_t *block_table, int max_pages,
                  const int32_t *seq_lens, const int32_t *row_req,
                  int R, int H, int D, int P, double *out, int64_t out_stride)
{
    oracle_problem pb = {q_is_e4m3, q, head_w, k_cache, k_scale, pool_pages,
                         block_table, max_pages, seq_lens, row_req, R, H, D, P};
    int r, st = check_problem(&pb);
    if (st != OR_OK)
        return st;
    for (r = 0; r < R; ++r) {
        int64_t j;
        if ((int64_t)seq_lens[r] > out_stride)
            return OR_ERR_ARG;
        for (j = 0; j < seq_lens[r]; ++j) {
            st = score_one(&pb, r, j, &out[(int64_t)r * out_stride + j]);
            if (st != OR_OK)
                return st;
        }
    }
    return OR_OK;
}

/* The scores of one row at the listed positions only (for sampled checks of
 * workloads too large to score whole on the CPU). */
int oracle_score_positions(int q_is_e4m3, const void *q, const float *head_w,
                           const uint8_t *k_cache, const float *k_scale, int64_t pool_pages,
                           const int32_t *block_table, int max_pages,
                           const int32_t *seq_lens, const int32_t *row_req,
                           int R, int H, int D, int P,
                           int row, const int64_t *positions, int64_t npos, double *out)
{
    oracle_problem pb = {q_is_e4m3, q, head_w, k_cache, k_scale, pool_pages,
                         block_table, max_pages, seq_lens, row_req, R, H, D, P};
    int64_t i;
    int st = check_problem(&pb);
    if (st != OR_OK)
        return st;
    if (row < 0 || row >= R)
        return OR_ERR_ARG;
    for (i = 0; i < npos; ++i) {
        st = score_one(&pb, row, positions[i], &out[i]);
        if (st != OR_OK)
            return st;
    }
    return OR_OK;
}

/* --------------------------------------------------------------- selection */

/* Ranking of f32 scores: larger first; every NaN ranks below every number and
 * all NaNs tie; -0 and +0 tie (plain float comparison). */
static int ranks_above(float a, float b)
{
    if (isnan(a))
        return 0;
    if (isnan(b))
        return 1;
    return a > b;
}

static int ties_with(float a, float b)
{
    if (isnan(a) || isnan(b))
        return isnan(a) && isnan(b);
    return a == b;
}

typedef struct {
    float s;
    int32_t pos;
} scored_pos;

/* Score descending, then position ascending: a total order on distinct
 * positions, so the sort result does not depend on qsort's stability. */
static int cmp_desc_then_pos(const void *pa, const void *pb)
{
    const scored_pos *a = (const scored_pos *)pa, *b = (const scored_pos *)pb;
    if (ranks_above(a->s, b->s))
        return -1;
    if (ranks_above(b->s, a->s))
        return 1;
    return (a->pos > b->pos) - (a->pos < b->pos);
}

/* Exact top-k list of one row of n scores (see the header comment). */
int oracle_topk(const float *scores, int64_t n, int k, int32_t *out)
{
    scored_pos *v;
    float t;
    int64_t j;
    int filled = 0;

    if (k <= 0 || n < 0 || (n > 0 && !scores) || !out)
        return OR_ERR_ARG;
    if (n <= k) {
        for (j = 0; j < k; ++j)
            out[j] = j < n ? (int32_t)j : -1;
        return OR_OK;
    }
    v = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)n);
    if (!v)
        return OR_ERR_ARG;
    for (j = 0; j < n; ++j) {
        v[j].s = scores[j];
        v[j].pos = (int32_t)j;
    }
    qsort(v, (size_t)n, sizeof(scored_pos), cmp_desc_then_pos);
    t = v[k - 1].s; /* the k-th largest score, counting repeats */
    free(v);

    for (j = 0; j < n && filled < k; ++j)
        if (ranks_above(scores[j], t))
            out[filled++] = (int32_t)j;
    for (j = 0; j < n && filled < k; ++j)
        if (ties_with(scores[j], t))
            out[filled++] = (int32_t)j;
    return filled == k ? OR_OK : OR_ERR_ARG;
}

/* Many rows at once: row r has n = lens[r] scores at scores + r*stride. */
int oracle_topk_rows(const float *scores, int64_t stride, const int32_t *lens, int R,
                     int k, int32_t *out)
{
    int r, st;
    for (r = 0; r < R; ++r) {
        st = oracle_topk(scores + (int64_t)r * stride, lens[r], k, out + (int64_t)r * k);
        if (st != OR_OK)
            return st;
    }
    return OR_OK;
}

/* ------------------------------------------------ FP8 query quantisation */

/* The FP8 (E4M3) query of a bf16 index query, one scale per (row, head):
 * amax = the largest |q| of the head's elements, scale = amax / 448 in f32,
 * inv = 1 / scale in f32, code = E4M3(q * inv) (f32 product, nearest-even
 * rounding, saturated), and the head weight w * scale in f32, so that
 * w' * relu(code . k) approximates w * relu(q . k).  A head whose elements
 * are all zero gets scale 0: codes 0 and weight 0.  This is the per-token FP8
 * quantisation that "[Perf] [MI355X] minimax_m31" (section "Modifications",
 * o_proj bullet) describes -- amax / 448, a reciprocal, clamp, round to
 * nearest even -- applied per head to the index query, with the reciprocal
 * taken as a correctly rounded f32 division.  q and q8 are [R][H][D], head_w
 * and w_out [R][H]. */
void oracle_quantize_query(const uint16_t *q, const float *head_w, int R, int H, int D,
                           uint8_t *q8, float *w_out)
{
    for (int r = 0; r < R; ++r)
        for (int h = 0; h < H; ++h) {
            const uint16_t *row = q + ((size_t)r * H + h) * D;
            uint8_t *out = q8 + ((size_t)r * H + h) * D;
            float amax = 0.0f;
            for (int d = 0; d < D; ++d) {
                const float a = fabsf((float)oracle_bf16_to_f64(row[d]));
                if (a > amax)
                    amax = a;
            }
            const float scale = amax / 448.0f;
            const float inv = scale > 0.0f ? 1.0f / scale : 0.0f;
            w_out[(size_t)r * H + h] = head_w[(size_t)r * H + h] * scale;
            for (int d = 0; d < D; ++d) {
                const float x = (float)oracle_bf16_to_f64(row[d]);
                out[d] = scale > 0.0f ? oracle_f32_to_e4m3(x * inv) : 0;
            }
        }
}

/* ------------------------------------------------------- physical slots */

/* A list of logical positions as rows of the paged key cache: position p of
 * row r lives in page block_table[row_req[r]][p / page], row p % page of it,
 * i.e. cache slot page_id * page + p % page; -1 (padding) stays -1.
 * idx and out are [R][k]. */
void oracle_slots(const int32_t *idx, int R, int k, const int32_t *block_table, int max_pages,
                  const int32_t *row_req, int page, int32_t *out)
{
    for (int r = 0; r < R; ++r)
        for (int j = 0; j < k; ++j) {
            const int32_t p = idx[(size_t)r * k + j];
            out[(size_t)r * k + j] =
                p < 0 ? -1 : block_table[(size_t)row_req[r] * max_pages + p / page] * page + p % page;
        }
}

/* Tagged pairs ("sgl-amd-mono-upstream PR 11", section "3. The selected tokens
 * are tagged pairs"): each list entry travels with the launch's tag, so a
 * reader can tell this launch's entries from an earlier launch's without a
 * separate flag.  The pair of entry e and tag t is the 64-bit word whose low
 * 32 bits are e (as an unsigned 32-bit pattern) and whose high 32 bits are t.
 * entries and out have n elements. */
void oracle_tagged(const int32_t *entries, int64_t n, uint32_t tag, int64_t *out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = (int64_t)(((uint64_t)tag << 32) | (uint64_t)(uint32_t)entries[i]);
}

/* The keys a step writes ("sgl-amd-mono-upstream PR 18", section
 * "Modifications / 2", keys this launch writes): row r of the step owns the
 * slot at its request's position seq_lens[r] - 1 and writes its own index key
 * there, 128 E4M3 codes new_k[r] and the scale new_scale[r].  Every row of the
 * request then scores the cache as it stands after these stores.  Rows are
 * stored in order; a row with no keys stores nothing.  Returns 0, or -1 if a
 * slot's page is outside the pool (that row's store is skipped). */
int oracle_store_keys(uint8_t *k_cache, float *k_scale, int64_t pool_pages, const int32_t *block_table,
                      int max_pages, const int32_t *seq_lens, const int32_t *row_req, int R,
                      const uint8_t *new_k, const float *new_scale, int page, int dim)
{
    int st = 0;
    for (int r = 0; r < R; ++r) {
        const int32_t len = seq_lens[r];
        if (len < 1) continue;
        const int32_t pos = len - 1;
        const int32_t pg = block_table[(size_t)row_req[r] * max_pages + pos / page];
        if (pg < 0 || (int64_t)pg >= pool_pages) {
            st = -1;
            continue;
        }
        memcpy(k_cache + ((size_t)pg * page + (size_t)(pos % page)) * dim, new_k + (size_t)r * dim, (size_t)dim);
        k_scale[(size_t)pg * page + pos % page] = new_scale[r];
    }
    return st;
}

/* ------------------------------------------- the pages' prefix list order */

/* The order-preserving 32-bit image of a score that the pages' radix select
 * works on ("sgl-amd-mono-upstream PR 18", section "Modifications / 3", keys
 * held "as radix keys"): the IEEE-754 bits with the sign bit set for a
 * non-negative value and every bit flipped for a negative one, so images
 * compare as the values do; -0 counts as +0 and a NaN as the lowest image. */
static uint32_t radix_image(float x)
{
    uint32_t b;
    if (isnan(x))
        return 0u;
    memcpy(&b, &x, sizeof b);
    if (b == 0x80000000u)
        b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

/* The list of one row in the pages' order ("sgl-amd-mono-upstream PR 18",
 * section "Modifications / 0", the list check, and "Modifications / 3",
 * Order): the radix stops at the first of the threshold's 12- and 24-bit
 * prefixes whose keys (the row's keys whose image shares that prefix with the
 * k-th largest, T) number at most `room`, else it runs to all 32 bits.  With
 * the stopping prefix P the list is
 *   the keys whose prefix is above P, in position order;
 *   then the keys with prefix P that rank above T, in position order;
 *   then the keys tied with T, in position order, until k entries.
 * At 32 bits the middle part is empty and the list is oracle_topk's; the set
 * is oracle_topk's at every stop.  Rows with n <= k: as oracle_topk. */
int oracle_prefix_order(const float *scores, int64_t n, int k, int64_t room, int32_t *out)
{
    scored_pos *v;
    uint32_t t, p12, p24, tp;
    int64_t j, c12 = 0, c24 = 0;
    int filled = 0, sh;

    if (k <= 0 || n < 0 || (n > 0 && !scores) || !out || room < 0)
        return OR_ERR_ARG;
    if (n <= k)
        return oracle_topk(scores, n, k, out);
    v = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)n);
    if (!v)
        return OR_ERR_ARG;
    for (j = 0; j < n; ++j) {
        v[j].s = scores[j];
        v[j].pos = (int32_t)j;
    }
    qsort(v, (size_t)n, sizeof(scored_pos), cmp_desc_then_pos);
    t = radix_image(v[k - 1].s); /* the k-th largest, counting repeats */
    free(v);
    p12 = t >> 20;
    p24 = t >> 8;
    for (j = 0; j < n; ++j) {
        const uint32_t u = radix_image(scores[j]);
        c12 += (u >> 20) == p12;
        c24 += (u >> 8) == p24;
    }
    sh = c12 <= room ? 20 : (c24 <= room ? 8 : 0);
    tp = t >> sh;
    for (j = 0; j < n && filled < k; ++j)
        if ((radix_image(scores[j]) >> sh) > tp)
            out[filled++] = (int32_t)j;
    for (j = 0; j < n && filled < k; ++j) {
        const uint32_t u = radix_image(scores[j]);
        if ((u >> sh) == tp && u > t)
            out[filled++] = (int32_t)j;
    }
    for (j = 0; j < n && filled < k; ++j)
        if (radix_image(scores[j]) == t)
            out[filled++] = (int32_t)j;
    return OR_OK;
}
