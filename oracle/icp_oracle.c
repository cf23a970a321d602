/*
 * icp_oracle.c - plain CPU oracle for the decode-time ICP block indexer.
 *
 * TEST INFRASTRUCTURE. This is the slow, obviously-correct reference that the
 * CUDA library is checked against. Only the tests, the smoke check and the
 * benchmark's CPU-baseline leg load it. It shares no code, header, table or
 * helper with the CUDA path, and the CUDA path never loads it.
 *
 * Sources (FlashInfer "msa_ops" API documentation pages):
 *   [SCORE]   flashinfer.msa_ops.msa_icp_decode_index_score_sharded
 *             - description: which score_out columns are written, the P128 /
 *               P256 column meaning; columns past those are left as they were;
 *             - parameter index_q: the position of a request's token j is
 *               seq_len - decode_query_len + j;
 *             - parameter index_k: the [pages, page_size / world_size, 128] shard.
 *   [SELECT]  flashinfer.msa_ops.msa_icp_topk_select_publish
 *             - description: row (t, h) goes to peer h // heads_per_rank at row
 *               ((slot * world_size + rank) * heads_per_rank + h % heads_per_rank)
 *               * capacity + t; legacy rows are 33 int32 words (16 raw scores,
 *               16 ascending global ids, ready flag); each call writes all the
 *               rows, padded ones too;
 *             - parameter num_valid_pages: global B128 block counts per token;
 *             - parameter errors: a publish that finds no free row within
 *               spin_limit polls increments it.
 *   [PLAN]    flashinfer.msa_ops.prepare_msa_icp_indexer
 *             - init_blocks / local_blocks: forced begin / end blocks (sum <= 16);
 *             - decode(): score plane -> Top16 select and publish -> owner merge.
 *
 * Readings where the pages leave a step open (each one is listed in the
 * design notes of the repository):
 *   - per-key score: the plain dot product of the 128 dequantised fp8 values;
 *     no scale, no activation, no head weights (no such argument exists);
 *   - a key is visible to token t iff its position is <= the token's position;
 *   - block score: the maximum over the block's visible keys; -inf if none;
 *   - Top16: forced ids first, then the best remaining ids by (score
 *     descending, id ascending); output in ascending id order, padded with
 *     id -1 and score -inf;
 *   - global id of column c is c * index_scale + index_offset;
 *   - merge: union of the published lists, maximum score per id, then the
 *     same Top16 rule with the token's num_valid_pages;
 *   - ready flag: 0 = free, 1 = full; the merge clears it back to 0;
 *   - P256 with world_size 1 (outside the pages' layouts): one column per
 *     B128 block, so column c is half c % 2 of page c / 2.
 *
 * Exactness: every float8_e4m3fn value is a multiple of 2^-9 with magnitude
 * at most 448, so each product is a multiple of 2^-18 below 2^17.7 and any
 * sum of 128 products fits in 43 bits.  fp64 accumulation is therefore exact
 * in any order; the score plane below holds exact values.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_HEADS 4
#define ORC_DIM 128
#define ORC_TOPK 16
#define ORC_ROW_WORDS 33

/* ------------------------------------------------------------------------ */
/* float8_e4m3fn decoding, from the format definition: 1 sign bit, 4        */
/* exponent bits with bias 7, 3 mantissa bits; exponent 0 is subnormal      */
/* (m * 2^-9); S.1111.111 is NaN; there is no infinity.                    */
/* ------------------------------------------------------------------------ */
double icp_orc_e4m3(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int expo = (code >> 3) & 15;
    int mant = code & 7;
    double mag;
    if (expo == 15 && mant == 7)
        return NAN;
    if (expo == 0)
        mag = ldexp((double)mant, -9);
    else
        mag = ldexp(1.0 + mant / 8.0, expo - 7);
    return sign ? -mag : mag;
}

/* Number of columns of a request that hold keys, and the number written
 * (padded to the next multiple of 4) [SCORE description]. */
static int unit_tokens(int page_size, int world_size)
{
    /* P128: a column is a global B128 block.  P256 sharded: a column is a
     * local page.  P256 unsharded (our extension): a column is a B128 block. */
    if (page_size == 256 && world_size == 1)
        return 128;
    return page_size;
}

int icp_orc_columns_with_keys(int seq_len, int page_size, int world_size)
{
    int u = unit_tokens(page_size, world_size);
    if (seq_len <= 0)
        return 0;
    return (seq_len + u - 1) / u;
}

int icp_orc_columns_written(int seq_len, int page_size, int world_size)
{
    int n = icp_orc_columns_with_keys(seq_len, page_size, world_size);
    return (n + 3) / 4 * 4;
}

/* Key rows of column c on this rank: count, page slot in the block table,
 * first row inside the shard page, and token position of the first row.
 * [SCORE description + parameter index_k]: the rank holds rows
 * [rank * page_size / world_size, (rank + 1) * page_size / world_size) of
 * every page, which is what makes the P256 column c map to global block
 * 2 c + rank * 2 // world_size. */
static void column_rows(int c, int rank, int world_size, int page_size,
                        int *nrows, int *page_slot, int *row0, int64_t *pos0)
{
    if (page_size == 256 && world_size == 1) {
        *nrows = 128;
        *page_slot = c / 2;
        *row0 = (c % 2) * 128;
        *pos0 = (int64_t)c * 128;
    } else {
        int rp = page_size / world_size;
        *nrows = rp;
        *page_slot = c;
        *row0 = 0;
        *pos0 = (int64_t)c * page_size + (int64_t)rank * rp;
    }
}

/*
 * Score plane rows of one request [SCORE]: its ntok tokens are plane rows
 * row0 .. row0 + ntok - 1 (index_q rows likewise), token j at position
 * seq_len - ntok + j.  For every such token, head h and column
 * c < columns_written(seq_len):
 *   plane[t][h][c]    = max over visible keys of sum_i deq(q[t,h,i]) deq(k[key,i])
 *                       (exact), or -inf when no key of the column is visible;
 *   absplane[t][h][c] = max over the same keys of sum_i |deq(q) deq(k)|
 *                       (0 when none), the scale of the rounding tolerance.
 * Columns c >= columns_written(seq_len) are left untouched.  qd holds room
 * for ntok * 4 * 128 doubles, kd for 128.  Returns 0, -2 on a NaN input
 * code, -3 on a page id outside [0, num_pages), -4 if the request needs more
 * than `cols` columns.
 */
static int score_request(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
                         const int32_t *bt_row, int seq_len, int64_t row0, int ntok, int cols,
                         int rank, int world_size, int page_size, double *qd, double *kd,
                         double *plane, double *absplane)
{
    int rows_per_page = page_size / world_size;
    int nkeys_cols = icp_orc_columns_with_keys(seq_len, page_size, world_size);
    int nwritten = icp_orc_columns_written(seq_len, page_size, world_size);
    if (nwritten > cols)
        return -4;
    /* dequantise this request's queries: rows t = row0 + j, heads 0..3 */
    for (int j = 0; j < ntok; ++j)
        for (int h = 0; h < ORC_HEADS; ++h)
            for (int i = 0; i < ORC_DIM; ++i) {
                int64_t t = row0 + j;
                double v = icp_orc_e4m3(index_q[(t * ORC_HEADS + h) * ORC_DIM + i]);
                if (isnan(v))
                    return -2;
                qd[((int64_t)j * ORC_HEADS + h) * ORC_DIM + i] = v;
            }

    /* start every written column at "no visible key" */
    for (int j = 0; j < ntok; ++j)
        for (int h = 0; h < ORC_HEADS; ++h)
            for (int c = 0; c < nwritten; ++c) {
                int64_t t = row0 + j;
                int64_t o = (t * ORC_HEADS + h) * cols + c;
                plane[o] = -INFINITY;
                if (absplane)
                    absplane[o] = 0.0;
            }

    for (int c = 0; c < nkeys_cols; ++c) {
        int nrows, page_slot, row_in_page;
        int64_t pos0;
        int32_t page;
        column_rows(c, rank, world_size, page_size, &nrows, &page_slot, &row_in_page, &pos0);
        if (pos0 >= seq_len)
            continue; /* this rank holds no key of the column below seq_len */
        page = bt_row[page_slot];
        if (page < 0 || page >= num_pages)
            return -3;
        for (int r = 0; r < nrows; ++r) {
            int64_t pos = pos0 + r;
            const uint8_t *krow =
                index_k + ((int64_t)page * rows_per_page + row_in_page + r) * ORC_DIM;
            if (pos >= seq_len)
                break;
            for (int i = 0; i < ORC_DIM; ++i) {
                kd[i] = icp_orc_e4m3(krow[i]);
                if (isnan(kd[i]))
                    return -2;
            }
            for (int j = 0; j < ntok; ++j) {
                int64_t p_t = (int64_t)seq_len - ntok + j; /* token position */
                int64_t t = row0 + j;
                if (pos > p_t)
                    continue; /* key after the token: masked */
                for (int h = 0; h < ORC_HEADS; ++h) {
                    const double *qv = qd + ((int64_t)j * ORC_HEADS + h) * ORC_DIM;
                    double dot = 0.0, adot = 0.0;
                    int64_t o = (t * ORC_HEADS + h) * cols + c;
                    for (int i = 0; i < ORC_DIM; ++i) {
                        dot += qv[i] * kd[i];
                        adot += fabs(qv[i] * kd[i]);
                    }
                    if (dot > plane[o])
                        plane[o] = dot;
                    if (absplane && adot > absplane[o])
                        absplane[o] = adot;
                }
            }
        }
    }
    return 0;
}

/*
 * Score plane [SCORE] of a decode batch: request b's tokens are rows
 * b * decode_query_len + j, at positions seq_len_b - decode_query_len + j
 * (parameter index_q).  Returns 0; -1 on a bad argument; otherwise the
 * first error of score_request.
 */
int icp_orc_score(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
                  const int32_t *block_table, int64_t bt_stride, const int32_t *seq_lens,
                  int batch, int cols, int rank, int world_size, int page_size,
                  int decode_query_len, double *plane, double *absplane)
{
    int dql = decode_query_len;
    double *qd = NULL, *kd = NULL;
    int rc = 0;

    if (batch < 0 || cols <= 0 || dql < 1 || world_size < 1 || rank < 0 || rank >= world_size)
        return -1;
    if (page_size != 128 && page_size != 256)
        return -1;
    if (page_size % world_size != 0)
        return -1;

    qd = (double *)malloc(sizeof(double) * (size_t)dql * ORC_HEADS * ORC_DIM);
    kd = (double *)malloc(sizeof(double) * ORC_DIM);
    if (!qd || !kd) {
        free(qd);
        free(kd);
        return -1;
    }
    for (int b = 0; b < batch && rc == 0; ++b)
        rc = score_request(index_q, index_k, num_pages, block_table + (int64_t)b * bt_stride,
                           seq_lens[b], (int64_t)b * dql, dql, cols, rank, world_size,
                           page_size, qd, kd, plane, absplane);
    free(qd);
    free(kd);
    return rc;
}

/*
 * Score plane of a prefill window.  The pages name the prefill chain
 * (prepare_msa_icp_indexer: prefill_window_plan, prefill_local,
 * prefill_merge) but its own pages are missing; the reading here is the
 * decode plane with a per-request query length.  Request b contributes the
 * tokens qo_indptr[b] .. qo_indptr[b+1] - 1 of the window, the newest
 * n_b = qo_indptr[b+1] - qo_indptr[b] positions of its seq_len_b (so token
 * j sits at seq_len_b - n_b + j, exactly as a decode query of length n_b),
 * and each gets the request's columns_written(seq_len_b) columns.
 * Returns 0; -1 on a bad argument (qo_indptr not starting at 0 or
 * decreasing, or a chunk longer than its seq_len); otherwise the first
 * error of score_request.
 */
int icp_orc_score_chunks(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
                         const int32_t *block_table, int64_t bt_stride, const int32_t *seq_lens,
                         const int32_t *qo_indptr, int batch, int cols, int rank,
                         int world_size, int page_size, double *plane, double *absplane)
{
    int maxn = 1;
    double *qd = NULL, *kd = NULL;
    int rc = 0;

    if (batch < 0 || cols <= 0 || world_size < 1 || rank < 0 || rank >= world_size)
        return -1;
    if ((page_size != 128 && page_size != 256) || page_size % world_size != 0)
        return -1;
    if (qo_indptr[0] != 0)
        return -1;
    for (int b = 0; b < batch; ++b) {
        int n = qo_indptr[b + 1] - qo_indptr[b];
        if (n < 0 || n > seq_lens[b])
            return -1;
        if (n > maxn)
            maxn = n;
    }
    qd = (double *)malloc(sizeof(double) * (size_t)maxn * ORC_HEADS * ORC_DIM);
    kd = (double *)malloc(sizeof(double) * ORC_DIM);
    if (!qd || !kd) {
        free(qd);
        free(kd);
        return -1;
    }
    for (int b = 0; b < batch && rc == 0; ++b) {
        int n = qo_indptr[b + 1] - qo_indptr[b];
        if (n == 0)
            continue;
        rc = score_request(index_q, index_k, num_pages, block_table + (int64_t)b * bt_stride,
                           seq_lens[b], qo_indptr[b], n, cols, rank, world_size, page_size, qd,
                           kd, plane, absplane);
    }
    free(qd);
    free(kd);
    return rc;
}

/* ------------------------------------------------------------------------ */
/* Top16 with forced blocks                                                 */
/* ------------------------------------------------------------------------ */
typedef struct {
    int32_t id;
    double score;
} orc_pair;

/* (score descending, id ascending); -0 and +0 compare equal as doubles. */
static int by_score_then_id(const void *a, const void *b)
{
    const orc_pair *x = (const orc_pair *)a, *y = (const orc_pair *)b;
    if (x->score > y->score)
        return -1;
    if (x->score < y->score)
        return 1;
    return (x->id < y->id) ? -1 : (x->id > y->id);
}

static int by_id(const void *a, const void *b)
{
    const orc_pair *x = (const orc_pair *)a, *y = (const orc_pair *)b;
    return (x->id < y->id) ? -1 : (x->id > y->id);
}

/*
 * Top16 of one row given as (id, score) pairs with distinct ids.
 * Valid ids are 0 <= id < nvp.  If nvp <= 16 every valid id is kept.
 * Otherwise ids in [0, init) and [nvp - local, nvp) are forced, and the
 * remaining 16 - |forced| slots go to the best other valid ids by
 * (score descending, id ascending).  Output: ids ascending, then padding
 * (-1, -inf).  Returns the number of real entries, or -1 on a NaN score or
 * duplicate id.
 */
int icp_orc_select_pairs(int n, const int32_t *ids, const float *scores, int nvp,
                         int init_blocks, int local_blocks, float *out_scores,
                         int32_t *out_ids)
{
    orc_pair *forced = NULL, *rest = NULL;
    int nf = 0, nr = 0, nout = 0;
    orc_pair out[ORC_TOPK];

    forced = (orc_pair *)malloc(sizeof(orc_pair) * (size_t)(n > 0 ? n : 1));
    rest = (orc_pair *)malloc(sizeof(orc_pair) * (size_t)(n > 0 ? n : 1));
    if (!forced || !rest) {
        free(forced);
        free(rest);
        return -1;
    }
    for (int i = 0; i < n; ++i) {
        orc_pair p;
        int is_forced;
        if (ids[i] < 0 || ids[i] >= nvp)
            continue;
        p.id = ids[i];
        p.score = (double)scores[i];
        if (isnan(p.score)) {
            free(forced);
            free(rest);
            return -1;
        }
        if (nvp <= ORC_TOPK)
            is_forced = 1;
        else
            is_forced = (p.id < init_blocks) || (p.id >= nvp - local_blocks);
        if (is_forced)
            forced[nf++] = p;
        else
            rest[nr++] = p;
    }
    /* duplicate ids are a caller error */
    {
        orc_pair *all = (orc_pair *)malloc(sizeof(orc_pair) * (size_t)(nf + nr + 1));
        int dup = 0;
        memcpy(all, forced, sizeof(orc_pair) * (size_t)nf);
        memcpy(all + nf, rest, sizeof(orc_pair) * (size_t)nr);
        qsort(all, (size_t)(nf + nr), sizeof(orc_pair), by_id);
        for (int i = 1; i < nf + nr; ++i)
            if (all[i].id == all[i - 1].id)
                dup = 1;
        free(all);
        if (dup || nf > ORC_TOPK) {
            free(forced);
            free(rest);
            return -1;
        }
    }
    for (int i = 0; i < nf; ++i)
        out[nout++] = forced[i];
    qsort(rest, (size_t)nr, sizeof(orc_pair), by_score_then_id);
    for (int i = 0; i < nr && nout < ORC_TOPK; ++i)
        out[nout++] = rest[i];
    qsort(out, (size_t)nout, sizeof(orc_pair), by_id);
    for (int i = 0; i < ORC_TOPK; ++i) {
        if (i < nout) {
            out_ids[i] = out[i].id;
            out_scores[i] = (float)out[i].score;
        } else {
            out_ids[i] = -1;
            out_scores[i] = -INFINITY;
        }
    }
    free(forced);
    free(rest);
    return nout;
}

/*
 * Top16 of every row (t, h) of a float32 plane [T, heads, K]: the pairs are
 * (c * index_scale + index_offset, scores[t][h][c]) for c < K.  Output
 * [T, heads, 16].  Returns 0 or -1.
 */
int icp_orc_select(const float *scores, int T, int heads, int K, const int32_t *num_valid_pages,
                   int init_blocks, int local_blocks, int index_scale, int index_offset,
                   float *out_scores, int32_t *out_ids)
{
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
    if (!ids || index_scale < 1)
        return -1;
    for (int c = 0; c < K; ++c)
        ids[c] = c * index_scale + index_offset;
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < heads; ++h) {
            int64_t row = (int64_t)t * heads + h;
            if (icp_orc_select_pairs(K, ids, scores + row * K, num_valid_pages[t], init_blocks,
                                     local_blocks, out_scores + row * ORC_TOPK,
                                     out_ids + row * ORC_TOPK) < 0) {
                free(ids);
                return -1;
            }
        }
    free(ids);
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Legacy receive rows [SELECT description]                                 */
/* ------------------------------------------------------------------------ */

/* Row index of (t, h) as published by `rank` into the owner h / hpr. */
int64_t icp_orc_recv_row(int slot, int rank, int world_size, int heads_per_rank, int h,
                         int capacity, int t)
{
    return (((int64_t)slot * world_size + rank) * heads_per_rank + h % heads_per_rank) *
               capacity +
           t;
}

/*
 * Publish: Top16 of every row of the float32 plane [T, ws*hpr, K], written
 * as a 33-word legacy row into recv[h / hpr] (host arrays, one per owner):
 * words 0..15 the fp32 bits of the scores, 16..31 the ids, 32 the ready flag
 * set to 1.  A row whose ready flag is not 0 is still occupied; the host
 * oracle has no second agent that could free it, so it counts it as a
 * timed-out wait and leaves the row alone.  Returns the number of such rows,
 * or -1 on a bad argument.
 */
int icp_orc_publish(const float *scores, int T, int K, const int32_t *num_valid_pages,
                    int32_t *const *recv, int slot, int rank, int world_size,
                    int heads_per_rank, int capacity, int force_begin_blocks,
                    int force_end_blocks, int index_scale, int index_offset)
{
    int heads = world_size * heads_per_rank;
    int errors = 0;
    float *sc = NULL;
    int32_t *id = NULL;
    if (T > capacity || slot < 0 || slot > 2 || rank < 0 || rank >= world_size)
        return -1;
    sc = (float *)malloc(sizeof(float) * (size_t)T * heads * ORC_TOPK);
    id = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * heads * ORC_TOPK);
    if (!sc || !id) {
        free(sc);
        free(id);
        return -1;
    }
    if (icp_orc_select(scores, T, heads, K, num_valid_pages, force_begin_blocks,
                       force_end_blocks, index_scale, index_offset, sc, id) != 0) {
        free(sc);
        free(id);
        return -1;
    }
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < heads; ++h) {
            int32_t *row = recv[h / heads_per_rank] +
                           icp_orc_recv_row(slot, rank, world_size, heads_per_rank, h,
                                            capacity, t) *
                               ORC_ROW_WORDS;
            const float *s = sc + ((int64_t)t * heads + h) * ORC_TOPK;
            const int32_t *d = id + ((int64_t)t * heads + h) * ORC_TOPK;
            if (row[32] != 0) {
                errors++;
                continue;
            }
            for (int i = 0; i < ORC_TOPK; ++i) {
                memcpy(&row[i], &s[i], sizeof(float));
                row[ORC_TOPK + i] = d[i];
            }
            row[32] = 1;
        }
    free(sc);
    free(id);
    return errors;
}

/*
 * Owner merge: for every token t and owned head hl, read the world_size
 * source rows of this owner's receive storage `recv`, take the union of
 * their ids (id -1 is padding) with the maximum score per id, and select
 * the Top16 again with num_valid_pages[t].  Each source row that was read
 * gets its flag cleared to 0 (free).  A source whose flag is not 1 is
 * skipped and counted.  Output [T, hpr, 16].  Returns the count of skipped
 * sources, or -1 on a bad argument.
 */
int icp_orc_merge(int32_t *recv, const int32_t *num_valid_pages, int T, int slot, int owner,
                  int world_size, int heads_per_rank, int capacity, int init_blocks,
                  int local_blocks, float *out_scores, int32_t *out_ids)
{
    int missing = 0;
    int32_t ids[4 * ORC_TOPK];
    float sc[4 * ORC_TOPK];
    (void)owner;
    if (world_size < 1 || world_size > 4 || T > capacity || slot < 0 || slot > 2)
        return -1;
    for (int t = 0; t < T; ++t)
        for (int hl = 0; hl < heads_per_rank; ++hl) {
            int n = 0;
            int64_t o = ((int64_t)t * heads_per_rank + hl) * ORC_TOPK;
            for (int s = 0; s < world_size; ++s) {
                int32_t *row = recv + icp_orc_recv_row(slot, s, world_size, heads_per_rank, hl,
                                                       capacity, t) *
                                          ORC_ROW_WORDS;
                if (row[32] != 1) {
                    missing++;
                    continue;
                }
                for (int i = 0; i < ORC_TOPK; ++i) {
                    float v;
                    int32_t d = row[ORC_TOPK + i];
                    int found = -1;
                    memcpy(&v, &row[i], sizeof(float));
                    if (d == -1)
                        continue;
                    for (int e = 0; e < n; ++e)
                        if (ids[e] == d)
                            found = e;
                    if (found < 0) {
                        ids[n] = d;
                        sc[n] = v;
                        n++;
                    } else if (v > sc[found]) {
                        sc[found] = v;
                    }
                }
                row[32] = 0;
            }
            if (icp_orc_select_pairs(n, ids, sc, num_valid_pages[t], init_blocks, local_blocks,
                                     out_scores + o, out_ids + o) < 0)
                return -1;
        }
    return missing;
}

/* ------------------------------------------------------------------------ */
/* Prefill carrier rows                                                     */
/* ------------------------------------------------------------------------ */
/*
 * prepare_msa_icp_indexer's prefill chain hands each rank's local Top16
 * lists to a carrier that the caller exchanges once per layer, then merges
 * what it received (prefill_merge(received, num_valid_pages, output)); the
 * pages that define the carrier are missing.  The reading here: a carrier
 * row is the legacy receive row without its ready flag (the caller's
 * exchange orders it), 32 int32 words: the fp32 bits of the 16 scores, then
 * the 16 ascending ids.  A rank's carrier is [ws][T][hpr][32], block o going
 * to owner o, so row (t, h) sits at ((h / hpr) * T + t) * hpr + h % hpr.
 * After the exchange an owner holds received [ws][T][hpr][32], block s from
 * source rank s.
 */
#define ORC_CARRIER_WORDS 32

/* Carrier of one rank: Top16 of every row of the plane [T, ws*hpr, K].
 * Returns 0 or -1. */
int icp_orc_carrier(const float *scores, int T, int K, const int32_t *num_valid_pages,
                    int world_size, int heads_per_rank, int init_blocks, int local_blocks,
                    int index_scale, int index_offset, int32_t *carrier)
{
    int heads = world_size * heads_per_rank;
    float *sc = NULL;
    int32_t *id = NULL;
    if (T < 0 || world_size < 1 || heads_per_rank < 1)
        return -1;
    sc = (float *)malloc(sizeof(float) * ((size_t)T * heads * ORC_TOPK + 1));
    id = (int32_t *)malloc(sizeof(int32_t) * ((size_t)T * heads * ORC_TOPK + 1));
    if (!sc || !id) {
        free(sc);
        free(id);
        return -1;
    }
    if (icp_orc_select(scores, T, heads, K, num_valid_pages, init_blocks, local_blocks,
                       index_scale, index_offset, sc, id) != 0) {
        free(sc);
        free(id);
        return -1;
    }
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < heads; ++h) {
            int32_t *row = carrier + (((int64_t)(h / heads_per_rank) * T + t) * heads_per_rank +
                                      h % heads_per_rank) *
                                         ORC_CARRIER_WORDS;
            const float *s = sc + ((int64_t)t * heads + h) * ORC_TOPK;
            const int32_t *d = id + ((int64_t)t * heads + h) * ORC_TOPK;
            for (int i = 0; i < ORC_TOPK; ++i) {
                memcpy(&row[i], &s[i], sizeof(float));
                row[ORC_TOPK + i] = d[i];
            }
        }
    free(sc);
    free(id);
    return 0;
}

/* Owner merge of received carrier rows: for every token t and owned head
 * hl, the union of the world_size source lists (id -1 is padding) with the
 * maximum score per id, then Top16 with num_valid_pages[t], as the decode
 * merge.  Output [T, hpr, 16].  Returns 0 or -1. */
int icp_orc_merge_carrier(const int32_t *received, const int32_t *num_valid_pages, int T,
                          int world_size, int heads_per_rank, int init_blocks, int local_blocks,
                          float *out_scores, int32_t *out_ids)
{
    int32_t ids[4 * ORC_TOPK];
    float sc[4 * ORC_TOPK];
    if (T < 0 || world_size < 1 || world_size > 4 || heads_per_rank < 1)
        return -1;
    for (int t = 0; t < T; ++t)
        for (int hl = 0; hl < heads_per_rank; ++hl) {
            int n = 0;
            int64_t o = ((int64_t)t * heads_per_rank + hl) * ORC_TOPK;
            for (int s = 0; s < world_size; ++s) {
                const int32_t *row =
                    received + (((int64_t)s * T + t) * heads_per_rank + hl) * ORC_CARRIER_WORDS;
                for (int i = 0; i < ORC_TOPK; ++i) {
                    float v;
                    int32_t d = row[ORC_TOPK + i];
                    int found = -1;
                    memcpy(&v, &row[i], sizeof(float));
                    if (d == -1)
                        continue;
                    for (int e = 0; e < n; ++e)
                        if (ids[e] == d)
                            found = e;
                    if (found < 0) {
                        ids[n] = d;
                        sc[n] = v;
                        n++;
                    } else if (v > sc[found]) {
                        sc[found] = v;
                    }
                }
            }
            if (icp_orc_select_pairs(n, ids, sc, num_valid_pages[t], init_blocks, local_blocks,
                                     out_scores + o, out_ids + o) < 0)
                return -1;
        }
    return 0;
}

/* ------------------------------------------------------------------------ */
/* Tagged receive rows [SELECT description, parameter generations]          */
/* ------------------------------------------------------------------------ */
/*
 * A tagged row is 32 int64 words, word i = (generation << 32) | payload_i,
 * payload 0..15 the fp32 bits of the scores and 16..31 the ids (the legacy
 * row without its ready flag).  Readings where the pages are silent:
 *   - the publisher keeps counters generations[slot][h][t] (int32
 *     [3, ws*hpr, capacity], zeroed once) and publishes row (t, h) with
 *     generation = counter + 1, storing the new value back;
 *   - the owner keeps expected counters expected[slot][src][hl][t] (int32
 *     [3, ws, hpr, capacity], zeroed once); a merge of slot `slot` takes a
 *     source row as arrived when all 32 words carry expected + 1, and the
 *     counter advances on every merge, arrived or not;
 *   - nothing waits for a free row: the pages instead ask for two or more
 *     sparse layers between two uses of one slot set.
 */
int icp_orc_publish_tagged(const float *scores, int T, int K, const int32_t *num_valid_pages,
                           int64_t *const *recv, int32_t *generations, int slot, int rank,
                           int world_size, int heads_per_rank, int capacity,
                           int force_begin_blocks, int force_end_blocks, int index_scale,
                           int index_offset)
{
    int heads = world_size * heads_per_rank;
    float *sc = NULL;
    int32_t *id = NULL;
    if (T > capacity || slot < 0 || slot > 2 || rank < 0 || rank >= world_size)
        return -1;
    sc = (float *)malloc(sizeof(float) * (size_t)T * heads * ORC_TOPK);
    id = (int32_t *)malloc(sizeof(int32_t) * (size_t)T * heads * ORC_TOPK);
    if (!sc || !id) {
        free(sc);
        free(id);
        return -1;
    }
    if (icp_orc_select(scores, T, heads, K, num_valid_pages, force_begin_blocks,
                       force_end_blocks, index_scale, index_offset, sc, id) != 0) {
        free(sc);
        free(id);
        return -1;
    }
    for (int t = 0; t < T; ++t)
        for (int h = 0; h < heads; ++h) {
            int32_t *gen = generations + ((int64_t)slot * heads + h) * capacity + t;
            uint32_t g = (uint32_t)(*gen) + 1u;
            int64_t *row = recv[h / heads_per_rank] +
                           icp_orc_recv_row(slot, rank, world_size, heads_per_rank, h,
                                            capacity, t) *
                               32;
            for (int i = 0; i < 32; ++i) {
                uint32_t payload;
                if (i < ORC_TOPK)
                    memcpy(&payload, &sc[((int64_t)t * heads + h) * ORC_TOPK + i], 4);
                else
                    payload = (uint32_t)id[((int64_t)t * heads + h) * ORC_TOPK + i - ORC_TOPK];
                row[i] = (int64_t)(((uint64_t)g << 32) | payload);
            }
            *gen = (int32_t)g;
        }
    free(sc);
    free(id);
    return 0;
}

int icp_orc_merge_tagged(const int64_t *recv, int32_t *expected, const int32_t *num_valid_pages,
                         int T, int slot, int world_size, int heads_per_rank, int capacity,
                         int init_blocks, int local_blocks, float *out_scores, int32_t *out_ids)
{
    int missing = 0;
    int32_t ids[4 * ORC_TOPK];
    float sc[4 * ORC_TOPK];
    if (world_size < 1 || world_size > 4 || T > capacity || slot < 0 || slot > 2)
        return -1;
    for (int t = 0; t < T; ++t)
        for (int hl = 0; hl < heads_per_rank; ++hl) {
            int n = 0;
            int64_t o = ((int64_t)t * heads_per_rank + hl) * ORC_TOPK;
            for (int s = 0; s < world_size; ++s) {
                int32_t *e = expected +
                             (((int64_t)slot * world_size + s) * heads_per_rank + hl) * capacity + t;
                uint32_t want = (uint32_t)(*e) + 1u;
                const int64_t *row = recv + icp_orc_recv_row(slot, s, world_size, heads_per_rank,
                                                             hl, capacity, t) *
                                                32;
                int arrived = 1;
                *e = (int32_t)want;
                for (int i = 0; i < 32; ++i)
                    if ((uint32_t)((uint64_t)row[i] >> 32) != want)
                        arrived = 0;
                if (!arrived) {
                    missing++;
                    continue;
                }
                for (int i = 0; i < ORC_TOPK; ++i) {
                    float v;
                    uint32_t pb = (uint32_t)((uint64_t)row[i] & 0xFFFFFFFFu);
                    int32_t d = (int32_t)(uint32_t)((uint64_t)row[ORC_TOPK + i] & 0xFFFFFFFFu);
                    int found = -1;
                    memcpy(&v, &pb, 4);
                    if (d == -1)
                        continue;
                    for (int q = 0; q < n; ++q)
                        if (ids[q] == d)
                            found = q;
                    if (found < 0) {
                        ids[n] = d;
                        sc[n] = v;
                        n++;
                    } else if (v > sc[found]) {
                        sc[found] = v;
                    }
                }
            }
            if (icp_orc_select_pairs(n, ids, sc, num_valid_pages[t], init_blocks, local_blocks,
                                     out_scores + o, out_ids + o) < 0)
                return -1;
        }
    return missing;
}
