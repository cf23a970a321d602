/*
 * icp.h - C ABI of the GB300 (sm_103a) decode-time ICP block indexer.
 *
 * The operations are the ones documented by FlashInfer's experimental
 * MiniMax-M3 ICP indexer API pages (flashinfer.msa_ops):
 *   msa_icp_decode_index_score_sharded  -> icp_score
 *   msa_icp_topk_select_publish         -> icp_top16_select (select only) and
 *                                          icp_publish_rows (select + legacy receive rows)
 *   prepare_msa_icp_indexer, decode()   -> icp_merge (owner merge of the chain
 *                                          whose steps are score plane, Top16 select and
 *                                          publish, owner merge)
 *                                          and icp_score_select (fused scorer + select)
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller, on the
 *     current CUDA device; the library never frees or keeps them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default stream).
 *     Calls only enqueue work: they allocate nothing and never synchronize,
 *     so they may be recorded into a CUDA graph.
 *   - fp8 tensors are float8_e4m3fn bit patterns passed as uint8_t; no scale.
 *   - Return value: ICP_OK, or ICP_ERR_INVALID_ARG when a host-side check
 *     fails (nothing is launched), ICP_ERR_UNSUPPORTED when the current device
 *     is not an sm_103 GPU, ICP_ERR_CUDA when a CUDA call or launch fails.
 *   - Device-side waits are bounded; a wait that runs out adds 1 to errors[0]
 *     (when `errors` is not NULL) and the kernel returns without trapping.
 *     The caller reads errors[0] after its own synchronization; a non-zero
 *     count maps to ICP_ERR_TIMEOUT, a status no entry point returns itself
 *     (none of them waits for the device).
 */
#ifndef ICP_H
#define ICP_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define ICP_OK 0
#define ICP_ERR_INVALID_ARG 1
#define ICP_ERR_CUDA 2
#define ICP_ERR_UNSUPPORTED 3
#define ICP_ERR_TIMEOUT 4  /* for callers: errors[0] > 0 after their own sync */

#define ICP_HEADS 4        /* index heads (prepare_msa_icp_indexer: num_index_heads must be 4) */
#define ICP_DIM 128        /* fp8 values per index query / key row */
#define ICP_TOPK 16        /* blocks kept per (token, head) row */
#define ICP_ROW_WORDS 33   /* legacy receive row: 16 scores, 16 ids, ready flag */
#define ICP_MAX_COLS 8192  /* msa_icp_decode_index_score_sharded: 0 < cols <= 8192 */
#define ICP_MAX_K 12287    /* msa_icp_topk_select_publish: 0 < K < 12288 */
#define ICP_MAX_BATCH 4096 /* requests per icp_score / icp_score_select call */

/* Human-readable name of a status code (static string). */
const char *icp_status_string(int status);

/*
 * Plane width for the longest request (msa_icp_decode_index_score_sharded,
 * parameter score_out, which defers to msa_icp_decode_score_columns()):
 * the number of columns of a request of max_seq_len tokens, padded to the
 * next multiple of 4.  A column is a global B128 block at page_size 128, a
 * local page at page_size 256 with world_size 2 or 4, and a B128 block at
 * page_size 256 with world_size 1.  Returns the width, or -1 when the
 * arguments are invalid or the width would exceed ICP_MAX_COLS.  Host only.
 */
int icp_score_columns(int max_seq_len, int page_size, int world_size);

/*
 * Decode index scores (msa_icp_decode_index_score_sharded).
 *   index_q      [batch * decode_query_len, 4, 128] fp8, contiguous, 16-byte aligned;
 *                token j of request b is row b * decode_query_len + j and sits at
 *                position seq_lens[b] - decode_query_len + j.
 *   index_k      [num_pages, page_size / world_size, 128] fp8 shard, contiguous,
 *                16-byte aligned; this rank holds rows
 *                [rank * page_size / world_size, (rank + 1) * page_size / world_size)
 *                of every page.
 *   block_table  int32 [batch, >= ceil(seq_len / page_size)], unit last stride,
 *                row stride block_table_stride (elements); entries must lie in
 *                [0, num_pages).  An entry outside is read as a page of zero
 *                keys, and every request whose pages hold such an entry adds 1
 *                to errors[0] (once per request and call, when errors is not
 *                NULL).
 *   seq_lens     int32 [batch].
 *   score_out    float32 [batch * decode_query_len, 4, cols], contiguous.  For
 *                each request only columns c < round_up(n, 4) are written, n
 *                being the request's column count (see icp_score_columns); the
 *                other columns are not touched.  Written value: the maximum over
 *                the column's keys at positions <= the token's position of the
 *                fp32 dot product of the 128 dequantised values, -inf when no
 *                key is visible.
 *   Limits: 0 < cols <= 8192, cols % 4 == 0; page_size 128 or 256; world_size
 *   1, 2 or 4 (1 is an extension of the documented 2 or 4); 0 <= rank <
 *   world_size; 1 <= decode_query_len <= max_decode_query_len,
 *   4 * max_decode_query_len <= 32; 0 <= batch <= ICP_MAX_BATCH.
 *   enable_pdl (parameter enable_pdl of the same page): non-zero launches with
 *   programmatic dependent launch.  Ahead of its griddepcontrol.wait the
 *   kernel only sets itself up (barriers, tensor memory, and the split of
 *   the work, read from seq_lens); no other load and no store precedes the
 *   wait.  The caller guarantees that the kernel queued just ahead leaves
 *   seq_lens alone, and that it is either an ordinary launch or one that
 *   waits for its own predecessor before it signals its dependents.
 *   0 removes the requirement.
 *   errors: optional int32 [>= 1] counter of timed-out internal waits,
 *           requests with block-table entries outside the pool, and requests
 *           wider than the plane.
 */
int icp_score(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
              const int32_t *block_table, int64_t block_table_stride, const int32_t *seq_lens,
              float *score_out, int batch, int cols, int rank, int world_size, int page_size,
              int decode_query_len, int max_decode_query_len, int enable_pdl, int32_t *errors,
              void *stream);

/*
 * Top16 select of every (token, head) row of a score plane (the selection
 * half of msa_icp_topk_select_publish, written to plain output arrays).
 *   scores           float32 [T, 4, K], contiguous, 0 < K <= 12287.
 *   num_valid_pages  int32 [T]: global B128 block count of each token.
 *   Column c carries global id c * index_scale + index_offset (index_scale
 *   >= 1, index_offset >= 0); valid ids are those below num_valid_pages[t].
 *   If num_valid_pages[t] <= 16 every valid id is kept.  Otherwise the ids
 *   in [0, init_blocks) and [nvp - local_blocks, nvp) are forced and the
 *   remaining slots take the best other valid ids by (score descending, id
 *   ascending).  init_blocks + local_blocks <= 16.
 *   out_scores float32 [T, 4, 16], out_ids int32 [T, 4, 16]: ids ascending,
 *   each with its raw score, then padding id -1 / score -inf.  Every row is
 *   written.
 */
int icp_top16_select(const float *scores, int T, int K, const int32_t *num_valid_pages,
                     int init_blocks, int local_blocks, int index_scale, int index_offset,
                     float *out_scores, int32_t *out_ids, void *stream);

/*
 * Top16 select and publish into legacy receive rows
 * (msa_icp_topk_select_publish, legacy mode).
 *   scores [T, world_size * heads_per_rank, K] (world_size * heads_per_rank
 *   must be 4), num_valid_pages, index_scale, index_offset,
 *   force_begin_blocks / force_end_blocks: as icp_top16_select.
 *   recv_bases  int64 [world_size] DEVICE array of device addresses: the
 *               receive storage of every owner rank, each int32
 *               [3][world_size][heads_per_rank][capacity][33] (row-major) and
 *               8-byte aligned.  On one GPU these are ws buffers of the device.
 *   Row (t, h) goes to owner h / heads_per_rank, row
 *   ((slot * world_size + rank) * heads_per_rank + h % heads_per_rank) * capacity + t:
 *   words 0-15 the fp32 bits of the scores, 16-31 the ascending ids, word 32
 *   the ready flag.  Before writing, the kernel polls the flag (acquire) until
 *   it reads 0 (free), at most spin_limit polls and at most about two seconds;
 *   it then stores the 32 data words and release-stores flag = 1.  A row
 *   whose wait runs out is skipped and adds 1 to errors[0] (no trap).
 *   Every row t < T, padding rows included, is written on every call.
 *   Limits: slot 0..2; world_size 1, 2 or 4; 0 <= rank < world_size;
 *   1 <= T <= capacity; spin_limit >= 1.  errors: int32 [>= 1], required.
 *   enable_pdl (msa_icp_topk_select_publish, enable_pdl): launch with
 *   programmatic dependent launch.  The kernel waits on the preceding
 *   kernel (griddepcontrol.wait) before it reads anything, and only then
 *   lets its own dependents launch, so it may follow a scorer launched with
 *   or without it.  0 launches it as an ordinary kernel.
 */
int icp_publish_rows(const float *scores, int T, int K, const int32_t *num_valid_pages,
                     const int64_t *recv_bases, int32_t *errors, int slot, int rank,
                     int world_size, int heads_per_rank, int capacity, int force_begin_blocks,
                     int force_end_blocks, int64_t spin_limit, int index_scale,
                     int index_offset, int enable_pdl, void *stream);

/*
 * Owner merge of the decode chain (prepare_msa_icp_indexer, decode(): the
 * score plane, then the Top16 select and publish, then this merge; the rule is
 * this library's reading: union of the world_size published lists, maximum
 * score per id, then the icp_top16_select rule with num_valid_pages[t]).
 *   recv   this owner's receive storage, int32 [3][world_size][heads_per_rank][capacity][33].
 *   For each token t < T and owned head hl < heads_per_rank it waits (acquire,
 *   at most spin_limit polls / about two seconds) for the flag of each source
 *   row of slot `slot` to read 1, merges, and then clears the flags it read
 *   back to 0 (rows free).  A source whose wait runs out is left out of the
 *   merge and adds 1 to errors[0].
 *   out_scores float32 [T, heads_per_rank, 16], out_ids int32 [T, heads_per_rank, 16].
 *   Limits as icp_publish_rows.  errors: required.
 *   enable_pdl: launch with programmatic dependent launch.  The kernel waits
 *   on the preceding kernel (griddepcontrol.wait) before it reads anything,
 *   and only then lets its own dependents launch.  0 launches it as an
 *   ordinary kernel.
 */
int icp_merge(int32_t *recv, const int32_t *num_valid_pages, int T, int slot, int world_size,
              int heads_per_rank, int capacity, int init_blocks, int local_blocks,
              int64_t spin_limit, int32_t *errors, float *out_scores, int32_t *out_ids,
              int enable_pdl, void *stream);

/*
 * Tagged publish (msa_icp_topk_select_publish with `generations`: tagged
 * mode).  The same Top16 select as icp_publish_rows; row (t, h) goes to owner
 * h / heads_per_rank at the same row index, as 32 int64 words
 * (generation << 32) | word, word 0-15 the fp32 bits of the scores and
 * 16-31 the ascending ids.
 *   recv_bases   int64 [world_size] DEVICE array of device addresses of each
 *                owner's tagged storage, int64 [3][world_size][hpr][capacity][32],
 *                8-byte aligned.
 *   generations  int32 [3, world_size * heads_per_rank, capacity] DEVICE
 *                publish counters of this rank, zeroed once by the caller and
 *                never between steps: row (t, h) of slot s is published with
 *                generation generations[s][h][t] + 1, which is stored back.
 *   Nothing waits for a free row: instead the page has the caller leave two
 *   or more sparse layers between two uses of the same slot set.  Every row t < T,
 *   padding rows included, is written on every call.  Limits and
 *   enable_pdl as icp_publish_rows (no spin_limit, no errors).
 */
int icp_publish_rows_tagged(const float *scores, int T, int K, const int32_t *num_valid_pages,
                            const int64_t *recv_bases, int32_t *generations, int slot, int rank,
                            int world_size, int heads_per_rank, int capacity,
                            int force_begin_blocks, int force_end_blocks, int index_scale,
                            int index_offset, int enable_pdl, void *stream);

/*
 * Owner merge of tagged rows (this library's reading; the counters of the
 * receiving side are described on a page the documentation does not carry).
 *   recv      this owner's tagged storage, int64 [3][world_size][hpr][capacity][32].
 *   expected  int32 [3][world_size][hpr][capacity] DEVICE counters of this owner,
 *             zeroed once.  A merge of slot s takes the source row of rank r
 *             as arrived when all 32 words carry generation expected + 1; the
 *             counter advances on every merge.  Each wait is bounded by
 *             spin_limit polls and about two seconds; a source that has not
 *             arrived is left out and adds 1 to errors[0].
 *   Output, rule and enable_pdl as icp_merge.  Rows are not modified (no
 *   flags to free).
 */
int icp_merge_tagged(const int64_t *recv, int32_t *expected, const int32_t *num_valid_pages,
                     int T, int slot, int world_size, int heads_per_rank, int capacity,
                     int init_blocks, int local_blocks, int64_t spin_limit, int32_t *errors,
                     float *out_scores, int32_t *out_ids, int enable_pdl, void *stream);

/*
 * Workspace bytes icp_score_select needs for `batch` requests of
 * decode_query_len tokens (per-request partial Top16 lists and counters).
 * Returns 0 for invalid arguments.  Host only.
 */
size_t icp_score_select_workspace_bytes(int batch, int decode_query_len);

/*
 * Fused scorer + Top16 select (the fused decode chain of
 * prepare_msa_icp_indexer, decode(pool=...), whose scorer feeds the select
 * directly and leaves no score plane).  Arguments as icp_score plus
 * num_valid_pages / init_blocks / local_blocks as icp_top16_select (global
 * id of column c = c * index_scale + index_offset, with index_scale 2 and
 * index_offset rank * 2 / world_size for page_size 256 with world_size 2 or 4,
 * else 1 and 0).  The output equals icp_score followed by icp_top16_select
 * on a plane of width cols, bit for bit, whenever num_valid_pages[t] does not
 * exceed the number of B128 blocks of the token's request (as in decode,
 * where it counts the blocks holding visible keys); ids beyond the request's
 * columns are treated as absent.
 *   workspace  device buffer of icp_score_select_workspace_bytes(batch, dql)
 *              bytes, 256-byte aligned; its contents need no initialisation
 *              and are scratch between calls.  Calls that share a workspace
 *              must not overlap on the GPU.
 *   out_scores float32 [batch * dql, 4, 16], out_ids int32 [batch * dql, 4, 16].
 */
int icp_score_select(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
                     const int32_t *block_table, int64_t block_table_stride,
                     const int32_t *seq_lens, int batch, int cols, int rank, int world_size,
                     int page_size, int decode_query_len, int max_decode_query_len,
                     const int32_t *num_valid_pages, int init_blocks, int local_blocks,
                     void *workspace, size_t workspace_bytes, float *out_scores,
                     int32_t *out_ids, int32_t *errors, void *stream);

/*
 * icp_score_select for callers that cannot allocate device memory when they
 * call: a serving engine that splits the GPU into fixed pools at start-up and
 * allows no later allocation, a decode step being recorded into a CUDA graph,
 * or a latency-critical path that cannot pay for cudaMalloc's implicit
 * synchronisation.  The pages document no counterpart of this entry point.
 *
 * Arguments, output and behaviour are those of icp_score_select without the
 * workspace: the scratch is a fixed array of ICP_NOALLOC_SCRATCH_BYTES held
 * by every GPU that loads this library until the process exits.  Nothing is
 * allocated or freed by the call.
 *   - Limit: accepted when icp_score_select_workspace_bytes(batch,
 *     decode_query_len) <= ICP_NOALLOC_SCRATCH_BYTES, which allows at most
 *     1654, 748, 446, 294, 203, 143, 100 or 67 requests at decode_query_len
 *     1 to 8; a larger batch returns ICP_ERR_INVALID_ARG and launches
 *     nothing.
 *   - The first call on each device looks up the array's device address
 *     (cudaGetSymbolAddress, with that device current); make that first call
 *     before any stream capture begins.  The address is kept for the life of
 *     the process and belongs to the device's primary context, the one the
 *     CUDA runtime uses: after cudaDeviceReset, or from another context on
 *     that device, it is stale, so such a caller must not use this entry
 *     point.
 *   - All calls on a device share the array and it keeps what the last call
 *     left; no part of it needs clearing, but calls that overlap on the GPU
 *     race on it, so the caller must not run two at once.
 */
#define ICP_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)
int icp_score_select_noalloc(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
                             const int32_t *block_table, int64_t block_table_stride,
                             const int32_t *seq_lens, int batch, int cols, int rank,
                             int world_size, int page_size, int decode_query_len,
                             int max_decode_query_len, const int32_t *num_valid_pages,
                             int init_blocks, int local_blocks, float *out_scores,
                             int32_t *out_ids, int32_t *errors, void *stream);

/*
 * Prefill window (prepare_msa_icp_indexer: one prefill_window_plan for each
 * window of queries in a step, prefill_local per query chunk, the caller's one
 * exchange per layer, then prefill_merge(received, num_valid_pages,
 * output)).  The pages that define these calls are missing; the reading
 * taken:
 *   - a window holds, for every request b, a chunk of its newest
 *     n_b = qo_indptr[b+1] - qo_indptr[b] tokens: window tokens
 *     qo_indptr[b] .. qo_indptr[b+1] - 1, token j at position
 *     seq_len_b - n_b + j (the decode placement of msa_icp_decode_index_
 *     score_sharded's index_q with a per-request query length);
 *   - the window's score plane is the decode plane of those queries: every
 *     token gets its request's columns (icp_score_columns of seq_len_b),
 *     -inf where no key at or before its position exists;
 *   - local Top16 lists go into carrier rows: the legacy receive row
 *     without its ready flag, 32 int32 words (fp32 bits of the 16 scores,
 *     then the 16 ascending ids), a rank's carrier int32
 *     [world_size][T][heads_per_rank][32] with block o bound for owner o
 *     (row (t, h) at ((h / hpr) * T + t) * hpr + h % hpr);
 *   - after the caller's exchange, an owner holds received
 *     [world_size][T][heads_per_rank][32] (block s from rank s) and merges
 *     it with the decode merge rule (union, maximum score per id, Top16 with
 *     num_valid_pages[t]).
 */

/*
 * int32 words of a prefill plan for a window of T tokens from `batch`
 * requests: room for ceil(T / 64) + batch records of 8 ints plus an 8-int
 * header.  Returns -1 when batch or T is negative or the records would
 * exceed ICP_MAX_BATCH.  Host only.
 */
int64_t icp_prefill_plan_words(int batch, int T);

/*
 * prefill_window_plan: cuts every request's chunk into records of at most 64
 * consecutive tokens, 256 query rows each (one kernel, no host
 * synchronisation).
 *   qo_indptr int32 [batch + 1], seq_lens int32 [batch] (each request's
 *   length after the window's tokens), both device memory.
 *   plan      int32 [plan_words] device memory, 16-byte aligned, written
 *             by the call; plan_words >= icp_prefill_plan_words(batch, T).
 *   errors    int32 [>= 1] or NULL: a request whose chunk is invalid (a
 *             decreasing qo_indptr, outside [0, T], or longer than its
 *             seq_len) gets no records and adds 1; its tokens' plane rows
 *             are then not written.
 */
int icp_prefill_plan(const int32_t *qo_indptr, const int32_t *seq_lens, int batch, int T,
                     int32_t *plan, int64_t plan_words, int32_t *errors, void *stream);

/*
 * prefill_local, scoring half: the window's score plane float32
 * [T, 4, cols] (unit last stride) from index_q uint8 [T, 4, 128] (the
 * window's tokens, 16-byte aligned) against the rank's index-K shard, as
 * icp_score does for decode (same index_k, block_table, cols, rank,
 * world_size and page_size rules).  `plan` is icp_prefill_plan's output for
 * this window.  Columns a token's request does not reach are left
 * untouched; errors (or NULL) counts a plane narrower than a request needs
 * and bounded waits that ran out.
 */
int icp_prefill_score(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
                      const int32_t *block_table, int64_t block_table_stride,
                      const int32_t *plan, int64_t plan_words, float *score_out, int T,
                      int cols, int rank, int world_size, int page_size, int32_t *errors,
                      void *stream);

/*
 * prefill_local, list half: the Top16 of every row of the plane float32
 * [T, world_size * heads_per_rank, K] (the icp_top16_select rule, with
 * num_valid_pages int32 [T]) into this rank's carrier int32
 * [world_size][T][heads_per_rank][32].  Every row is written.  Limits as
 * icp_top16_select; world_size 1, 2 or 4 and world_size * heads_per_rank = 4.
 */
int icp_prefill_select(const float *scores, int T, int K, const int32_t *num_valid_pages,
                       int world_size, int heads_per_rank, int init_blocks, int local_blocks,
                       int index_scale, int index_offset, int32_t *carrier, void *stream);

/*
 * prefill_merge: an owner's Top16 per (token, owned head) from the received
 * carrier rows int32 [world_size][T][heads_per_rank][32] (all present: the
 * caller's exchange has completed), out_scores float32 / out_ids int32
 * [T, heads_per_rank, 16], ids ascending, (-1, -inf) padding.
 */
int icp_prefill_merge(const int32_t *received, const int32_t *num_valid_pages, int T,
                      int world_size, int heads_per_rank, int init_blocks, int local_blocks,
                      float *out_scores, int32_t *out_ids, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* ICP_H */
