// icp_internal.h - host-side declarations shared by the library's .cu files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace icp {

// Geometry of one scoring call, derived on the host from the layout
// arguments of msa_icp_decode_index_score_sharded.
struct ScoreGeom {
  int rows_per_page;  // K rows of one page held by this rank: page_size / world_size
  int R;              // K rows feeding one plane column (32, 64 or 128)
  int cpt;            // plane columns per 128-row MMA tile: 128 / R
  int split;          // 1 when a column is one half of a 256-row page (P256, world_size 1)
  int nq;             // query rows staged per request: 32 (4 * dql of them are used)
};

// The fused scorer + select covers at most this many CTAs (workspace sizing).
constexpr int kFusedMaxGrid = 160;
// Largest batch a scoring launch accepts (shared-memory sizing).
constexpr int kMaxBatchDevice = 4096;

struct ScoreArgs {
  const int32_t *block_table;
  int64_t bt_stride;
  const int32_t *seq_lens;
  float *score_out;  // plane (icp_score only)
  int32_t *errors;
  int batch, cols, rank, world_size, page_size, dql;
  int num_pages;  // pages of the index-K shard: valid block-table entries are below it
  ScoreGeom g;
  int pdl;  // launched with programmatic dependent launch (early start)
  // fused scorer + select only
  const int32_t *nvp;
  int init_blocks, local_blocks, index_scale, index_offset;
  float *out_scores;
  int32_t *out_ids;
  int32_t *ws_counters;  // [batch] 16-byte records: where each request's lists are
  void *ws_records;      // partial Top16 lists
  // prefill window: requests come from a plan of kPlanRecordInts-int records
  // (see icp_prefill.cu) instead of seq_lens / dql; batch is then the plan's
  // capacity and *vcount the records in use
  const int32_t *vreq;
  const int32_t *vcount;
  int wide;  // prefill scorer: 256 distinct query rows per request (records of <= 64 tokens)
};

// Prefill plan: word 0 = records in use; records from word kPlanHeaderInts,
// kPlanRecordInts ints each: {first token, block-table row, seq_len seen by
// the record's tokens (last position + 1), tokens (<= 32), the request's
// seq_len, 0, 0, 0}.
constexpr int kPlanHeaderInts = 8;
constexpr int kPlanRecordInts = 8;
constexpr int kPlanTokens = 64;  // tokens per record: 4 * 64 = 256 query rows, two MMA row halves

struct SelectArgs {
  const float *scores;
  int T, K;
  const int32_t *nvp;
  int init_blocks, local_blocks, index_scale, index_offset;
  // plain output
  float *out_scores;
  int32_t *out_ids;
  // publish
  const int64_t *recv_bases;
  int32_t *errors;
  int slot, rank, world_size, heads_per_rank, capacity;
  long long spin_limit;
  int32_t *generations;  // tagged publish: [3][ws * hpr][capacity] counters
  int32_t *carrier;      // prefill carrier rows [ws][T][hpr][32]
  int pdl;               // launched with programmatic dependent launch
};

struct MergeArgs {
  int32_t *recv;
  const int32_t *nvp;
  int T, slot, world_size, heads_per_rank, capacity, init_blocks, local_blocks;
  long long spin_limit;
  int32_t *errors;
  float *out_scores;
  int32_t *out_ids;
  const unsigned long long *recv64;  // tagged merge: this owner's tagged rows
  int32_t *expected;                 // tagged merge: [3][ws][hpr][capacity] counters
  const int32_t *received;           // prefill merge: carrier rows [ws][T][hpr][32]
  int pdl;                           // launched with programmatic dependent launch
};

// Launchers (return a cudaError_t from the launch).
cudaError_t launch_score(const CUtensorMap &tmk, const CUtensorMap &tmq, const ScoreArgs &a,
                         int grid, cudaStream_t stream);
size_t score_smem_bytes(int batch);
cudaError_t score_prepare(int device);  // one-time per-device kernel attributes

size_t fused_workspace_bytes(int batch, int dql);
cudaError_t launch_fused_merge(const ScoreArgs &a, int grid_a, cudaStream_t stream);
cudaError_t launch_score_select(const CUtensorMap &tmk, const CUtensorMap &tmq, ScoreArgs a,
                                int grid, cudaStream_t stream);

cudaError_t select_prepare();  // one-time per-device kernel attributes
// mode: 0 plain output, 1 legacy receive rows, 2 tagged receive rows,
// 3 prefill carrier rows
cudaError_t launch_select(const SelectArgs &a, int mode, int sm_count, cudaStream_t stream);
cudaError_t launch_merge(const MergeArgs &a, bool tagged, cudaStream_t stream);
cudaError_t launch_merge_carrier(const MergeArgs &a, cudaStream_t stream);

// Prefill plan of a window (one CTA): records for `batch` requests into plan
// (room for `capacity` records); a request with a bad chunk adds 1 to errors.
cudaError_t launch_prefill_plan(const int32_t *qo_indptr, const int32_t *seq_lens, int batch,
                                int T, int32_t *plan, int capacity, int32_t *errors,
                                cudaStream_t stream);

}  // namespace icp
