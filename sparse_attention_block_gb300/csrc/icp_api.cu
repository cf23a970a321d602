// icp_api.cu - the extern "C" entry points declared in include/icp.h.
//
// Host side only: argument checks (limits from the msa_icp_* API pages),
// TMA descriptor encoding, one-time per-device set-up, and kernel launches.
// Nothing here allocates device memory or synchronizes.
#include <cudaTypedefs.h>
#include <mutex>
#include <stdint.h>
#include <string.h>

#include "icp.h"
#include "icp_internal.h"

namespace {

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int status = ICP_OK;
  int sm_count = 0;
};

std::mutex g_mutex;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

// Current device, checked to be an sm_103 part, with one-time set-up done.
int current_device(int *dev_out, int *sm_count) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ICP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ICP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mutex);
  DeviceInfo &d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return ICP_ERR_CUDA;
    if (major != 10 || minor != 3) {
      d.status = ICP_ERR_UNSUPPORTED;
    } else if (icp::score_prepare(dev) != cudaSuccess || icp::select_prepare() != cudaSuccess) {
      d.status = ICP_ERR_CUDA;
    } else {
      d.status = ICP_OK;
    }
    if (!g_encode && d.status == ICP_OK) {
      void *fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                           cudaEnableDefault, &q) != cudaSuccess ||
          q != cudaDriverEntryPointSuccess || !fn)
        d.status = ICP_ERR_CUDA;
      else
        g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    }
    d.ready = true;
  }
  *dev_out = dev;
  *sm_count = d.sm_count;
  return d.status;
}

// 2D uint8 tensor map over [rows, 128] bytes with a {128, box_rows} box and
// the 128-byte swizzle (the layout the MMA descriptors expect).
int encode_rows(CUtensorMap *map, const void *base, uint64_t rows, uint32_t box_rows) {
  cuuint64_t dims[2] = {128, rows};
  cuuint64_t strides[1] = {128};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  CUresult r = g_encode(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? ICP_OK : ICP_ERR_CUDA;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

int units_for(int seq_len, int page_size, int world_size) {
  const int u = (page_size == 256 && world_size == 1) ? 128 : page_size;
  return seq_len <= 0 ? 0 : (int)(((long long)seq_len + u - 1) / u);
}

// Checks shared by icp_score (and the fused scorer).
int check_score_args(const uint8_t *q, const uint8_t *k, int64_t num_pages, const int32_t *bt,
                     int64_t bt_stride, const int32_t *seq_lens, int batch, int cols, int rank,
                     int ws, int ps, int dql, int maxdql) {
  if (batch < 0 || batch > ICP_MAX_BATCH) return ICP_ERR_INVALID_ARG;
  if (cols <= 0 || cols > ICP_MAX_COLS || cols % 4 != 0) return ICP_ERR_INVALID_ARG;
  if (ps != 128 && ps != 256) return ICP_ERR_INVALID_ARG;
  if (ws != 1 && ws != 2 && ws != 4) return ICP_ERR_INVALID_ARG;
  if (rank < 0 || rank >= ws) return ICP_ERR_INVALID_ARG;
  if (dql < 1 || dql > maxdql || 4 * maxdql > 32) return ICP_ERR_INVALID_ARG;
  if (batch == 0) return ICP_OK;
  if (!q || !k || !bt || !seq_lens) return ICP_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k)) return ICP_ERR_INVALID_ARG;
  if (num_pages <= 0 || bt_stride < 1) return ICP_ERR_INVALID_ARG;
  if ((uint64_t)num_pages * (uint64_t)(ps / ws) >= (1ull << 31)) return ICP_ERR_INVALID_ARG;
  return ICP_OK;
}

icp::ScoreGeom make_geom(int ps, int ws, int dql) {
  icp::ScoreGeom g;
  g.rows_per_page = ps / ws;
  g.split = (ps == 256 && ws == 1) ? 1 : 0;
  g.R = g.split ? 128 : g.rows_per_page;
  g.cpt = 128 / g.R;
  g.nq = 32;  // query rows staged per request (4 * dql <= 32), one TMA box
  (void)dql;
  return g;
}

int to_status(cudaError_t e) { return e == cudaSuccess ? ICP_OK : ICP_ERR_CUDA; }

bool valid_select_common(int T, int K, int init, int local, int scale, int offset) {
  if (T < 0 || K <= 0 || K > ICP_MAX_K) return false;
  if (init < 0 || local < 0 || init + local > ICP_TOPK) return false;
  if (scale < 1 || offset < 0) return false;
  if ((long long)(K - 1) * scale + offset > 0x7FFFFFF0LL) return false;
  return true;
}

}  // namespace

extern "C" {

const char *icp_status_string(int status) {
  switch (status) {
    case ICP_OK: return "ok";
    case ICP_ERR_INVALID_ARG: return "invalid argument";
    case ICP_ERR_CUDA: return "CUDA error";
    case ICP_ERR_UNSUPPORTED: return "unsupported device (needs sm_103)";
    case ICP_ERR_TIMEOUT: return "a bounded device wait timed out (errors > 0)";
    default: return "unknown status";
  }
}

int icp_score_columns(int max_seq_len, int page_size, int world_size) {
  if (max_seq_len < 0) return -1;
  if (page_size != 128 && page_size != 256) return -1;
  if (world_size != 1 && world_size != 2 && world_size != 4) return -1;
  const int u = units_for(max_seq_len, page_size, world_size);
  const int cols = (u + 3) / 4 * 4;
  if (cols > ICP_MAX_COLS) return -1;
  return cols < 4 ? 4 : cols;
}

int icp_score(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
              const int32_t *block_table, int64_t block_table_stride, const int32_t *seq_lens,
              float *score_out, int batch, int cols, int rank, int world_size, int page_size,
              int decode_query_len, int max_decode_query_len, int enable_pdl, int32_t *errors,
              void *stream) {
  int st = check_score_args(index_q, index_k, num_pages, block_table, block_table_stride,
                            seq_lens, batch, cols, rank, world_size, page_size, decode_query_len,
                            max_decode_query_len);
  if (st != ICP_OK) return st;
  if (batch == 0) return ICP_OK;
  if (!score_out) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;

  icp::ScoreArgs a;
  memset(&a, 0, sizeof(a));
  a.block_table = block_table;
  a.bt_stride = block_table_stride;
  a.num_pages = (int)num_pages;
  a.seq_lens = seq_lens;
  a.score_out = score_out;
  a.errors = errors;
  a.batch = batch;
  a.cols = cols;
  a.rank = rank;
  a.world_size = world_size;
  a.page_size = page_size;
  a.dql = decode_query_len;
  a.g = make_geom(page_size, world_size, decode_query_len);
  a.pdl = enable_pdl ? 1 : 0;

  CUtensorMap tmk, tmq;
  st = encode_rows(&tmk, index_k, (uint64_t)num_pages * a.g.rows_per_page, (uint32_t)a.g.R);
  if (st != ICP_OK) return st;
  st = encode_rows(&tmq, index_q, (uint64_t)batch * decode_query_len * ICP_HEADS,
                   (uint32_t)a.g.nq);
  if (st != ICP_OK) return st;
  return to_status(icp::launch_score(tmk, tmq, a, sms, static_cast<cudaStream_t>(stream)));
}

int icp_top16_select(const float *scores, int T, int K, const int32_t *num_valid_pages,
                     int init_blocks, int local_blocks, int index_scale, int index_offset,
                     float *out_scores, int32_t *out_ids, void *stream) {
  if (!valid_select_common(T, K, init_blocks, local_blocks, index_scale, index_offset))
    return ICP_ERR_INVALID_ARG;
  if (T == 0) return ICP_OK;
  if (!scores || !num_valid_pages || !out_scores || !out_ids) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  int st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;
  icp::SelectArgs a;
  memset(&a, 0, sizeof(a));
  a.scores = scores;
  a.T = T;
  a.K = K;
  a.nvp = num_valid_pages;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  a.index_scale = index_scale;
  a.index_offset = index_offset;
  a.out_scores = out_scores;
  a.out_ids = out_ids;
  return to_status(icp::launch_select(a, 0, sms, static_cast<cudaStream_t>(stream)));
}

int icp_publish_rows(const float *scores, int T, int K, const int32_t *num_valid_pages,
                     const int64_t *recv_bases, int32_t *errors, int slot, int rank,
                     int world_size, int heads_per_rank, int capacity, int force_begin_blocks,
                     int force_end_blocks, int64_t spin_limit, int index_scale,
                     int index_offset, int enable_pdl, void *stream) {
  if (!valid_select_common(T, K, force_begin_blocks, force_end_blocks, index_scale,
                           index_offset))
    return ICP_ERR_INVALID_ARG;
  if (world_size != 1 && world_size != 2 && world_size != 4) return ICP_ERR_INVALID_ARG;
  if (heads_per_rank * world_size != ICP_HEADS) return ICP_ERR_INVALID_ARG;
  if (rank < 0 || rank >= world_size || slot < 0 || slot > 2) return ICP_ERR_INVALID_ARG;
  if (T < 1 || T > capacity || spin_limit < 1) return ICP_ERR_INVALID_ARG;
  if (!scores || !num_valid_pages || !recv_bases || !errors) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  int st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;
  icp::SelectArgs a;
  memset(&a, 0, sizeof(a));
  a.scores = scores;
  a.T = T;
  a.K = K;
  a.nvp = num_valid_pages;
  a.init_blocks = force_begin_blocks;
  a.local_blocks = force_end_blocks;
  a.index_scale = index_scale;
  a.index_offset = index_offset;
  a.recv_bases = recv_bases;
  a.errors = errors;
  a.slot = slot;
  a.rank = rank;
  a.world_size = world_size;
  a.heads_per_rank = heads_per_rank;
  a.capacity = capacity;
  a.spin_limit = spin_limit;
  a.pdl = enable_pdl ? 1 : 0;
  return to_status(icp::launch_select(a, 1, sms, static_cast<cudaStream_t>(stream)));
}

int icp_merge(int32_t *recv, const int32_t *num_valid_pages, int T, int slot, int world_size,
              int heads_per_rank, int capacity, int init_blocks, int local_blocks,
              int64_t spin_limit, int32_t *errors, float *out_scores, int32_t *out_ids,
              int enable_pdl, void *stream) {
  if (world_size != 1 && world_size != 2 && world_size != 4) return ICP_ERR_INVALID_ARG;
  if (heads_per_rank * world_size != ICP_HEADS) return ICP_ERR_INVALID_ARG;
  if (slot < 0 || slot > 2 || T < 1 || T > capacity || spin_limit < 1)
    return ICP_ERR_INVALID_ARG;
  if (init_blocks < 0 || local_blocks < 0 || init_blocks + local_blocks > ICP_TOPK)
    return ICP_ERR_INVALID_ARG;
  if (!recv || !num_valid_pages || !errors || !out_scores || !out_ids) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  int st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;
  icp::MergeArgs a;
  memset(&a, 0, sizeof(a));
  a.recv = recv;
  a.nvp = num_valid_pages;
  a.T = T;
  a.slot = slot;
  a.world_size = world_size;
  a.heads_per_rank = heads_per_rank;
  a.capacity = capacity;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  a.spin_limit = spin_limit;
  a.errors = errors;
  a.out_scores = out_scores;
  a.out_ids = out_ids;
  a.pdl = enable_pdl ? 1 : 0;
  return to_status(icp::launch_merge(a, false, static_cast<cudaStream_t>(stream)));
}

int icp_publish_rows_tagged(const float *scores, int T, int K, const int32_t *num_valid_pages,
                            const int64_t *recv_bases, int32_t *generations, int slot, int rank,
                            int world_size, int heads_per_rank, int capacity,
                            int force_begin_blocks, int force_end_blocks, int index_scale,
                            int index_offset, int enable_pdl, void *stream) {
  if (!valid_select_common(T, K, force_begin_blocks, force_end_blocks, index_scale,
                           index_offset))
    return ICP_ERR_INVALID_ARG;
  if (world_size != 1 && world_size != 2 && world_size != 4) return ICP_ERR_INVALID_ARG;
  if (heads_per_rank * world_size != ICP_HEADS) return ICP_ERR_INVALID_ARG;
  if (rank < 0 || rank >= world_size || slot < 0 || slot > 2) return ICP_ERR_INVALID_ARG;
  if (T < 1 || T > capacity) return ICP_ERR_INVALID_ARG;
  if (!scores || !num_valid_pages || !recv_bases || !generations) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  int st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;
  icp::SelectArgs a;
  memset(&a, 0, sizeof(a));
  a.scores = scores;
  a.T = T;
  a.K = K;
  a.nvp = num_valid_pages;
  a.init_blocks = force_begin_blocks;
  a.local_blocks = force_end_blocks;
  a.index_scale = index_scale;
  a.index_offset = index_offset;
  a.recv_bases = recv_bases;
  a.generations = generations;
  a.slot = slot;
  a.rank = rank;
  a.world_size = world_size;
  a.heads_per_rank = heads_per_rank;
  a.capacity = capacity;
  a.pdl = enable_pdl ? 1 : 0;
  return to_status(icp::launch_select(a, 2, sms, static_cast<cudaStream_t>(stream)));
}

int icp_merge_tagged(const int64_t *recv, int32_t *expected, const int32_t *num_valid_pages,
                     int T, int slot, int world_size, int heads_per_rank, int capacity,
                     int init_blocks, int local_blocks, int64_t spin_limit, int32_t *errors,
                     float *out_scores, int32_t *out_ids, int enable_pdl, void *stream) {
  if (world_size != 1 && world_size != 2 && world_size != 4) return ICP_ERR_INVALID_ARG;
  if (heads_per_rank * world_size != ICP_HEADS) return ICP_ERR_INVALID_ARG;
  if (slot < 0 || slot > 2 || T < 1 || T > capacity || spin_limit < 1)
    return ICP_ERR_INVALID_ARG;
  if (init_blocks < 0 || local_blocks < 0 || init_blocks + local_blocks > ICP_TOPK)
    return ICP_ERR_INVALID_ARG;
  if (!recv || !expected || !num_valid_pages || !errors || !out_scores || !out_ids)
    return ICP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(recv) & 7u) != 0) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  int st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;
  icp::MergeArgs a;
  memset(&a, 0, sizeof(a));
  a.recv64 = reinterpret_cast<const unsigned long long *>(recv);
  a.expected = expected;
  a.nvp = num_valid_pages;
  a.T = T;
  a.slot = slot;
  a.world_size = world_size;
  a.heads_per_rank = heads_per_rank;
  a.capacity = capacity;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  a.spin_limit = spin_limit;
  a.errors = errors;
  a.out_scores = out_scores;
  a.out_ids = out_ids;
  a.pdl = enable_pdl ? 1 : 0;
  return to_status(icp::launch_merge(a, true, static_cast<cudaStream_t>(stream)));
}

size_t icp_score_select_workspace_bytes(int batch, int decode_query_len) {
  if (batch < 0 || batch > ICP_MAX_BATCH || decode_query_len < 1 || decode_query_len > 8)
    return 0;
  return icp::fused_workspace_bytes(batch, decode_query_len);
}

int icp_score_select(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
                     const int32_t *block_table, int64_t block_table_stride,
                     const int32_t *seq_lens, int batch, int cols, int rank, int world_size,
                     int page_size, int decode_query_len, int max_decode_query_len,
                     const int32_t *num_valid_pages, int init_blocks, int local_blocks,
                     void *workspace, size_t workspace_bytes, float *out_scores,
                     int32_t *out_ids, int32_t *errors, void *stream) {
  int st = check_score_args(index_q, index_k, num_pages, block_table, block_table_stride,
                            seq_lens, batch, cols, rank, world_size, page_size, decode_query_len,
                            max_decode_query_len);
  if (st != ICP_OK) return st;
  if (init_blocks < 0 || local_blocks < 0 || init_blocks + local_blocks > ICP_TOPK)
    return ICP_ERR_INVALID_ARG;
  if (batch == 0) return ICP_OK;
  if (!num_valid_pages || !out_scores || !out_ids || !workspace) return ICP_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ICP_ERR_INVALID_ARG;
  if (workspace_bytes < icp::fused_workspace_bytes(batch, decode_query_len))
    return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;

  icp::ScoreArgs a;
  memset(&a, 0, sizeof(a));
  a.block_table = block_table;
  a.bt_stride = block_table_stride;
  a.num_pages = (int)num_pages;
  a.seq_lens = seq_lens;
  a.errors = errors;
  a.batch = batch;
  a.cols = cols;
  a.rank = rank;
  a.world_size = world_size;
  a.page_size = page_size;
  a.dql = decode_query_len;
  a.g = make_geom(page_size, world_size, decode_query_len);
  a.nvp = num_valid_pages;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  // global id of column c (msa_icp_decode_index_score_sharded: P256 sharded
  // columns are local pages of global block 2 c + rank * 2 // world_size)
  const bool local_pages = page_size == 256 && world_size > 1;
  a.index_scale = local_pages ? 2 : 1;
  a.index_offset = local_pages ? rank * 2 / world_size : 0;
  a.out_scores = out_scores;
  a.out_ids = out_ids;
  const size_t counters = ((size_t)batch * 16 + 255) / 256 * 256;  // per-request info
  a.ws_counters = static_cast<int32_t *>(workspace);
  a.ws_records = static_cast<uint8_t *>(workspace) + counters;

  CUtensorMap tmk, tmq;
  st = encode_rows(&tmk, index_k, (uint64_t)num_pages * a.g.rows_per_page, (uint32_t)a.g.R);
  if (st != ICP_OK) return st;
  st = encode_rows(&tmq, index_q, (uint64_t)batch * decode_query_len * ICP_HEADS,
                   (uint32_t)a.g.nq);
  if (st != ICP_OK) return st;
  return to_status(
      icp::launch_score_select(tmk, tmq, a, sms, static_cast<cudaStream_t>(stream)));
}

int64_t icp_prefill_plan_words(int batch, int T) {
  if (batch < 0 || T < 0) return -1;
  const long long records = ((long long)T + icp::kPlanTokens - 1) / icp::kPlanTokens + batch;
  if (records > icp::kMaxBatchDevice) return -1;
  return icp::kPlanHeaderInts + (int64_t)icp::kPlanRecordInts * (records > 0 ? records : 1);
}

int icp_prefill_plan(const int32_t *qo_indptr, const int32_t *seq_lens, int batch, int T,
                     int32_t *plan, int64_t plan_words, int32_t *errors, void *stream) {
  const int64_t need = icp_prefill_plan_words(batch, T);
  if (need < 0 || plan_words < need || !plan || !aligned16(plan)) return ICP_ERR_INVALID_ARG;
  if (batch > 0 && (!qo_indptr || !seq_lens)) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  int st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;
  const int capacity = (int)((plan_words - icp::kPlanHeaderInts) / icp::kPlanRecordInts);
  const int cap = capacity < icp::kMaxBatchDevice ? capacity : icp::kMaxBatchDevice;
  return to_status(icp::launch_prefill_plan(qo_indptr, seq_lens, batch, T, plan, cap, errors,
                                            static_cast<cudaStream_t>(stream)));
}

int icp_prefill_score(const uint8_t *index_q, const uint8_t *index_k, int64_t num_pages,
                      const int32_t *block_table, int64_t block_table_stride,
                      const int32_t *plan, int64_t plan_words, float *score_out, int T,
                      int cols, int rank, int world_size, int page_size, int32_t *errors,
                      void *stream) {
  if (T < 0 || plan_words < icp::kPlanHeaderInts + icp::kPlanRecordInts || !aligned16(plan))
    return ICP_ERR_INVALID_ARG;
  const int64_t records = (plan_words - icp::kPlanHeaderInts) / icp::kPlanRecordInts;
  const int capacity = (int)(records < icp::kMaxBatchDevice ? records : icp::kMaxBatchDevice);
  // the decode checks on layout, pointers and sizes (query length 1: the
  // records carry their own)
  int st = check_score_args(index_q, index_k, num_pages, block_table, block_table_stride, plan,
                            T > 0 ? capacity : 0, cols, rank, world_size, page_size, 1, 1);
  if (st != ICP_OK) return st;
  if (T == 0) return ICP_OK;
  if (!score_out) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;

  icp::ScoreArgs a;
  memset(&a, 0, sizeof(a));
  a.block_table = block_table;
  a.bt_stride = block_table_stride;
  a.num_pages = (int)num_pages;
  a.score_out = score_out;
  a.errors = errors;
  a.batch = capacity;
  a.cols = cols;
  a.rank = rank;
  a.world_size = world_size;
  a.page_size = page_size;
  a.dql = icp::kPlanTokens;
  a.g = make_geom(page_size, world_size, icp::kPlanTokens);
  a.vreq = plan;
  a.vcount = plan;
  a.wide = 1;

  CUtensorMap tmk, tmq;
  st = encode_rows(&tmk, index_k, (uint64_t)num_pages * a.g.rows_per_page, (uint32_t)a.g.R);
  if (st != ICP_OK) return st;
  // one box of a record's 4 * 64 query rows
  st = encode_rows(&tmq, index_q, (uint64_t)T * ICP_HEADS, (uint32_t)(4 * icp::kPlanTokens));
  if (st != ICP_OK) return st;
  return to_status(icp::launch_score(tmk, tmq, a, sms, static_cast<cudaStream_t>(stream)));
}

int icp_prefill_select(const float *scores, int T, int K, const int32_t *num_valid_pages,
                       int world_size, int heads_per_rank, int init_blocks, int local_blocks,
                       int index_scale, int index_offset, int32_t *carrier, void *stream) {
  if (!valid_select_common(T, K, init_blocks, local_blocks, index_scale, index_offset))
    return ICP_ERR_INVALID_ARG;
  if (world_size != 1 && world_size != 2 && world_size != 4) return ICP_ERR_INVALID_ARG;
  if (heads_per_rank * world_size != ICP_HEADS) return ICP_ERR_INVALID_ARG;
  if (T == 0) return ICP_OK;
  if (!scores || !num_valid_pages || !carrier) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  int st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;
  icp::SelectArgs a;
  memset(&a, 0, sizeof(a));
  a.scores = scores;
  a.T = T;
  a.K = K;
  a.nvp = num_valid_pages;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  a.index_scale = index_scale;
  a.index_offset = index_offset;
  a.world_size = world_size;
  a.heads_per_rank = heads_per_rank;
  a.carrier = carrier;
  return to_status(icp::launch_select(a, 3, sms, static_cast<cudaStream_t>(stream)));
}

int icp_prefill_merge(const int32_t *received, const int32_t *num_valid_pages, int T,
                      int world_size, int heads_per_rank, int init_blocks, int local_blocks,
                      float *out_scores, int32_t *out_ids, void *stream) {
  if (world_size != 1 && world_size != 2 && world_size != 4) return ICP_ERR_INVALID_ARG;
  if (heads_per_rank * world_size != ICP_HEADS) return ICP_ERR_INVALID_ARG;
  if (T < 0) return ICP_ERR_INVALID_ARG;
  if (init_blocks < 0 || local_blocks < 0 || init_blocks + local_blocks > ICP_TOPK)
    return ICP_ERR_INVALID_ARG;
  if (T == 0) return ICP_OK;
  if (!received || !num_valid_pages || !out_scores || !out_ids) return ICP_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  int st = current_device(&dev, &sms);
  if (st != ICP_OK) return st;
  icp::MergeArgs a;
  memset(&a, 0, sizeof(a));
  a.received = received;
  a.nvp = num_valid_pages;
  a.T = T;
  a.world_size = world_size;
  a.heads_per_rank = heads_per_rank;
  a.init_blocks = init_blocks;
  a.local_blocks = local_blocks;
  a.out_scores = out_scores;
  a.out_ids = out_ids;
  return to_status(icp::launch_merge_carrier(a, static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
