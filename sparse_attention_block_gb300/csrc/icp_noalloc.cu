// icp_noalloc.cu - icp_score_select_noalloc: the fused scorer + Top16 select
// with its scratch in a fixed device array instead of a caller workspace.
//
// Who needs this: callers that cannot allocate device memory at the point of
// the call.  Examples are a serving engine that carves the whole GPU into
// fixed pools at start-up and forbids later allocations, code that records
// the decode step into a CUDA graph (an allocation there is either illegal
// or changes what the graph captures), and latency-critical paths where
// cudaMalloc's implicit device synchronisation cannot be paid.  Such a
// caller still passes its own inputs and outputs; only the scratch comes
// from here.
//
// The scratch is one file-scope array per device, kept by every GPU that
// loads the library until the process exits.  In host code its name is only
// a host-side stand-in, never a device address, so the address is looked up
// once per device with cudaGetSymbolAddress while that device is current and
// then passed to the kernels.
//
// Nothing in the scratch has to start at zero: the scorer writes every
// per-request record and every partial list before the merge kernel reads
// it, so contents left by an earlier call are never read.  All calls on a
// device share the one array, so calls that overlap on the GPU (other
// streams, or other threads) race on it and must be serialised by the
// caller.
#include <mutex>

#include "icp.h"
#include "icp_internal.h"

namespace {

static __device__ __align__(256) unsigned char g_noalloc_scratch[ICP_NOALLOC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDevices] = {};

// Device address of this device's scratch array; resolved on first use and
// kept for the life of the process.  It is the address in the device's
// primary context (the CUDA runtime's); after cudaDeviceReset, or under
// another context on the same device, it would be stale, which the header
// tells callers.
int scratch_for_current_device(void **out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ICP_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return ICP_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_scratch_mutex);
  if (!g_scratch_ptr[dev]) {
    void *ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr)
      return ICP_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return ICP_OK;
}

}  // namespace

extern "C" int icp_score_select_noalloc(const uint8_t *index_q, const uint8_t *index_k,
                                        int64_t num_pages, const int32_t *block_table,
                                        int64_t block_table_stride, const int32_t *seq_lens,
                                        int batch, int cols, int rank, int world_size,
                                        int page_size, int decode_query_len,
                                        int max_decode_query_len,
                                        const int32_t *num_valid_pages, int init_blocks,
                                        int local_blocks, float *out_scores, int32_t *out_ids,
                                        int32_t *errors, void *stream) {
  if (batch < 0 || decode_query_len < 1) return ICP_ERR_INVALID_ARG;
  if (batch == 0) return ICP_OK;
  const size_t need = icp_score_select_workspace_bytes(batch, decode_query_len);
  // a batch whose scratch does not fit the fixed array is refused up front
  if (need == 0 || need > (size_t)ICP_NOALLOC_SCRATCH_BYTES) return ICP_ERR_INVALID_ARG;
  void *scratch = nullptr;
  const int st = scratch_for_current_device(&scratch);
  if (st != ICP_OK) return st;
  return icp_score_select(index_q, index_k, num_pages, block_table, block_table_stride, seq_lens,
                          batch, cols, rank, world_size, page_size, decode_query_len,
                          max_decode_query_len, num_valid_pages, init_blocks, local_blocks,
                          scratch, (size_t)ICP_NOALLOC_SCRATCH_BYTES, out_scores, out_ids,
                          errors, stream);
}
