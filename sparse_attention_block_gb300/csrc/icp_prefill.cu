// icp_prefill.cu - the prefill window plan (prepare_msa_icp_indexer:
// prefill_window_plan, built one time for each window of queries in a step).
//
// A window holds, for every request b, a chunk of its newest
// n_b = qo_indptr[b+1] - qo_indptr[b] tokens (window tokens qo_indptr[b] ..
// qo_indptr[b+1] - 1), token j at position seq_len_b - n_b + j: the decode
// placement with a per-request query length.  The plan cuts every chunk into
// records of at most kPlanTokens (64) consecutive tokens, 256 query rows: two
// 128-row MMA operands of distinct rows for the prefill scorer.  A record is a request of
// its own for the scorer: the request's block-table row, the record's tokens
// as its queries, and seq_len = its last position + 1, so the causal mask
// and the key stream are the decode ones.  The scorer writes each record's
// rows across the request's full column range.
#include "icp_device.cuh"
#include "icp_internal.h"

namespace icp {
namespace {

constexpr int kPlanThreads = 1024;

// Records of request b, or -1 when its chunk is not a valid one: qo_indptr
// must not decrease, stay within [0, T], and a chunk cannot hold more tokens
// than its request's seq_len.
__device__ __forceinline__ int records_of(const int32_t *qo, const int32_t *seq_lens, int b,
                                          int T) {
  const int q0 = qo[b], q1 = qo[b + 1], n = q1 - q0, sl = seq_lens[b];
  if (q0 < 0 || n < 0 || q1 > T || n > sl) return -1;
  return (n + kPlanTokens - 1) / kPlanTokens;
}

__global__ void __launch_bounds__(kPlanThreads) prefill_plan_kernel(
    const int32_t *qo, const int32_t *seq_lens, int batch, int T, int32_t *plan, int capacity,
    int32_t *errors) {
  __shared__ int s_part[kPlanThreads / 32];
  __shared__ int s_first[kMaxBatchDevice + 1];  // first record of every request
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunk = (batch + kPlanThreads - 1) / kPlanThreads;
  const int lo = min(batch, tid * chunk), hi = min(batch, lo + chunk);

  int sum = 0, bad = 0;
  for (int b = lo; b < hi; ++b) {
    const int r = records_of(qo, seq_lens, b, T);
    if (r < 0) ++bad;
    else sum += r;
  }
  // exclusive scan of the per-thread record counts
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) s_part[warp] = incl;
  __syncthreads();
  int base = 0;
  for (int w = 0; w < warp; ++w) base += s_part[w];
  int run = base + incl - sum;
  for (int b = lo; b < hi; ++b) {
    s_first[b] = run;
    run += max(records_of(qo, seq_lens, b, T), 0);
  }
  if (tid == kPlanThreads - 1) {
    s_first[batch] = base + incl;
    plan[0] = min(base + incl, capacity);
  }
  __syncthreads();

  // every thread writes records tid, tid + kPlanThreads, ...; the request
  // of record idx is the last one whose first record is <= idx (requests
  // without records share their successor's first record)
  const int total = s_first[batch];
  const int n_out = min(total, capacity);
  for (int idx = tid; idx < n_out; idx += kPlanThreads) {
    int b0 = 0, b1 = batch - 1;
    while (b0 < b1) {
      const int mid = (b0 + b1 + 1) >> 1;
      if (s_first[mid] <= idx) b0 = mid;
      else b1 = mid - 1;
    }
    const int b = b0, k = idx - s_first[b0];
    const int q0 = qo[b], n = qo[b + 1] - q0, sl = seq_lens[b];
    const int ntok = min(kPlanTokens, n - kPlanTokens * k);
    int4 *rec = reinterpret_cast<int4 *>(plan + kPlanHeaderInts + (long long)kPlanRecordInts * idx);
    // {first token, block-table row, last position + 1, tokens}, {the
    // request's seq_len, 0, 0, 0}
    rec[0] = make_int4(q0 + kPlanTokens * k, b, sl - n + kPlanTokens * k + ntok, ntok);
    rec[1] = make_int4(sl, 0, 0, 0);
  }
  const int over = tid == 0 ? max(total - capacity, 0) : 0;
  if ((bad || over) && errors) atomicAdd(errors, bad + over);
}

}  // namespace

cudaError_t launch_prefill_plan(const int32_t *qo_indptr, const int32_t *seq_lens, int batch,
                                int T, int32_t *plan, int capacity, int32_t *errors,
                                cudaStream_t stream) {
  prefill_plan_kernel<<<1, kPlanThreads, 0, stream>>>(qo_indptr, seq_lens, batch, T, plan,
                                                       capacity, errors);
  return cudaGetLastError();
}

}  // namespace icp
