// icp_prefill.cu - the prefill window plan (prepare_msa_icp_indexer:
// prefill_window_plan, once per query window and step).
//
// A window holds, for every request b, a chunk of its newest
// n_b = qo_indptr[b+1] - qo_indptr[b] tokens (window tokens qo_indptr[b] ..
// qo_indptr[b+1] - 1), token j at position seq_len_b - n_b + j: the decode
// placement with a per-request query length.  The plan cuts every chunk into
// records of at most kPlanTokens (32) consecutive tokens, 128 query rows: one
// MMA tile of distinct rows for the prefill scorer.  A record is a request of
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
  if (tid == kPlanThreads - 1) plan[0] = min(base + incl, capacity);

  int run = base + incl - sum;
  int over = 0;
  for (int b = lo; b < hi; ++b) {
    const int r = records_of(qo, seq_lens, b, T);
    if (r <= 0) continue;
    const int q0 = qo[b], n = qo[b + 1] - q0, sl = seq_lens[b];
    for (int k = 0; k < r; ++k) {
      const int idx = run + k;
      if (idx >= capacity) {
        ++over;
        continue;
      }
      const int ntok = min(kPlanTokens, n - kPlanTokens * k);
      int32_t *rec = plan + kPlanHeaderInts + (long long)kPlanRecordInts * idx;
      rec[0] = q0 + kPlanTokens * k;                 // first token
      rec[1] = b;                                    // block-table row
      rec[2] = sl - n + kPlanTokens * k + ntok;      // last position + 1
      rec[3] = ntok;
      rec[4] = sl;                                   // the request's seq_len
      rec[5] = 0;
      rec[6] = 0;
      rec[7] = 0;
    }
    run += r;
  }
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
