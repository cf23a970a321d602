// icp_fused.cuh - records the fused scorer + Top16 select leaves in its
// workspace for the merge kernel, and helpers both kernels share.
#pragma once

#include "icp_device.cuh"
#include "icp_internal.h"

namespace icp {

// Plane columns of a request: B128 blocks, local pages, or (P256 with one
// rank) halves of 256-row pages.
__device__ __forceinline__ int units_of(int seq_len, int page_size, int split) {
  const int u = split ? 128 : page_size;
  return seq_len <= 0 ? 0 : (seq_len + u - 1) / u;
}

// Workspace record of one (partial list, query row), 288 bytes:
//   u64 keys[16]   best non-forced entries seen (unsorted, 0 = empty)
//   u64 max        largest of keys (0 = none)
//   i32 fcount     forced entries that follow
//   i32 fid[16], f32 fsc[16]
struct alignas(16) PartialRec {
  unsigned long long keys[16];
  unsigned long long max;
  int fcount;
  int pad_;
  int fid[16];
  float fsc[16];
  int pad2_[4];
};
static_assert(sizeof(PartialRec) == 288, "record layout");

__device__ __forceinline__ PartialRec *partial_rec(const ScoreArgs &a, int pidx, int row) {
  return reinterpret_cast<PartialRec *>(a.ws_records) + (size_t)pidx * (4 * a.dql) + row;
}

// Index of the CTA whose tile range contains tile x.
__device__ __forceinline__ int cta_of(long long total, int grid, long long x) {
  int lo = 0, hi = grid - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (total * mid / grid <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Per-request facts the fused scorer leaves for the merge kernel.
struct alignas(16) ReqInfo {
  int i0, i1;   // first and last CTA whose tile range covers the request (i1 < i0: none)
  int total;    // tiles of the whole launch
  int nunits;   // plane columns of the request
};


}  // namespace icp
