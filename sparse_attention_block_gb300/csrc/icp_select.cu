// icp_select.cu - Top16 select, legacy receive-row publish and owner merge.
//
// Top16 rule (msa_icp_topk_select_publish with the forced blocks of
// prepare_msa_icp_indexer): valid ids are c * index_scale + index_offset <
// num_valid_pages[t].  If num_valid_pages[t] <= 16 every valid id is kept;
// otherwise ids in [0, init) and [nvp - local, nvp) are forced and the other
// slots go to the best remaining ids by (score descending, id ascending).
// Output: ids ascending with their raw scores, then (-1, -inf) padding.
//
// Select: one CTA per (token, head) row, the row held in registers.  Every
// non-forced valid score becomes a unique 64-bit key (score order, then
// lower id).  With m free slots, tau = the m-th largest per-thread maximum
// is a lower bound of the m-th largest key, and only the m threads whose
// maximum reaches tau can hold keys >= tau, so at most m * EPT candidates
// survive; one warp then picks the m largest candidates exactly.
#include "icp_device.cuh"
#include "icp_internal.h"

namespace icp {
namespace {

constexpr int kRowWords = 33;

// Bounded poll of a ready flag until it equals `want`.  Returns false after
// spin_limit polls or kWaitTimeoutNs, whichever comes first.
__device__ __forceinline__ bool poll_flag(const int *flag, int want, long long spin_limit) {
  const unsigned long long t0 = globaltimer_ns();
  for (long long it = 0; it < spin_limit; ++it) {
    if (ld_acquire_gpu(flag) == want) return true;
    if ((it & 255) == 255 && globaltimer_ns() - t0 > kWaitTimeoutNs) return false;
  }
  return false;
}

template <int NT, int EPT, bool PUBLISH>
__global__ void __launch_bounds__(NT) select_kernel(const SelectArgs a) {
  constexpr int NW = NT / 32;
  constexpr int LPT = NT / 32;            // thread maxima per lane in warp 0
  constexpr int CAP = kTopK * EPT;        // candidate bound
  constexpr int CPL = (CAP + 31) / 32;    // candidates per lane in warp 0
  static_assert(NW >= 1, "NT");

  __shared__ int s_nf, s_nc;
  __shared__ int s_fid[kTopK];
  __shared__ float s_fsc[kTopK];
  __shared__ unsigned long long s_tm[NT];
  __shared__ unsigned long long s_cand[CAP];
  __shared__ unsigned long long s_tau;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = blockIdx.x;
  const int t = row >> 2;
  const int h = row & 3;
  const float *src = a.scores + (long long)row * a.K;
  const int nvp = a.nvp[t];

  if (tid == 0) {
    s_nf = 0;
    s_nc = 0;
  }
  __syncthreads();

  unsigned long long key[EPT];
  unsigned long long tm = 0;
#pragma unroll
  for (int i = 0; i < EPT; ++i) {
    const int c = tid + i * NT;
    key[i] = 0;
    if (c < a.K) {
      const float v = src[c];
      const int id = c * a.index_scale + a.index_offset;
      if (id < nvp) {
        if (forced_id(id, nvp, a.init_blocks, a.local_blocks)) {
          const int slot = atomicAdd(&s_nf, 1);
          if (slot < kTopK) {
            s_fid[slot] = id;
            s_fsc[slot] = v;
          }
        } else {
          key[i] = make_key(v, id);
        }
      }
    }
    tm = key[i] > tm ? key[i] : tm;
  }
  s_tm[tid] = tm;
  __syncthreads();
  const int nf = min(s_nf, kTopK);
  const int m = kTopK - nf;

  // tau = m-th largest thread maximum (1 = "take every key" when fewer than
  // m threads hold one)
  if (warp == 0) {
    unsigned long long loc[LPT];
    unsigned long long lmax = 0;
#pragma unroll
    for (int j = 0; j < LPT; ++j) {
      loc[j] = s_tm[lane + 32 * j];
      lmax = loc[j] > lmax ? loc[j] : lmax;
    }
    unsigned long long tau = 0;
    int found = 0;
    for (int r = 0; r < m; ++r) {
      const unsigned long long w = warp_max_key(lmax);
      if (w == 0) break;
      tau = w;
      ++found;
      if (lmax == w) {
        lmax = 0;
#pragma unroll
        for (int j = 0; j < LPT; ++j) {
          if (loc[j] == w) loc[j] = 0;
          lmax = loc[j] > lmax ? loc[j] : lmax;
        }
      }
    }
    if (lane == 0) s_tau = (found < m) ? 1ull : tau;
  }
  __syncthreads();
  if (m > 0) {
    const unsigned long long tau = s_tau;
#pragma unroll
    for (int i = 0; i < EPT; ++i) {
      if (key[i] != 0 && key[i] >= tau) {
        const int slot = atomicAdd(&s_nc, 1);
        if (slot < CAP) s_cand[slot] = key[i];
      }
    }
  }
  __syncthreads();

  if (warp != 0) return;
  const int nc = min(s_nc, CAP);
  // pick the m largest candidates; lane nf + r receives the r-th
  unsigned long long cl[CPL];
  unsigned long long lmax = 0;
#pragma unroll
  for (int j = 0; j < CPL; ++j) {
    const int k = lane + 32 * j;
    cl[j] = (k < nc) ? s_cand[k] : 0ull;
    lmax = cl[j] > lmax ? cl[j] : lmax;
  }
  unsigned long long mine = 0;
  int nch = 0;
  for (int r = 0; r < m; ++r) {
    const unsigned long long w = warp_max_key(lmax);
    if (w == 0) break;
    if (lane == nf + r) mine = w;
    ++nch;
    if (lmax == w) {
      lmax = 0;
#pragma unroll
      for (int j = 0; j < CPL; ++j) {
        if (cl[j] == w) cl[j] = 0;
        lmax = cl[j] > lmax ? cl[j] : lmax;
      }
    }
  }
  const int n = nf + nch;
  int my_id = 0x7FFFFFFF;
  float my_sc = -INFINITY;
  if (lane < nf) {
    my_id = s_fid[lane];
    my_sc = s_fsc[lane];
  } else if (lane < n) {
    my_id = key_id(mine);
    my_sc = src[(my_id - a.index_offset) / a.index_scale];  // raw score bits
  }
  int out_id;
  float out_sc;
  sort_by_id_16(lane, n, my_id, my_sc, out_id, out_sc);

  if constexpr (!PUBLISH) {
    if (lane < kTopK) {
      a.out_scores[(long long)row * kTopK + lane] = out_sc;
      a.out_ids[(long long)row * kTopK + lane] = out_id;
    }
  } else {
    const int hpr = a.heads_per_rank;
    int *base = reinterpret_cast<int *>(a.recv_bases[h / hpr]);
    const long long r =
        (((long long)a.slot * a.world_size + a.rank) * hpr + h % hpr) * a.capacity + t;
    int *dst = base + r * kRowWords;
    int ok = 0;
    if (lane == 0) ok = poll_flag(dst + 32, 0, a.spin_limit) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) {
      if (lane == 0) atomicAdd(a.errors, 1);
      return;
    }
    if (lane < kTopK) {
      dst[lane] = __float_as_int(out_sc);
      dst[kTopK + lane] = out_id;
    }
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release_gpu(dst + 32, 1);
  }
}

// One warp per (token, owned head).
__global__ void __launch_bounds__(128) merge_kernel(const MergeArgs a) {
  __shared__ int s_id[4][64];
  __shared__ float s_sc[4][64];
  __shared__ unsigned long long s_key[4][64];
  __shared__ int s_sel[4][64];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + warp;
  const int hpr = a.heads_per_rank;
  if (item >= a.T * hpr) return;
  const int t = item / hpr, hl = item % hpr;
  const int nvp = a.nvp[t];
  const int ws = a.world_size;

  unsigned read_mask = 0;
  for (int s = 0; s < 4; ++s) {
    const int e = s * 16 + (lane & 15);
    if (lane < 16) {
      s_id[warp][e] = -1;
      s_sc[warp][e] = -INFINITY;
    }
    if (s >= ws) continue;
    const long long r = (((long long)a.slot * ws + s) * hpr + hl) * a.capacity + t;
    int *row = a.recv + r * kRowWords;
    int ok = 0;
    if (lane == 0) ok = poll_flag(row + 32, 1, a.spin_limit) ? 1 : 0;
    ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
    if (!ok) {
      if (lane == 0) atomicAdd(a.errors, 1);
      continue;
    }
    read_mask |= 1u << s;
    if (lane < 16) {
      (void)ld_acquire_gpu(row + 32);  // order this lane's reads after the flag
      s_sc[warp][e] = __int_as_float(row[lane]);
      s_id[warp][e] = row[16 + lane];
    }
  }
  __syncwarp();
  // free the rows that were read
  if (lane == 0) {
    for (int s = 0; s < ws; ++s)
      if (read_mask & (1u << s)) {
        const long long r = (((long long)a.slot * ws + s) * hpr + hl) * a.capacity + t;
        st_release_gpu(a.recv + r * kRowWords + 32, 0);
      }
  }

  // union with the maximum score per id (first source wins a tie)
  int nforced = 0;
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int e = lane + 32 * k;
    const int id = s_id[warp][e];
    const float sc = s_sc[warp][e];
    bool keep = (id >= 0) && (id < nvp);
    if (keep) {
      for (int e2 = 0; e2 < 64; ++e2) {
        if (e2 == e || s_id[warp][e2] != id) continue;
        const float s2 = s_sc[warp][e2];
        if (s2 > sc || (s2 == sc && e2 < e)) {
          keep = false;
          break;
        }
      }
    }
    const bool f = keep && forced_id(id, nvp, a.init_blocks, a.local_blocks);
    s_key[warp][e] = (keep && !f) ? make_key(sc, id) : 0ull;
    s_sel[warp][e] = f ? 1 : 0;
    nforced += f ? 1 : 0;
  }
  nforced = __reduce_add_sync(0xFFFFFFFFu, nforced);
  __syncwarp();
  const int m = kTopK - min(nforced, kTopK);
  // keep the m best free entries: rank = number of larger keys
#pragma unroll
  for (int k = 0; k < 2; ++k) {
    const int e = lane + 32 * k;
    const unsigned long long my = s_key[warp][e];
    if (my != 0) {
      int rank = 0;
      for (int e2 = 0; e2 < 64; ++e2) rank += (s_key[warp][e2] > my) ? 1 : 0;
      if (rank < m) s_sel[warp][e] = 1;
    }
  }
  __syncwarp();
  // compact the selected entries into lanes and order them by id
  int nsel = 0, my_id = 0x7FFFFFFF;
  float my_sc = -INFINITY;
  for (int e = 0; e < 64; ++e) {
    if (s_sel[warp][e]) {
      if (nsel == lane) {
        my_id = s_id[warp][e];
        my_sc = s_sc[warp][e];
      }
      ++nsel;
    }
  }
  int out_id;
  float out_sc;
  sort_by_id_16(lane, min(nsel, kTopK), my_id, my_sc, out_id, out_sc);
  if (lane < kTopK) {
    const long long o = ((long long)t * hpr + hl) * kTopK + lane;
    a.out_scores[o] = out_sc;
    a.out_ids[o] = out_id;
  }
}

}  // namespace

cudaError_t launch_select(const SelectArgs &a, bool publish, cudaStream_t stream) {
  const int rows = a.T * 4;
  if (rows == 0) return cudaSuccess;
  if (a.K <= 1024) {
    if (publish) select_kernel<128, 8, true><<<rows, 128, 0, stream>>>(a);
    else select_kernel<128, 8, false><<<rows, 128, 0, stream>>>(a);
  } else if (a.K <= 4096) {
    if (publish) select_kernel<256, 16, true><<<rows, 256, 0, stream>>>(a);
    else select_kernel<256, 16, false><<<rows, 256, 0, stream>>>(a);
  } else {
    if (publish) select_kernel<512, 24, true><<<rows, 512, 0, stream>>>(a);
    else select_kernel<512, 24, false><<<rows, 512, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs &a, cudaStream_t stream) {
  const int items = a.T * a.heads_per_rank;
  if (items == 0) return cudaSuccess;
  merge_kernel<<<(items + 3) / 4, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace icp
