// icp_select.cu - Top16 select, legacy receive-row publish and owner merge.
//
// Top16 rule (msa_icp_topk_select_publish with the forced blocks of
// prepare_msa_icp_indexer): valid ids are c * index_scale + index_offset <
// num_valid_pages[t].  If num_valid_pages[t] <= 16 every valid id is kept;
// otherwise ids in [0, init) and [nvp - local, nvp) are forced and the other
// slots go to the best remaining ids by (score descending, id ascending).
// Output: ids ascending with their raw scores, then (-1, -inf) padding.
//
// Select: one warp per row for rows up to 2048 columns, a CTA per row
// (persistent, double-buffered in shared memory) for longer rows.  Every
// non-forced valid score
// becomes a unique 64-bit key (score order, then lower id).  With m free
// slots, tau = the m-th largest per-thread best is a lower bound of the m-th
// largest key, and only the m threads whose best reaches tau can hold keys
// >= tau; those are collected and the m largest picked exactly.
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

// Persistent block select (long rows): each CTA takes rows blockIdx.x, blockIdx.x + gridDim.x,
// ... and stages them in shared memory with bulk async copies into two
// buffers, so the next row streams in while the current one is processed.
// MAXK bounds the row length of the variant.
// Where a selected row goes: the plain output arrays, a legacy receive row
// (bounded wait for a free row, 32 data words, release-stored ready flag) or
// a tagged receive row (32 int64 words of generation << 32 | word, the
// generation taken from the publisher's counter for (slot, head, token)).
enum EmitMode { kEmitPlain = 0, kEmitLegacy = 1, kEmitTagged = 2 };

// Address of the legacy receive row (t, h) of this publish.
__device__ __forceinline__ int *legacy_row(const SelectArgs &a, int t, int h) {
  const int hpr = a.heads_per_rank;
  const long long r =
      (((long long)a.slot * a.world_size + a.rank) * hpr + h % hpr) * a.capacity + t;
  return reinterpret_cast<int *>(a.recv_bases[h / hpr]) + r * kRowWords;
}

// The ready flag of that row, read with acquire when the row's work starts so
// that the read overlaps the selection; -1 when not a legacy publish.
template <int MODE>
__device__ __forceinline__ int early_flag(const SelectArgs &a, int lane, int t, int h) {
  if constexpr (MODE == kEmitLegacy) {
    if (lane == 0) return ld_acquire_gpu(legacy_row(a, t, h) + 32);
  }
  return -1;
}

template <int MODE>
__device__ __forceinline__ void emit_row(const SelectArgs &a, int lane, int row, int t, int h,
                                         int out_id, float out_sc, int flag0) {
  if constexpr (MODE == kEmitPlain) {
    if (lane < kTopK) {
      a.out_scores[(long long)row * kTopK + lane] = out_sc;
      a.out_ids[(long long)row * kTopK + lane] = out_id;
    }
  } else {
    const int hpr = a.heads_per_rank;
    const long long r =
        (((long long)a.slot * a.world_size + a.rank) * hpr + h % hpr) * a.capacity + t;
    if constexpr (MODE == kEmitLegacy) {
      int *dst = legacy_row(a, t, h);
      int ok = 0;
      // the flag read when the row started (acquire) usually shows the row
      // free already; otherwise poll (bounded)
      if (lane == 0) ok = (flag0 == 0 || poll_flag(dst + 32, 0, a.spin_limit)) ? 1 : 0;
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0);
      if (!ok) {
        if (lane == 0) atomicAdd(a.errors, 1);
      } else {
        if (lane < kTopK) {
          dst[lane] = __float_as_int(out_sc);
          dst[kTopK + lane] = out_id;
        }
        // the warp barrier orders every lane's data stores before lane 0's
        // release store of the flag (release is cumulative)
        __syncwarp();
        if (lane == 0) st_release_gpu(dst + 32, 1);
      }
    } else {
      int *gen = a.generations +
                 ((long long)a.slot * (a.world_size * hpr) + h) * a.capacity + t;
      unsigned g = 0;
      if (lane == 0) {
        g = (unsigned)*gen + 1u;
        *gen = (int)g;
      }
      g = __shfl_sync(0xFFFFFFFFu, g, 0);
      const unsigned sb = __shfl_sync(0xFFFFFFFFu, __float_as_uint(out_sc), lane & 15);
      const unsigned ib = __shfl_sync(0xFFFFFFFFu, (unsigned)out_id, lane & 15);
      const unsigned long long word =
          ((unsigned long long)g << 32) | (unsigned long long)(lane < kTopK ? sb : ib);
      unsigned long long *dst =
          reinterpret_cast<unsigned long long *>(a.recv_bases[h / hpr]) + r * 32;
      st_relaxed_gpu_u64(dst + lane, word);
    }
  }
}

template <int NT, int MAXK, int MODE>
__global__ void __launch_bounds__(NT) select_block_kernel(const SelectArgs a) {
  constexpr int NW = NT / 32;
  constexpr int EPT = ((MAXK + 4 * NT - 1) / (4 * NT)) * 4;  // row entries per thread
  constexpr int CAP = kTopK * EPT;           // candidate bound (see the file comment)
  constexpr int WL = (NW * kTopK + 31) / 32; // per-warp maxima per lane in warp 0
  constexpr int BUF = ((MAXK + 3) / 4) * 4;  // floats per row buffer

  extern __shared__ __align__(16) unsigned char dyn_smem[];
  float *bufs = reinterpret_cast<float *>(dyn_smem);  // [2][BUF] (bulk) or [1][BUF]
  __shared__ __align__(8) unsigned long long s_bar[2];
  __shared__ int s_nc, s_nf, s_abort;
  __shared__ int s_fid[kTopK];
  __shared__ float s_fsc[kTopK];
  __shared__ unsigned long long s_wtop[NW][kTopK];
  __shared__ unsigned long long s_tau;
  __shared__ unsigned long long s_cand[CAP];
  __shared__ unsigned long long s_sel[kTopK];

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int K = a.K;
  const int rows = a.T * 4;
  const int scale = a.index_scale, off = a.index_offset;
  const bool bulk = (K % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 15u) == 0);
  const uint32_t bytes = (uint32_t)K * 4u;

  if (tid == 0) {
    s_abort = 0;
    if (bulk) {
      mbar_init(smem_u32(&s_bar[0]), 1);
      mbar_init(smem_u32(&s_bar[1]), 1);
      fence_mbarrier_init();
    }
  }
  __syncthreads();
  if (bulk && tid == 0 && (int)blockIdx.x < rows) {
    mbar_arrive_expect_tx(smem_u32(&s_bar[0]), bytes);
    bulk_load(smem_u32(bufs), a.scores + (long long)blockIdx.x * K, bytes, smem_u32(&s_bar[0]));
  }

  int it = 0;
  int nvp_next = (int)blockIdx.x < rows ? __ldg(a.nvp + (blockIdx.x >> 2)) : 0;
  for (int row = blockIdx.x; row < rows; row += gridDim.x, ++it) {
    const int cur = bulk ? (it & 1) : 0;
    float *rowv = bufs + cur * BUF;
    const int nvp = nvp_next;  // loaded one row ahead, off the critical path
    if (row + (int)gridDim.x < rows) nvp_next = __ldg(a.nvp + ((row + gridDim.x) >> 2));
    if (bulk) {
      const int next = row + gridDim.x;
      if (tid == 0 && next < rows) {
        const int nb = cur ^ 1;  // freed by the previous iteration's last barrier
        mbar_arrive_expect_tx(smem_u32(&s_bar[nb]), bytes);
        bulk_load(smem_u32(bufs + nb * BUF), a.scores + (long long)next * K, bytes,
                  smem_u32(&s_bar[nb]));
      }
      if (!mbar_wait(smem_u32(&s_bar[cur]), (uint32_t)((it >> 1) & 1), &s_abort)) {
        // a copy did not land in time: report and stop (no trap)
        if (tid == 0 && a.errors) atomicAdd(a.errors, 1);
        return;
      }
    } else {
      const float *src = a.scores + (long long)row * K;
      for (int c = tid; c < K; c += NT) rowv[c] = src[c];
    }
    if (tid == 0) s_nc = 0;
    const int t = row >> 2;
    const int h = row & 3;
    const int flag0 = warp == 0 ? early_flag<MODE>(a, lane, t, h) : -1;

    // forced ids, in increasing order: every valid id when nvp <= 16, else
    // [0, init) then [nvp - local, nvp); each exists when it maps to a column
    if (warp == 0) {
      const bool all = nvp <= kTopK;
      const int nforced = all ? max(nvp, 0) : a.init_blocks + a.local_blocks;
      int id = -1;
      bool ok = false;
      if (lane < nforced && lane < kTopK) {
        id = all ? lane
                 : (lane < a.init_blocks ? lane : nvp - a.local_blocks + (lane - a.init_blocks));
        const int d = id - off;
        ok = id >= 0 && id < nvp && d >= 0 &&
             (scale == 1 ? d < K : (d % scale == 0 && d / scale < K));
      }
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
      if (ok) s_fid[__popc(bal & ((1u << lane) - 1u))] = id;
      if (lane == 0) s_nf = __popc(bal);
    }
    __syncthreads();  // the row buffer and the forced ids are ready
    const int nf = s_nf;
    const int m = kTopK - nf;
    if (tid < nf) {
      const int d = s_fid[tid] - off;
      s_fsc[tid] = rowv[scale == 1 ? d : d / scale];
    }

    // free columns: ids in [init, nvp - local) when nvp > 16, else none
    int c_lo = 0, c_hi = 0;
    if (nvp > kTopK) {
      const int id_lo = a.init_blocks, id_hi = nvp - a.local_blocks;   // [id_lo, id_hi)
      c_lo = id_lo - off <= 0 ? 0 : (id_lo - off + scale - 1) / scale;
      c_hi = id_hi - off <= 0 ? 0 : (id_hi - off + scale - 1) / scale;
      c_hi = min(c_hi, K);
      c_lo = min(c_lo, c_hi);
    }
    // phase 1: per-thread best free entry (score, then lower column)
    float best = 0.0f;
    int bc = -1;
    {
      const float4 *r4 = reinterpret_cast<const float4 *>(rowv);
      const int f_lo = c_lo >> 2, f_hi = (c_hi + 3) >> 2;
      for (int f = f_lo + tid; f < f_hi; f += NT) {
        const float4 x = r4[f];
        const float vv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 4 * f + k;
          if ((unsigned)(c - c_lo) < (unsigned)(c_hi - c_lo) && (bc < 0 || vv[k] > best)) {
            best = vv[k];
            bc = c;
          }
        }
      }
    }
    const unsigned long long tm = bc < 0 ? 0ull : make_key(best, bc * scale + off);

    // tau = m-th largest thread maximum, in two levels: each warp's top m of
    // its lanes' maxima, then the top m of those lists (1 = fewer than m exist)
    {
      unsigned long long my = tm;
      for (int r = 0; r < m; ++r) {
        const unsigned long long w = warp_max_key(my);
        if (lane == 0) s_wtop[warp][r] = w;
        if (w != 0 && my == w) my = 0;
      }
    }
    __syncthreads();
    if (warp == 0) {
      unsigned long long loc[WL];
      unsigned long long lmax = 0;
#pragma unroll
      for (int j = 0; j < WL; ++j) {
        const int k = lane + 32 * j;
        const int w = k / kTopK, r = k % kTopK;
        loc[j] = (w < NW && r < m) ? s_wtop[w][r] : 0ull;
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
          for (int j = 0; j < WL; ++j) {
            if (loc[j] == w) loc[j] = 0;
            lmax = loc[j] > lmax ? loc[j] : lmax;
          }
        }
      }
      if (lane == 0) s_tau = (found < m) ? 1ull : tau;
    }
    __syncthreads();

    // candidates: keys >= tau (only the m threads whose maximum reached tau hold any)
    if (m > 0 && tm != 0 && tm >= s_tau) {
      const unsigned long long tau = s_tau;
      // keys >= tau have scores >= tau's score (tau = 1 has none: -inf)
      const float ts = (tau >> 32) == 0 ? -INFINITY : unord_float((uint32_t)(tau >> 32));
      const float4 *r4 = reinterpret_cast<const float4 *>(rowv);
      const int f_lo = c_lo >> 2, f_hi = (c_hi + 3) >> 2;
      for (int f = f_lo + tid; f < f_hi; f += NT) {
        const float4 x = r4[f];
        const float vv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 4 * f + k;
          if (!(vv[k] >= ts) || (unsigned)(c - c_lo) >= (unsigned)(c_hi - c_lo)) continue;
          const unsigned long long key = make_key(vv[k], c * scale + off);
          if (key >= tau) {
            const int slot = atomicAdd(&s_nc, 1);
            if (slot < CAP) s_cand[slot] = key;
          }
        }
      }
    }
    __syncthreads();
    const int nc = min(s_nc, CAP);
    const int nch = min(nc, m);

    // the m largest candidates: by rank when few, else by rounds in warp 0
    if (nc <= m) {
      if (tid < nc) s_sel[tid] = s_cand[tid];
    } else if (nc <= NT) {
      if (tid < nc) {
        const unsigned long long my = s_cand[tid];
        int rank = 0;
        for (int j = 0; j < nc; ++j) rank += (s_cand[j] > my) ? 1 : 0;
        if (rank < m) s_sel[rank] = my;
      }
    } else if (warp == 0) {
      unsigned long long prev = ~0ull;
      for (int r = 0; r < m; ++r) {
        unsigned long long local = 0;
        for (int j = lane; j < nc; j += 32) {
          const unsigned long long x = s_cand[j];
          if (x < prev && x > local) local = x;
        }
        const unsigned long long w = warp_max_key(local);
        if (lane == 0) s_sel[r] = w;
        prev = w;
      }
    }
    __syncthreads();

    if (warp == 0) {
      const int n = nf + nch;
      int my_id = 0x7FFFFFFF;
      float my_sc = -INFINITY;
      if (lane < nf) {
        my_id = s_fid[lane];
        my_sc = s_fsc[lane];
      } else if (lane < n) {
        my_id = key_id(s_sel[lane - nf]);
        const int d = my_id - off;
        my_sc = rowv[scale == 1 ? d : d / scale];  // raw score bits
      }
      int out_id;
      float out_sc;
      sort_by_id_16(lane, n, my_id, my_sc, out_id, out_sc);
      emit_row<MODE>(a, lane, row, t, h, out_id, out_sc, flag0);
    }
    __syncthreads();  // this row's buffer and scratch may be reused
  }
}

// Warp-per-row select: each warp owns whole rows (row = global warp index,
// then + total warps), so no CTA barrier sits between the phases and every
// row of a launch can be in flight at once.
//   1. forced ids (at most 16, read directly) go to lanes 0..nf-1;
//   2. every lane scans its strided float4s of the free column range and
//      keeps its best entry (score, then lower column);
//   3. tau = m-th largest lane best (m = 16 - nf, rounds of a warp max);
//      only the <= m lanes whose best reaches tau hold keys >= tau, and they
//      rescan their share into a per-warp candidate buffer (a float compare
//      against tau's score filters first);
//   4. the m largest candidates (rounds of a warp max), forced + chosen
//      ordered by id, written or published.
// If a row has more candidates than the buffer holds (only possible with
// very many equal scores), the warp picks the m largest directly from the
// row by rounds instead.  Rows are read with float4 loads when K % 4 == 0 and
// the plane is 16-byte aligned, else with scalar loads.
constexpr int kSelWarps = 4;    // warps (rows in flight) per CTA
constexpr int kCandCap = 256;   // candidates per warp
constexpr int kChunk = 8;       // float4 loads in flight per lane

// Best (score, then lower column) over columns [c_lo, c_hi) owned by this
// lane, and keys >= tau collected into cand[] when collect is set.
template <bool VEC>
__device__ __forceinline__ void scan_row(const float *src, int c_lo, int c_hi, int lane,
                                         float &best, int &bc) {
  if constexpr (VEC) {
    const float4 *r4 = reinterpret_cast<const float4 *>(src);
    const int f_lo = c_lo >> 2, f_hi = (c_hi + 3) >> 2;
    for (int f0 = f_lo + lane; f0 < f_hi; f0 += 32 * kChunk) {
      float4 x[kChunk];
#pragma unroll
      for (int u = 0; u < kChunk; ++u) {
        const int f = f0 + 32 * u;
        x[u] = f < f_hi ? __ldg(r4 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < kChunk; ++u) {
        const int f = f0 + 32 * u;
        const float vv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 4 * f + k;
          if ((unsigned)(c - c_lo) < (unsigned)(c_hi - c_lo) && (bc < 0 || vv[k] > best)) {
            best = vv[k];
            bc = c;
          }
        }
      }
    }
  } else {
    for (int c = c_lo + lane; c < c_hi; c += 32) {
      const float v = __ldg(src + c);
      if (bc < 0 || v > best) {
        best = v;
        bc = c;
      }
    }
  }
}

// Appends this lane's keys >= tau among columns [c_lo, c_hi) to cand.
template <bool VEC>
__device__ __forceinline__ void collect_row(const float *src, int c_lo, int c_hi, int lane,
                                            int scale, int off, unsigned long long tau,
                                            unsigned long long *cand, int *ncand) {
  const float ts = (tau >> 32) == 0 ? -INFINITY : unord_float((uint32_t)(tau >> 32));
  auto offer = [&](float v, int c) {
    if (!(v >= ts)) return;
    const unsigned long long key = make_key(v, c * scale + off);
    if (key >= tau) {
      const int slot = atomicAdd(ncand, 1);
      if (slot < kCandCap) cand[slot] = key;
    }
  };
  if constexpr (VEC) {
    const float4 *r4 = reinterpret_cast<const float4 *>(src);
    const int f_lo = c_lo >> 2, f_hi = (c_hi + 3) >> 2;
    for (int f = f_lo + lane; f < f_hi; f += 32) {
      const float4 x = __ldg(r4 + f);
      const float vv[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = 4 * f + k;
        if ((unsigned)(c - c_lo) < (unsigned)(c_hi - c_lo)) offer(vv[k], c);
      }
    }
  } else {
    for (int c = c_lo + lane; c < c_hi; c += 32) offer(__ldg(src + c), c);
  }
}

// The m largest keys < prev among this lane's free columns, by rounds (the
// exact path for rows whose candidates overflow the buffer).
template <bool VEC>
__device__ void rounds_from_row(const float *src, int c_lo, int c_hi, int lane, int scale,
                                int off, int m, unsigned long long *sel) {
  unsigned long long prev = ~0ull;
  for (int r = 0; r < m; ++r) {
    unsigned long long local = 0;
    for (int c = c_lo + lane; c < c_hi; c += 32) {
      const unsigned long long key = make_key(__ldg(src + c), c * scale + off);
      if (key < prev && key > local) local = key;
    }
    const unsigned long long w = warp_max_key(local);
    if (lane == 0) sel[r] = w;
    prev = w;
    if (w == 0) break;
  }
  (void)VEC;
}

template <int MODE, bool VEC>
__global__ void __launch_bounds__(32 * kSelWarps, 8) select_warp_kernel(const SelectArgs a) {
  __shared__ unsigned long long s_cand[kSelWarps][kCandCap];
  __shared__ unsigned long long s_sel[kSelWarps][kTopK];
  __shared__ int s_nc[kSelWarps];

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int K = a.K;
  const int rows = a.T * 4;
  const int scale = a.index_scale, off = a.index_offset;
  unsigned long long *cand = s_cand[warp];
  unsigned long long *sel = s_sel[warp];

  for (int row = blockIdx.x * kSelWarps + warp; row < rows; row += gridDim.x * kSelWarps) {
    const int t = row >> 2, h = row & 3;
    const int nvp = __ldg(a.nvp + t);
    const float *src = a.scores + (long long)row * K;
    const int flag0 = early_flag<MODE>(a, lane, t, h);

    // forced ids in increasing order: every valid id when nvp <= 16, else
    // [0, init) then [nvp - local, nvp); lane f < nf holds the f-th
    int fid = 0x7FFFFFFF;
    float fsc = -INFINITY;
    int nf;
    {
      const bool all = nvp <= kTopK;
      const int nforced = all ? max(nvp, 0) : a.init_blocks + a.local_blocks;
      int id = -1, col = 0;
      bool ok = false;
      if (lane < nforced && lane < kTopK) {
        id = all ? lane
                 : (lane < a.init_blocks ? lane : nvp - a.local_blocks + (lane - a.init_blocks));
        const int d = id - off;
        if (scale == 1) {
          col = d;
          ok = id >= 0 && id < nvp && d >= 0 && d < K;
        } else {
          col = d / scale;
          ok = id >= 0 && id < nvp && d >= 0 && d % scale == 0 && col < K;
        }
      }
      const float v = ok ? __ldg(src + col) : 0.0f;
      const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
      nf = __popc(bal);
      // move entry of lane L (pos p) to lane p
      const int pos = __popc(bal & ((1u << lane) - 1u));
      for (int p = 0; p < nf; ++p) {
        const int srcl = __fns(bal, 0, p + 1);
        const int i2 = __shfl_sync(0xFFFFFFFFu, id, srcl);
        const float v2 = __shfl_sync(0xFFFFFFFFu, v, srcl);
        if (lane == p) {
          fid = i2;
          fsc = v2;
        }
      }
      (void)pos;
    }
    const int m = kTopK - nf;

    // free columns: ids in [init, nvp - local) when nvp > 16, else none
    int c_lo = 0, c_hi = 0;
    if (nvp > kTopK) {
      const int id_lo = a.init_blocks, id_hi = nvp - a.local_blocks;
      c_lo = id_lo - off <= 0 ? 0 : (id_lo - off + scale - 1) / scale;
      c_hi = id_hi - off <= 0 ? 0 : (id_hi - off + scale - 1) / scale;
      c_hi = min(c_hi, K);
      c_lo = min(c_lo, c_hi);
    }
    float best = 0.0f;
    int bc = -1;
    scan_row<VEC>(src, c_lo, c_hi, lane, best, bc);
    const unsigned long long tm = bc < 0 ? 0ull : make_key(best, bc * scale + off);

    // tau = m-th largest lane best (1 = fewer than m lanes hold an entry)
    unsigned long long tau = 0;
    {
      unsigned long long my = tm;
      int found = 0;
      for (int r = 0; r < m; ++r) {
        const unsigned long long w = warp_max_key(my);
        if (w == 0) break;
        tau = w;
        ++found;
        if (my == w) my = 0;
      }
      if (found < m) tau = 1;
    }
    if (lane == 0) s_nc[warp] = 0;
    __syncwarp();
    if (m > 0 && tm != 0 && tm >= tau)
      collect_row<VEC>(src, c_lo, c_hi, lane, scale, off, tau, cand, &s_nc[warp]);
    __syncwarp();
    const int nc = s_nc[warp];
    int nch = 0;
    if (m > 0) {
      if (nc > kCandCap) {
        rounds_from_row<VEC>(src, c_lo, c_hi, lane, scale, off, m, sel);
        nch = 0;
        __syncwarp();
        for (int r = 0; r < m; ++r) nch += sel[r] != 0 ? 1 : 0;
      } else if (nc <= m) {
        for (int j = lane; j < nc; j += 32) sel[j] = cand[j];
        nch = nc;
      } else {
        // rank each candidate among the others (nc <= 256: 8 per lane)
        for (int j = lane; j < nc; j += 32) {
          const unsigned long long my = cand[j];
          int rank = 0;
          for (int i = 0; i < nc; ++i) rank += (cand[i] > my) ? 1 : 0;
          if (rank < m) sel[rank] = my;
        }
        nch = m;
      }
    }
    __syncwarp();
    const int n = nf + nch;
    int my_id = fid;
    float my_sc = fsc;
    if (lane >= nf && lane < n) {
      my_id = key_id(sel[lane - nf]);
      const int d = my_id - off;
      my_sc = __ldg(src + (scale == 1 ? d : d / scale));  // raw score bits
    }
    int out_id;
    float out_sc;
    sort_by_id_16(lane, n, my_id, my_sc, out_id, out_sc);
    emit_row<MODE>(a, lane, row, t, h, out_id, out_sc, flag0);
    __syncwarp();
  }
}

// Second half of a merge, once lane i < 16 holds entry i of every source in
// ids[s] / scs[s] (id -1 = nothing): union with the maximum score per id,
// the Top16 rule with num_valid_pages, and the output ordered by id.
__device__ __forceinline__ void merge_finish(const MergeArgs &a, int lane, int t, int hl, int nvp,
                                             const int (&ids)[4], const float (&scs)[4],
                                             int *s_idw, float *s_scw) {
  const int hpr = a.heads_per_rank;
  const int ws = a.world_size;
  // keep an entry unless another source holds the same id with a higher
  // score (an exact tie goes to the lower source)
  bool keep[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) keep[s] = lane < kTopK && ids[s] >= 0 && ids[s] < nvp;
  if (ws > 1) {
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
      if (s2 >= ws) break;
      for (int j = 0; j < kTopK; ++j) {
        const int id2 = __shfl_sync(0xFFFFFFFFu, ids[s2], j);
        const float sc2 = __shfl_sync(0xFFFFFFFFu, scs[s2], j);
#pragma unroll
        for (int s = 0; s < 4; ++s) {
          if (s == s2 || !keep[s] || ids[s] != id2) continue;
          if (sc2 > scs[s] || (sc2 == scs[s] && s2 < s)) keep[s] = false;
        }
      }
    }
  }
  int total = 0, nforced = 0;
  bool forced[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    forced[s] = keep[s] && forced_id(ids[s], nvp, a.init_blocks, a.local_blocks);
    total += __popc(__ballot_sync(0xFFFFFFFFu, keep[s]));
    nforced += __popc(__ballot_sync(0xFFFFFFFFu, forced[s]));
  }
  bool sel[4];
  if (total <= kTopK) {
#pragma unroll
    for (int s = 0; s < 4; ++s) sel[s] = keep[s];
  } else {
    // m best free entries by (score desc, id asc)
    const int m = kTopK - min(nforced, kTopK);
    unsigned long long key[4];
#pragma unroll
    for (int s = 0; s < 4; ++s) key[s] = (keep[s] && !forced[s]) ? make_key(scs[s], ids[s]) : 0ull;
    int rank[4] = {0, 0, 0, 0};
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2) {
      if (s2 >= ws) break;
      for (int j = 0; j < kTopK; ++j) {
        const unsigned long long k2 = __shfl_sync(0xFFFFFFFFu, key[s2], j);
#pragma unroll
        for (int s = 0; s < 4; ++s) rank[s] += (k2 > key[s]) ? 1 : 0;
      }
    }
#pragma unroll
    for (int s = 0; s < 4; ++s) sel[s] = forced[s] || (key[s] != 0 && rank[s] < m);
  }
  // compact the selected entries (at most 16) and order them by id
  int n = 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, sel[s]);
    if (sel[s]) {
      const int pos = n + __popc(bal & ((1u << lane) - 1u));
      if (pos < kTopK) {
        s_idw[pos] = ids[s];
        s_scw[pos] = scs[s];
      }
    }
    n += __popc(bal);
  }
  n = min(n, kTopK);
  __syncwarp();
  int my_id = 0x7FFFFFFF;
  float my_sc = -INFINITY;
  if (lane < n) {
    my_id = s_idw[lane];
    my_sc = s_scw[lane];
  }
  int out_id;
  float out_sc;
  sort_by_id_16(lane, n, my_id, my_sc, out_id, out_sc);
  if (lane < kTopK) {
    const long long o = ((long long)t * hpr + hl) * kTopK + lane;
    a.out_scores[o] = out_sc;
    a.out_ids[o] = out_id;
  }
}

// One warp per (token, owned head).  Lane i < 16 holds entry i of every
// source row (at most 4 sources), so the union, the per-id maximum and the
// ranking are done with shuffles; the result is compacted through shared
// memory and ordered by id.
__global__ void __launch_bounds__(128) merge_kernel(const MergeArgs a) {
  __shared__ int s_id[4][kTopK];
  __shared__ float s_sc[4][kTopK];
  // a scorer launched next with early start may begin its set-up now: it
  // reads nothing this kernel writes before waiting for it
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + warp;
  const int hpr = a.heads_per_rank;
  if (item >= a.T * hpr) return;
  const int t = item / hpr, hl = item % hpr;
  const int nvp = a.nvp[t];
  const int ws = a.world_size;

  int ids[4];
  float scs[4];
  unsigned read_mask = 0;
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    ids[s] = -1;
    scs[s] = -INFINITY;
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
    if (lane < kTopK) {
      (void)ld_acquire_gpu(row + 32);  // order this lane's reads after the flag
      scs[s] = __int_as_float(row[lane]);
      ids[s] = row[kTopK + lane];
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

  merge_finish(a, lane, t, hl, nvp, ids, scs, s_id[warp], s_sc[warp]);
}

// Owner merge of tagged rows: a source row has arrived when all 32 words
// carry the owner's expected generation + 1 (the counter advances on every
// merge).  Polls are bounded by spin_limit and the wait timeout.
__global__ void __launch_bounds__(128) merge_tagged_kernel(const MergeArgs a) {
  __shared__ int s_id[4][kTopK];
  __shared__ float s_sc[4][kTopK];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + warp;
  const int hpr = a.heads_per_rank;
  if (item >= a.T * hpr) return;
  const int t = item / hpr, hl = item % hpr;
  const int nvp = a.nvp[t];
  const int ws = a.world_size;

  int ids[4];
  float scs[4];
#pragma unroll
  for (int s = 0; s < 4; ++s) {
    ids[s] = -1;
    scs[s] = -INFINITY;
    if (s >= ws) continue;
    const long long r = (((long long)a.slot * ws + s) * hpr + hl) * a.capacity + t;
    int *e = a.expected + r;  // same [slot][src][hl][t] layout as the rows
    unsigned want = 0;
    if (lane == 0) {
      want = (unsigned)*e + 1u;
      *e = (int)want;
    }
    want = __shfl_sync(0xFFFFFFFFu, want, 0);
    const unsigned long long *row = a.recv64 + r * 32;
    const unsigned long long t0 = globaltimer_ns();
    bool arrived = false;
    unsigned long long w = 0;
    for (long long it = 0; it < a.spin_limit; ++it) {
      w = ld_relaxed_gpu_u64(row + lane);
      if (__all_sync(0xFFFFFFFFu, (unsigned)(w >> 32) == want)) {
        arrived = true;
        break;
      }
      if ((it & 255) == 255 && globaltimer_ns() - t0 > kWaitTimeoutNs) break;
    }
    if (!arrived) {
      if (lane == 0) atomicAdd(a.errors, 1);
      continue;
    }
    const unsigned payload = (unsigned)w;
    const unsigned idw = __shfl_sync(0xFFFFFFFFu, payload, (lane & 15) + kTopK);
    if (lane < kTopK) {
      scs[s] = __uint_as_float(payload);
      ids[s] = (int)idw;
    }
  }
  merge_finish(a, lane, t, hl, nvp, ids, scs, s_id[warp], s_sc[warp]);
}

}  // namespace

constexpr int kWarpRowMaxK = 2048;  // rows up to this long: one warp per row
constexpr int kLargeK = 12288;

cudaError_t select_prepare() {
  const int big = 2 * kLargeK * 4;
  cudaError_t e = cudaFuncSetAttribute(select_block_kernel<256, kLargeK, kEmitPlain>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, big);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(select_block_kernel<256, kLargeK, kEmitLegacy>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize, big);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(select_block_kernel<256, kLargeK, kEmitTagged>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, big);
}

cudaError_t launch_select(const SelectArgs &a, int mode, int sm_count, cudaStream_t stream) {
  const int rows = a.T * 4;
  if (rows == 0) return cudaSuccess;
  if (a.K > kWarpRowMaxK) {
    // long rows: two CTAs per SM, each double-buffering rows in shared memory
    const size_t smem = 2 * (size_t)kLargeK * 4;
    const int grid = rows < 2 * sm_count ? rows : 2 * sm_count;
    if (mode == kEmitLegacy)
      select_block_kernel<256, kLargeK, kEmitLegacy><<<grid, 256, smem, stream>>>(a);
    else if (mode == kEmitTagged)
      select_block_kernel<256, kLargeK, kEmitTagged><<<grid, 256, smem, stream>>>(a);
    else
      select_block_kernel<256, kLargeK, kEmitPlain><<<grid, 256, smem, stream>>>(a);
    return cudaGetLastError();
  }
  // short rows: one warp per row; float4 loads when every row is 16-byte aligned
  const bool vec = (a.K % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 15u) == 0);
  const int grid = (rows + kSelWarps - 1) / kSelWarps;
  const int threads = 32 * kSelWarps;
  if (mode == kEmitLegacy) {
    if (vec) select_warp_kernel<kEmitLegacy, true><<<grid, threads, 0, stream>>>(a);
    else select_warp_kernel<kEmitLegacy, false><<<grid, threads, 0, stream>>>(a);
  } else if (mode == kEmitTagged) {
    if (vec) select_warp_kernel<kEmitTagged, true><<<grid, threads, 0, stream>>>(a);
    else select_warp_kernel<kEmitTagged, false><<<grid, threads, 0, stream>>>(a);
  } else {
    if (vec) select_warp_kernel<kEmitPlain, true><<<grid, threads, 0, stream>>>(a);
    else select_warp_kernel<kEmitPlain, false><<<grid, threads, 0, stream>>>(a);
  }
  return cudaGetLastError();
}

cudaError_t launch_merge(const MergeArgs &a, bool tagged, cudaStream_t stream) {
  const int items = a.T * a.heads_per_rank;
  if (items == 0) return cudaSuccess;
  if (tagged) merge_tagged_kernel<<<(items + 3) / 4, 128, 0, stream>>>(a);
  else merge_kernel<<<(items + 3) / 4, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace icp
