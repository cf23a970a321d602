// icp_select.cu - Top16 select; its outputs (plain lists, legacy and tagged
// receive rows, prefill carrier rows); the owner merges.
//
// Top16 rule (msa_icp_topk_select_publish with the forced blocks of
// prepare_msa_icp_indexer): valid ids are c * index_scale + index_offset <
// num_valid_pages[t].  If num_valid_pages[t] <= 16 every valid id is kept;
// otherwise ids in [0, init) and [nvp - local, nvp) are forced and the other
// slots go to the best remaining ids by (score descending, id ascending).
// Output: ids ascending with their raw scores, then (-1, -inf) padding.
//
// Select kernels by row length: rows of at most 256 columns with the row in
// registers; one warp per row up to 2048 columns; longer rows on a CTA of
// four warps.  The steps they share are described below, above kSelWarps.
#include "icp_device.cuh"
#include "icp_internal.h"

namespace icp {
namespace {

constexpr int kRowWords = 33;

// Bounded poll of a ready flag until it equals `want` (acquire loads).
// Returns false after spin_limit polls or kWaitTimeoutNs, whichever comes
// first; the global timer is first read after 256 polls (reading it can
// stall the warp, and most polls succeed at once).
__device__ __forceinline__ bool poll_flag(const int *flag, int want, long long spin_limit) {
  unsigned long long t0 = 0;
  for (long long it = 0; it < spin_limit; ++it) {
    if (ld_acquire_gpu(flag) == want) return true;
    if ((it & 255) == 255) {
      const unsigned long long now = globaltimer_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kWaitTimeoutNs) return false;
    }
  }
  return false;
}

// Where a selected row goes: the plain output arrays, a legacy receive row
// (bounded wait for a free row, 32 data words, release-stored ready flag), a
// tagged receive row (32 int64 words of generation << 32 | word, the
// generation taken from the publisher's counter for (slot, head, token)), or
// a prefill carrier row (the 32 data words, no flag: the caller's exchange
// orders it), row ((h / hpr) * T + t) * hpr + h % hpr of the carrier.
enum EmitMode { kEmitPlain = 0, kEmitLegacy = 1, kEmitTagged = 2, kEmitCarrier = 3 };

// heads_per_rank is 4 / world_size (4, 2 or 1), so dividing by it is a
// shift and the remainder a mask.
__device__ __forceinline__ int hpr_shift(int hpr) { return hpr == 4 ? 2 : (hpr == 2 ? 1 : 0); }

// Address of the legacy receive row (t, h) of this publish.
__device__ __forceinline__ int *legacy_row(const SelectArgs &a, int t, int h) {
  const int hpr = a.heads_per_rank;
  const long long r =
      (((long long)a.slot * a.world_size + a.rank) * hpr + (h & (hpr - 1))) * a.capacity + t;
  return reinterpret_cast<int *>(a.recv_bases[h >> hpr_shift(hpr)]) + r * kRowWords;
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
  } else if constexpr (MODE == kEmitCarrier) {
    const int hpr = a.heads_per_rank;
    int *dst =
        a.carrier + (((long long)(h >> hpr_shift(hpr)) * a.T + t) * hpr + (h & (hpr - 1))) * 32;
    if (lane < kTopK) {
      dst[lane] = __float_as_int(out_sc);
      dst[kTopK + lane] = out_id;
    }
  } else {
    const int hpr = a.heads_per_rank;
    const long long r =
        (((long long)a.slot * a.world_size + a.rank) * hpr + (h & (hpr - 1))) * a.capacity + t;
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
          reinterpret_cast<unsigned long long *>(a.recv_bases[h >> hpr_shift(hpr)]) + r * 32;
      st_relaxed_gpu_u64(dst + lane, word);
    }
  }
}

// Select.  Every non-forced valid score becomes a unique 64-bit key (score
// order, then the lower id), and a row's m = 16 - (forced ids) free slots go
// to its m largest keys.  Rows up to 2048 columns: one warp per row; longer
// rows: kRowWarps warps per row, each taking the top m of its share, then
// the top m of their lists.  A warp takes the top m of its columns so:
//   1. every lane scans its strided float4s (or elements), keeps its best key
//      (the vector kernels keep only its score: step 2 needs no more) and
//      records each float4's largest value in shared memory; the first
//      batch of loads is issued before num_valid_pages is known;
//   2. tau = a lower bound of the m-th largest lane best (rounds of a warp
//      max on the score half); only lanes whose best reaches tau can hold
//      keys >= tau;
//   3. those lanes re-read the float4s whose recorded maximum reaches tau's
//      score, all at once, and append the keys >= tau to a candidate buffer;
//   4. the m largest candidates, placed by rank, in order.
// If the candidates overflow the buffer (only with very many equal scores),
// the warp takes the m largest directly from its columns by rounds.  Rows
// are read with float4 loads when K % 4 == 0 and the plane is 16-byte
// aligned, else with scalar loads (and a plain rescan in step 3).
constexpr int kSelWarps = 4;     // warps (rows in flight) per CTA, rows <= 2048 columns
constexpr int kRowWarps = 4;     // warps per row, longer rows
constexpr int kChunk = 8;        // float4 loads in flight per lane
constexpr int kCandCap = 128;    // candidates per warp
constexpr int kWarpRowMaxK = 2048;  // rows up to this long: one warp per row
constexpr int kLongRowMaxK = 12287;  // the widest plane
// float4s per lane: 2048 / 4 / 32 for a warp row, ceil(12287 / 4 / 128) for a long row
constexpr int kWarpRowChunks = 16;
constexpr int kLongRowChunks = 24;
static_assert(kWarpRowChunks * 32 >= kWarpRowMaxK / 4, "warp-row chunk record too small");

// Lane holding the (r+1)-th set bit of mask (r < popc(mask)): a five-step
// search over halves of the remaining bit range.
__device__ __forceinline__ int nth_set_lane(unsigned mask, int r) {
  int pos = 0;
#pragma unroll
  for (int w = 16; w > 0; w >>= 1) {
    const int c = __popc((mask >> pos) & ((1u << w) - 1u));
    if (r >= c) {
      r -= c;
      pos += w;
    }
  }
  return pos;
}

// Forced ids of a row in increasing order: every valid id when nvp <= 16,
// else [0, init) then [nvp - local, nvp), each kept only when it is a valid
// id of a column of the plane.  Every lane gets nf; with keep, lane q < nf
// also gets the q-th id and its raw score.
struct Forced {
  int fid;
  float fsc;
  int nf;
};

__device__ __forceinline__ Forced forced_ids(const SelectArgs &a, const float *src, int nvp,
                                             int lane, bool keep) {
  const int scale = a.index_scale, off = a.index_offset;
  const bool all = nvp <= kTopK;
  const int nforced = all ? max(nvp, 0) : a.init_blocks + a.local_blocks;
  int id = -1, col = 0;
  bool ok = false;
  if (lane < nforced && lane < kTopK) {
    id = all ? lane : (lane < a.init_blocks ? lane : nvp - a.local_blocks + (lane - a.init_blocks));
    const int d = id - off;
    if (scale == 1) {
      col = d;
      ok = id >= 0 && id < nvp && d >= 0 && d < a.K;
    } else {
      col = d / scale;
      ok = id >= 0 && id < nvp && d >= 0 && d % scale == 0 && col < a.K;
    }
  }
  const unsigned bal = __ballot_sync(0xFFFFFFFFu, ok);
  Forced f{0x7FFFFFFF, -INFINITY, __popc(bal)};
  if (keep) {
    const float v = ok ? __ldg(src + col) : 0.0f;
    // lane q < nf takes the entry of the lane holding the (q+1)-th set bit
    const int srcl = nth_set_lane(bal, lane < f.nf ? lane : 0);
    const int i2 = __shfl_sync(0xFFFFFFFFu, id, srcl);
    const float v2 = __shfl_sync(0xFFFFFFFFu, v, srcl);
    if (lane < f.nf) {
      f.fid = i2;
      f.fsc = v2;
    }
  }
  return f;
}

// First free column: ids from init on (valid whenever nvp > 16).
__device__ __forceinline__ int free_lo(const SelectArgs &a) {
  const int scale = a.index_scale, off = a.index_offset;
  const int d = a.init_blocks - off;
  if (d <= 0) return 0;
  return min(scale == 1 ? d : (d + scale - 1) / scale, a.K);
}

// Free columns of a row: ids in [init, nvp - local) when nvp > 16, else none.
__device__ __forceinline__ void free_range(const SelectArgs &a, int nvp, int &c_lo, int &c_hi) {
  const int scale = a.index_scale, off = a.index_offset;
  c_lo = 0;
  c_hi = 0;
  if (nvp > kTopK) {
    const int id_hi = nvp - a.local_blocks;
    const int d = id_hi - off;
    c_hi = d <= 0 ? 0 : (scale == 1 ? d : (d + scale - 1) / scale);
    c_hi = min(c_hi, a.K);
    c_lo = min(free_lo(a), c_hi);
  }
}

// A lower bound of the m-th largest of the lanes' keys (0 = no key): the
// score half of that key with the id half 0, found by rounds of a warp max
// over the score halves (lanes tied on a score leave together); 1 when fewer
// than m lanes hold a key, 0 when m <= 0.  Every key >= the m-th largest
// lane key is >= the bound.
__device__ __forceinline__ unsigned long long tau_lower_bound(unsigned long long k, int m) {
  if (m <= 0) return 0ull;
  uint32_t hi = (uint32_t)(k >> 32);  // real keys have a non-zero score half
  int found = 0;
  for (;;) {
    const uint32_t cur = __reduce_max_sync(0xFFFFFFFFu, hi);
    if (cur == 0u) return 1ull;
    found += __popc(__ballot_sync(0xFFFFFFFFu, hi == cur));
    if (found >= m) return (unsigned long long)cur << 32;
    if (hi == cur) hi = 0u;
  }
}

// The m largest keys < prev among this lane's free columns, by rounds (the
// exact path when the candidate buffer overflows).  Covers columns first,
// first + stride, ... for the scalar layout, and element indices
// 4 f .. 4 f + 3 for f = f_lo + first + j * stride with float4 reads.
template <bool VEC>
__device__ void rounds_from_row(const float *src, int c_lo, int c_hi, int lane, int first,
                                int stride, int scale, int off, int m, unsigned long long *sel) {
  unsigned long long prev = ~0ull;
  for (int r = 0; r < m; ++r) {
    unsigned long long local = 0;
    auto look = [&](int c) {
      if ((unsigned)(c - c_lo) >= (unsigned)(c_hi - c_lo)) return;
      const unsigned long long key = make_key(__ldg(src + c), c * scale + off);
      if (key < prev && key > local) local = key;
    };
    if constexpr (VEC) {
      const int f_lo = c_lo >> 2, f_hi = (c_hi + 3) >> 2;
      for (int f = f_lo + first; f < f_hi; f += stride)
        for (int k = 0; k < 4; ++k) look(4 * f + k);
    } else {
      for (int c = c_lo + first; c < c_hi; c += stride) look(c);
    }
    const unsigned long long w = warp_max_key(local);
    if (lane == 0) sel[r] = w;
    prev = w;
    if (w == 0) break;
  }
}

// kChunk float4 loads at f0, f0 + stride, ... (those below f_end).
__device__ __forceinline__ void load_batch(const float4 *r4, int f0, int stride, int f_end,
                                           float4 (&x)[kChunk]) {
#pragma unroll
  for (int u = 0; u < kChunk; ++u) {
    const int f = f0 + stride * u;
    x[u] = f < f_end ? __ldg(r4 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
}

// Shared state of one warp's selection: its candidate buffer and count,
// and a column of recorded float4 maxima per lane (entry j at cm[32 j]).
struct WarpScratch {
  unsigned long long *cand;
  int *nc;
  float *cm;
};

// Candidates (keys >= tau) from the m largest: placed by rank into sel
// (descending), or taken by rounds from the columns on overflow.  Returns
// their number; sel is readable after __syncwarp.
template <bool VEC>
__device__ __forceinline__ int place_candidates(const float *src, int c_lo, int c_hi, int first,
                                                int stride, int scale, int off, int m, int lane,
                                                const WarpScratch &w, unsigned long long *sel) {
  __syncwarp();
  const int nc = *w.nc;
  if (nc > kCandCap) {
    rounds_from_row<VEC>(src, c_lo, c_hi, lane, first, stride, scale, off, m, sel);
    __syncwarp();
    int n = 0;
    while (n < m && sel[n] != 0ull) ++n;
    return n;
  }
  for (int j = lane; j < nc; j += 32) {
    const unsigned long long my = w.cand[j];
    int rank = 0;
    for (int i = 0; i < nc; ++i) rank += (w.cand[i] > my) ? 1 : 0;
    if (rank < m) sel[rank] = my;
  }
  return min(nc, m);
}

// Appends key (v, c) to the candidates when it is >= tau.
__device__ __forceinline__ void offer_key(float v, int c, float ts, unsigned long long tau,
                                          int scale, int off, const WarpScratch &w) {
  if (!(v >= ts)) return;
  const unsigned long long key = make_key(v, c * scale + off);
  if (key >= tau) {
    const int slot = atomicAdd(w.nc, 1);
    if (slot < kCandCap) w.cand[slot] = key;
  }
}

// This warp's m largest keys among float4 chunks f_lo + first + j * stride
// of the free range [c_lo, c_hi), into sel (descending; readable after
// __syncwarp); returns how many.  x holds the lane's first batch, loaded
// from the same chunks before the range was known (and is reused for the
// later batches).
__device__ __forceinline__ int warp_top_m_vec(const float *src, float4 (&x)[kChunk],
                                              int c_lo, int c_hi, int first, int stride,
                                              int scale, int off, int m, int lane,
                                              const WarpScratch &w, unsigned long long *sel) {
  if (m <= 0) return 0;
  const float4 *r4 = reinterpret_cast<const float4 *>(src);
  const int f_lo = c_lo >> 2, f_hi = (c_hi + 3) >> 2;
  const int f_first = f_lo + first;
  // 1. scan: the lane's largest score in the range (tau only needs the
  //    score half of the lane's best key), and every chunk's largest value
  //    into cm; only the range's first and last float4 can hold columns
  //    outside it, and every float4 of [f_lo, f_hi) holds one inside
  float best = -INFINITY;
  const bool has = c_lo < c_hi && f_first < f_hi;
  int nj = 0;
  for (int f0 = f_first; f0 < f_hi; f0 += stride * kChunk) {
    if (f0 != f_first) load_batch(r4, f0, stride, f_hi, x);
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      const int f = f0 + stride * u;
      if (f >= f_hi) break;
      const float m4 = fmaxf(fmaxf(x[u].x, x[u].y), fmaxf(x[u].z, x[u].w));
      w.cm[32 * nj++] = m4;
      if (f == f_lo || f == f_hi - 1) {
        const float vv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 4 * f + k;
          if ((unsigned)(c - c_lo) < (unsigned)(c_hi - c_lo)) best = fmaxf(best, vv[k]);
        }
      } else {
        best = fmaxf(best, m4);
      }
    }
  }
  // 2. tau
  const unsigned long long tm = has ? (unsigned long long)ord_float(best) << 32 : 0ull;
  const unsigned long long tau = tau_lower_bound(tm, m);
  if (lane == 0) *w.nc = 0;
  __syncwarp();
  // 3. the chunks whose maximum reaches tau's score offer their keys: from
  //    x when the lane's chunks all came in the first batch (x still holds
  //    them), else re-read four at a time
  if (tm != 0ull && tm >= tau && nj <= kChunk) {
    const float ts = (tau >> 32) == 0 ? -INFINITY : unord_float((uint32_t)(tau >> 32));
#pragma unroll
    for (int u = 0; u < kChunk; ++u) {
      if (u >= nj) break;
      if (!(w.cm[32 * u] >= ts)) continue;
      const int f = f_first + stride * u;
      const float vv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = 4 * f + k;
        if ((unsigned)(c - c_lo) < (unsigned)(c_hi - c_lo)) offer_key(vv[k], c, ts, tau, scale, off, w);
      }
    }
  } else if (tm != 0ull && tm >= tau) {
    const float ts = (tau >> 32) == 0 ? -INFINITY : unord_float((uint32_t)(tau >> 32));
    unsigned mask = 0;
    for (int j = 0; j < nj; ++j)
      if (w.cm[32 * j] >= ts) mask |= 1u << j;
    while (mask != 0u) {
      int fq[4];
      float4 y[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        fq[q] = -1;
        if (mask != 0u) {
          fq[q] = f_first + stride * (__ffs(mask) - 1);
          mask &= mask - 1u;
        }
      }
#pragma unroll
      for (int q = 0; q < 4; ++q)
        y[q] = fq[q] >= 0 ? __ldg(r4 + fq[q]) : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        if (fq[q] < 0) continue;
        const float vv[4] = {y[q].x, y[q].y, y[q].z, y[q].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 4 * fq[q] + k;
          if ((unsigned)(c - c_lo) < (unsigned)(c_hi - c_lo)) offer_key(vv[k], c, ts, tau, scale, off, w);
        }
      }
    }
  }
  // 4. the m largest candidates
  return place_candidates<true>(src, c_lo, c_hi, first, stride, scale, off, m, lane, w, sel);
}

// Same for the scalar layout (columns c_lo + first + j * stride), with a
// plain rescan of the lane's columns in step 3.
__device__ __forceinline__ int warp_top_m_scalar(const float *src, int c_lo, int c_hi, int first,
                                                 int stride, int scale, int off, int m, int lane,
                                                 const WarpScratch &w, unsigned long long *sel) {
  if (m <= 0) return 0;
  float best = 0.0f;
  int bc = -1;
  for (int c = c_lo + first; c < c_hi; c += stride) {
    const float v = __ldg(src + c);
    if (bc < 0 || v > best) {
      best = v;
      bc = c;
    }
  }
  const unsigned long long tm = bc < 0 ? 0ull : make_key(best, bc * scale + off);
  const unsigned long long tau = tau_lower_bound(tm, m);
  if (lane == 0) *w.nc = 0;
  __syncwarp();
  if (tm != 0ull && tm >= tau) {
    const float ts = (tau >> 32) == 0 ? -INFINITY : unord_float((uint32_t)(tau >> 32));
    for (int c = c_lo + first; c < c_hi; c += stride)
      offer_key(__ldg(src + c), c, ts, tau, scale, off, w);
  }
  return place_candidates<false>(src, c_lo, c_hi, first, stride, scale, off, m, lane, w, sel);
}

// Raw score of a selected key: the key's score half is exact for every
// score but a zero, whose sign is read back from the row.
__device__ __forceinline__ float key_score(unsigned long long k, const float *row_src, int scale,
                                           int off) {
  const uint32_t o = (uint32_t)(k >> 32);
  if (o != 0x80000000u) return unord_float(o);
  const int d = key_id(k) - off;
  return __ldg(row_src + (scale == 1 ? d : d / scale));
}

// Rows of at most 256 columns with float4 loads: a lane's share of a row
// (two float4s) stays in registers, so the candidate pass re-reads nothing,
// and the loads of the warp's next row (with its num_valid_pages) are in
// flight while the current row is selected.
constexpr int kShortMaxK = 256;
constexpr int kShortF4 = kShortMaxK / 4 / 32;

template <int MODE>
__global__ void __launch_bounds__(32 * kSelWarps, 8) select_short_kernel(const SelectArgs a) {
  __shared__ unsigned long long s_cand[kSelWarps][kCandCap];
  __shared__ unsigned long long s_sel[kSelWarps][kTopK];
  __shared__ int s_nc[kSelWarps];
  // under programmatic dependent launch: wait for the preceding kernel
  // (the scorer) before reading its scores, then let dependents launch
  pdl_wait();
  pdl_launch_dependents();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = a.T * 4;
  const int scale = a.index_scale, off = a.index_offset;
  const int nf4 = a.K >> 2;
  unsigned long long *sel = s_sel[warp];
  const WarpScratch ws{s_cand[warp], &s_nc[warp], nullptr};
  const int step = gridDim.x * kSelWarps;

  float4 cur[kShortF4], nxt[kShortF4];
  int nvp_cur = 0, nvp_nxt = 0;
  auto load_row = [&](int row, float4 (&x)[kShortF4], int &nvp) {
    const float4 *r4 = reinterpret_cast<const float4 *>(a.scores + (long long)row * a.K);
#pragma unroll
    for (int u = 0; u < kShortF4; ++u) {
      const int f = lane + 32 * u;
      x[u] = f < nf4 ? __ldg(r4 + f) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
    nvp = __ldg(a.nvp + (row >> 2));
  };

  int row = blockIdx.x * kSelWarps + warp;
  if (row < rows) load_row(row, cur, nvp_cur);
  for (; row < rows; row += step) {
    if (row + step < rows) load_row(row + step, nxt, nvp_nxt);
    const int t = row >> 2, h = row & 3;
    const int nvp = nvp_cur;
    const float *src = a.scores + (long long)row * a.K;
    const int flag0 = early_flag<MODE>(a, lane, t, h);
    const Forced f = forced_ids(a, src, nvp, lane, true);
    const int m = kTopK - f.nf;
    int c_lo, c_hi;
    free_range(a, nvp, c_lo, c_hi);
    // the lane's largest score among its free columns 4 (lane + 32 u) + k
    // (tau only needs the score half of the lane's best key)
    float best = -INFINITY;
    bool has = false;
#pragma unroll
    for (int u = 0; u < kShortF4; ++u) {
      const float vv[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int c = 4 * (lane + 32 * u) + k;
        const bool in = (unsigned)(c - c_lo) < (unsigned)(c_hi - c_lo);
        best = fmaxf(best, in ? vv[k] : -INFINITY);
        has |= in;
      }
    }
    const unsigned long long tm = has ? (unsigned long long)ord_float(best) << 32 : 0ull;
    const unsigned long long tau = tau_lower_bound(tm, m);
    if (lane == 0) *ws.nc = 0;
    __syncwarp();
    if (m > 0 && tm != 0ull && tm >= tau) {
      const float ts = (tau >> 32) == 0 ? -INFINITY : unord_float((uint32_t)(tau >> 32));
#pragma unroll
      for (int u = 0; u < kShortF4; ++u) {
        const float vv[4] = {cur[u].x, cur[u].y, cur[u].z, cur[u].w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const int c = 4 * (lane + 32 * u) + k;
          if ((unsigned)(c - c_lo) < (unsigned)(c_hi - c_lo)) offer_key(vv[k], c, ts, tau, scale, off, ws);
        }
      }
    }
    const int nch = m > 0 ? place_candidates<true>(src, c_lo, c_hi, lane, 32, scale, off, m, lane, ws, sel) : 0;
    __syncwarp();
    const int n = f.nf + nch;
    int my_id = f.fid;
    float my_sc = f.fsc;
    if (lane >= f.nf && lane < n) {
      const unsigned long long k = sel[lane - f.nf];
      my_id = key_id(k);
      my_sc = key_score(k, src, scale, off);
    }
    int out_id;
    float out_sc;
    sort_by_id_16(lane, n, my_id, my_sc, out_id, out_sc, reinterpret_cast<int *>(sel),
                  reinterpret_cast<float *>(sel) + kTopK);
    emit_row<MODE>(a, lane, row, t, h, out_id, out_sc, flag0);
    __syncwarp();
#pragma unroll
    for (int u = 0; u < kShortF4; ++u) cur[u] = nxt[u];
    nvp_cur = nvp_nxt;
  }
}

// Rows up to 2048 columns: one warp per row (row = global warp index, then
// + total warps), no CTA barrier.
template <int MODE, bool VEC>
__global__ void __launch_bounds__(32 * kSelWarps, 8) select_warp_kernel(const SelectArgs a) {
  __shared__ unsigned long long s_cand[kSelWarps][kCandCap];
  __shared__ unsigned long long s_sel[kSelWarps][kTopK];
  __shared__ float s_cm[kSelWarps][kWarpRowChunks * 32];
  __shared__ int s_nc[kSelWarps];
  // under programmatic dependent launch: wait for the preceding kernel
  // (the scorer) before reading its scores, then let dependents launch
  pdl_wait();
  pdl_launch_dependents();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = a.T * 4;
  const int scale = a.index_scale, off = a.index_offset;
  unsigned long long *sel = s_sel[warp];
  const WarpScratch ws{s_cand[warp], &s_nc[warp], &s_cm[warp][lane]};
  const int f_start = (free_lo(a) >> 2) + lane;

  for (int row = blockIdx.x * kSelWarps + warp; row < rows; row += gridDim.x * kSelWarps) {
    const int t = row >> 2, h = row & 3;
    const float *src = a.scores + (long long)row * a.K;
    float4 x0[kChunk];
    if constexpr (VEC) load_batch(reinterpret_cast<const float4 *>(src), f_start, 32, a.K >> 2, x0);
    const int nvp = __ldg(a.nvp + t);
    const int flag0 = early_flag<MODE>(a, lane, t, h);
    const Forced f = forced_ids(a, src, nvp, lane, true);
    const int m = kTopK - f.nf;
    int c_lo, c_hi;
    free_range(a, nvp, c_lo, c_hi);
    int nch;
    if constexpr (VEC)
      nch = warp_top_m_vec(src, x0, c_lo, c_hi, lane, 32, scale, off, m, lane, ws, sel);
    else
      nch = warp_top_m_scalar(src, c_lo, c_hi, lane, 32, scale, off, m, lane, ws, sel);
    __syncwarp();
    const int n = f.nf + nch;
    int my_id = f.fid;
    float my_sc = f.fsc;
    if (lane >= f.nf && lane < n) {
      const unsigned long long k = sel[lane - f.nf];
      my_id = key_id(k);
      my_sc = key_score(k, src, scale, off);
    }
    int out_id;
    float out_sc;
    sort_by_id_16(lane, n, my_id, my_sc, out_id, out_sc, reinterpret_cast<int *>(sel),
                  reinterpret_cast<float *>(sel) + kTopK);
    emit_row<MODE>(a, lane, row, t, h, out_id, out_sc, flag0);
    __syncwarp();
  }
}

// Rows longer than 2048 columns: one CTA of RW warps per row (grid-stride
// over the rows).  Warp w takes the top m of the float4 chunks (or
// elements) w * 32 + lane + j * 32 * RW of the free range; after one barrier
// the last warp, which keeps the forced ids, takes the top m of the warps'
// lists (the m largest keys of the row are the m largest of their union)
// and emits the row.  lb = the largest m-th entry of a full list bounds the
// row's m-th largest key from below, so only keys >= lb are ranked.
template <int RW, int MODE, bool VEC>
__global__ void __launch_bounds__(32 * RW, 32 / RW) select_row_kernel(const SelectArgs a) {
  // float4 rows have K % 4 == 0: at most kLongRowMaxK / 4 float4s
  static_assert(kLongRowChunks * 32 * RW >= kLongRowMaxK / 4, "chunk record too small");
  __shared__ unsigned long long s_cand[RW][kCandCap];
  __shared__ unsigned long long s_wsel[RW][kTopK];
  __shared__ unsigned long long s_surv[RW * kTopK];
  __shared__ unsigned long long s_mout[kTopK];
  __shared__ float s_cm[RW][kLongRowChunks * 32];
  __shared__ int s_nc[RW];
  __shared__ int s_wn[RW];
  // under programmatic dependent launch: wait for the preceding kernel
  // (the scorer) before reading its scores, then let dependents launch
  pdl_wait();
  pdl_launch_dependents();

  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int rows = a.T * 4;
  const int scale = a.index_scale, off = a.index_offset;
  const bool merger = warp == RW - 1;
  const int first = warp * 32 + lane, stride = 32 * RW;
  const WarpScratch ws{s_cand[warp], &s_nc[warp], &s_cm[warp][lane]};
  const int f_start = (free_lo(a) >> 2) + first;
  for (int row = blockIdx.x; row < rows; row += gridDim.x) {
    const int t = row >> 2, h = row & 3;
    const float *src = a.scores + (long long)row * a.K;
    float4 x0[kChunk];
    if constexpr (VEC)
      load_batch(reinterpret_cast<const float4 *>(src), f_start, stride, a.K >> 2, x0);
    const int nvp = __ldg(a.nvp + t);
    const int flag0 = merger ? early_flag<MODE>(a, lane, t, h) : -1;
    const Forced f = forced_ids(a, src, nvp, lane, merger);
    const int m = kTopK - f.nf;
    int c_lo, c_hi;
    free_range(a, nvp, c_lo, c_hi);
    int nw;
    if constexpr (VEC)
      nw = warp_top_m_vec(src, x0, c_lo, c_hi, first, stride, scale, off, m, lane, ws, s_wsel[warp]);
    else
      nw = warp_top_m_scalar(src, c_lo, c_hi, first, stride, scale, off, m, lane, ws, s_wsel[warp]);
    if (lane == 0) s_wn[warp] = nw;
    __syncthreads();

    if (merger) {
      int nch = 0;
      if (m > 0) {
        unsigned long long lb = 0;
        if (lane < RW && s_wn[lane] >= m) lb = s_wsel[lane][m - 1];
        lb = warp_max_key(lb);
        constexpr int PL = (RW * kTopK + 31) / 32;
        int ns = 0;
#pragma unroll
        for (int j = 0; j < PL; ++j) {
          const int q = lane + 32 * j;
          const int w = q / kTopK, i = q % kTopK;
          const unsigned long long k = (w < RW && i < s_wn[w]) ? s_wsel[w][i] : 0ull;
          const bool keep = k != 0ull && k >= lb;
          const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
          if (keep) s_surv[ns + __popc(bal & ((1u << lane) - 1u))] = k;
          ns += __popc(bal);
        }
        __syncwarp();
        for (int j = lane; j < ns; j += 32) {
          const unsigned long long my = s_surv[j];
          int rank = 0;
          for (int i = 0; i < ns; ++i) rank += (s_surv[i] > my) ? 1 : 0;
          if (rank < m) s_mout[rank] = my;
        }
        nch = min(m, ns);
        __syncwarp();
      }
      const int n = f.nf + nch;
      int my_id = f.fid;
      float my_sc = f.fsc;
      if (lane >= f.nf && lane < n) {
        const unsigned long long k = s_mout[lane - f.nf];
        my_id = key_id(k);
        my_sc = key_score(k, src, scale, off);
      }
      int out_id;
      float out_sc;
      sort_by_id_16(lane, n, my_id, my_sc, out_id, out_sc, reinterpret_cast<int *>(s_mout),
                    reinterpret_cast<float *>(s_mout) + kTopK);
      emit_row<MODE>(a, lane, row, t, h, out_id, out_sc, flag0);
    }
    __syncthreads();  // lists are reused by the next row
  }
}

// Second half of a merge of NS sources (the world size), once lane i < 16
// holds entry i of every source in ids[s] / scs[s] (id -1 = nothing): union
// with the maximum score per id, the Top16 rule with num_valid_pages, and
// the output ordered by id.
template <int NS>
__device__ __forceinline__ void merge_finish(const MergeArgs &a, int lane, int t, int hl, int nvp,
                                             const int (&ids)[NS], const float (&scs)[NS],
                                             int *s_idw, float *s_scw) {
  const int hpr = a.heads_per_rank;
  // keep an entry unless another source holds the same id with a higher
  // score (an exact tie goes to the lower source)
  bool keep[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) keep[s] = lane < kTopK && ids[s] >= 0 && ids[s] < nvp;
  if constexpr (NS > 1) {
#pragma unroll
    for (int s2 = 0; s2 < NS; ++s2) {
      for (int j = 0; j < kTopK; ++j) {
        const int id2 = __shfl_sync(0xFFFFFFFFu, ids[s2], j);
        const float sc2 = __shfl_sync(0xFFFFFFFFu, scs[s2], j);
#pragma unroll
        for (int s = 0; s < NS; ++s) {
          if (s == s2 || !keep[s] || ids[s] != id2) continue;
          if (sc2 > scs[s] || (sc2 == scs[s] && s2 < s)) keep[s] = false;
        }
      }
    }
  }
  int total = 0, nforced = 0;
  bool forced[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    forced[s] = keep[s] && forced_id(ids[s], nvp, a.init_blocks, a.local_blocks);
    total += __popc(__ballot_sync(0xFFFFFFFFu, keep[s]));
    nforced += __popc(__ballot_sync(0xFFFFFFFFu, forced[s]));
  }
  bool sel[NS];
  if (total <= kTopK) {
#pragma unroll
    for (int s = 0; s < NS; ++s) sel[s] = keep[s];
  } else {
    // m best free entries by (score desc, id asc)
    const int m = kTopK - min(nforced, kTopK);
    unsigned long long key[NS];
    int rank[NS];
#pragma unroll
    for (int s = 0; s < NS; ++s) {
      key[s] = (keep[s] && !forced[s]) ? make_key(scs[s], ids[s]) : 0ull;
      rank[s] = 0;
    }
#pragma unroll
    for (int s2 = 0; s2 < NS; ++s2) {
      for (int j = 0; j < kTopK; ++j) {
        const unsigned long long k2 = __shfl_sync(0xFFFFFFFFu, key[s2], j);
#pragma unroll
        for (int s = 0; s < NS; ++s) rank[s] += (k2 > key[s]) ? 1 : 0;
      }
    }
#pragma unroll
    for (int s = 0; s < NS; ++s) sel[s] = forced[s] || (key[s] != 0 && rank[s] < m);
  }
  // compact the selected entries (at most 16) and order them by id
  int n = 0;
#pragma unroll
  for (int s = 0; s < NS; ++s) {
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
  sort_by_id_16(lane, n, my_id, my_sc, out_id, out_sc, s_idw, s_scw);
  if (lane < kTopK) {
    const long long o = ((long long)t * hpr + hl) * kTopK + lane;
    a.out_scores[o] = out_sc;
    a.out_ids[o] = out_id;
  }
}

// One warp per (token, owned head).  Lane i < 16 holds entry i of every
// source row (NS = world size sources), so the union, the per-id maximum
// and the ranking are done with shuffles; the result is compacted through
// shared memory and ordered by id.
template <int NS>
__global__ void __launch_bounds__(128) merge_kernel(const MergeArgs a) {
  __shared__ int s_id[4][kTopK];
  __shared__ float s_sc[4][kTopK];
  // under programmatic dependent launch: wait for the preceding kernel (the
  // publish) before reading anything; then a scorer launched next with early
  // start may begin its set-up (it reads nothing this kernel writes before
  // waiting for it)
  if (a.pdl) pdl_wait();
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + warp;
  const int hpr = a.heads_per_rank;
  if (item >= a.T * hpr) return;
  const int t = item >> hpr_shift(hpr), hl = item & (hpr - 1);
  const int nvp = a.nvp[t];
  constexpr int ws = NS;

  // lane s < ws polls source s's flag (acquire); the warp barrier then
  // orders every lane's reads of the rows after those acquires, so all the
  // rows are read at once (gpu-scope loads: the rows are reused every step)
  int *row_of_lane = nullptr;
  int ok = 1;
  if (lane < ws) {
    const long long r = (((long long)a.slot * ws + lane) * hpr + hl) * a.capacity + t;
    row_of_lane = a.recv + r * kRowWords;
    ok = poll_flag(row_of_lane + 32, 1, a.spin_limit) ? 1 : 0;
  }
  const unsigned read_mask = __ballot_sync(0xFFFFFFFFu, ok) & ((1u << ws) - 1u);
  __syncwarp();
  if (lane == 0 && read_mask != (1u << ws) - 1u)
    atomicAdd(a.errors, ws - __popc(read_mask));
  int ids[NS];
  float scs[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    ids[s] = -1;
    scs[s] = -INFINITY;
    if (((read_mask >> s) & 1u) && lane < kTopK) {
      const long long r = (((long long)a.slot * ws + s) * hpr + hl) * a.capacity + t;
      const int *row = a.recv + r * kRowWords;
      scs[s] = __int_as_float(ld_relaxed_gpu(row + lane));
      ids[s] = ld_relaxed_gpu(row + kTopK + lane);
    }
  }
  // free the rows that were read, after every lane's reads
  __syncwarp();
  if (lane < ws && ok) st_release_gpu(row_of_lane + 32, 0);

  merge_finish<NS>(a, lane, t, hl, nvp, ids, scs, s_id[warp], s_sc[warp]);
}

// Owner merge of tagged rows: a source row has arrived when all 32 words
// carry the owner's expected generation + 1 (the counter advances on every
// merge).  Polls are bounded by spin_limit and the wait timeout.
template <int NS>
__global__ void __launch_bounds__(128) merge_tagged_kernel(const MergeArgs a) {
  __shared__ int s_id[4][kTopK];
  __shared__ float s_sc[4][kTopK];
  // as merge_kernel
  if (a.pdl) pdl_wait();
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + warp;
  const int hpr = a.heads_per_rank;
  if (item >= a.T * hpr) return;
  const int t = item >> hpr_shift(hpr), hl = item & (hpr - 1);
  const int nvp = a.nvp[t];
  constexpr int ws = NS;

  int ids[NS];
  float scs[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    ids[s] = -1;
    scs[s] = -INFINITY;
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
  merge_finish<NS>(a, lane, t, hl, nvp, ids, scs, s_id[warp], s_sc[warp]);
}

// Owner merge of received prefill carrier rows [ws][T][hpr][32]: every
// source row is there already (the caller's exchange has completed), so
// there is nothing to wait for.
template <int NS>
__global__ void __launch_bounds__(128) merge_carrier_kernel(const MergeArgs a) {
  __shared__ int s_id[4][kTopK];
  __shared__ float s_sc[4][kTopK];

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int item = blockIdx.x * 4 + warp;
  const int hpr = a.heads_per_rank;
  if (item >= a.T * hpr) return;
  const int t = item >> hpr_shift(hpr), hl = item & (hpr - 1);
  const int nvp = a.nvp[t];
  int ids[NS];
  float scs[NS];
#pragma unroll
  for (int s = 0; s < NS; ++s) {
    ids[s] = -1;
    scs[s] = -INFINITY;
    if (lane < kTopK) {
      const int *row = a.received + (((long long)s * a.T + t) * hpr + hl) * 32;
      scs[s] = __int_as_float(row[lane]);
      ids[s] = row[kTopK + lane];
    }
  }
  merge_finish<NS>(a, lane, t, hl, nvp, ids, scs, s_id[warp], s_sc[warp]);
}

}  // namespace

cudaError_t select_prepare() { return cudaSuccess; }

// One select kernel launch, with the programmatic-serialization attribute
// when a.pdl is set.
template <typename Kernel>
cudaError_t launch_one(Kernel kernel, int grid, int threads, const SelectArgs &a,
                       cudaStream_t stream) {
  if (!a.pdl) {
    kernel<<<grid, threads, 0, stream>>>(a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3((unsigned)threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int MODE>
cudaError_t launch_select_mode(const SelectArgs &a, bool vec, int rows, int sm_count,
                               cudaStream_t stream) {
  if (a.K > kWarpRowMaxK) {
    const int threads = 32 * kRowWarps;
    return vec ? launch_one(select_row_kernel<kRowWarps, MODE, true>, rows, threads, a, stream)
               : launch_one(select_row_kernel<kRowWarps, MODE, false>, rows, threads, a, stream);
  }
  const int threads = 32 * kSelWarps;
  const int need = (rows + kSelWarps - 1) / kSelWarps;
  if (vec && a.K <= kShortMaxK) {
    // persistent: eight CTAs per SM, each warp a row at a time with the next
    // row's loads in flight
    const int g2 = need < 8 * sm_count ? need : 8 * sm_count;
    return launch_one(select_short_kernel<MODE>, g2, threads, a, stream);
  }
  return vec ? launch_one(select_warp_kernel<MODE, true>, need, threads, a, stream)
             : launch_one(select_warp_kernel<MODE, false>, need, threads, a, stream);
}

cudaError_t launch_select(const SelectArgs &a, int mode, int sm_count, cudaStream_t stream) {
  const int rows = a.T * 4;
  if (rows == 0) return cudaSuccess;
  // float4 rows when every row starts on a 16-byte boundary
  const bool vec = (a.K % 4 == 0) && ((reinterpret_cast<uintptr_t>(a.scores) & 15u) == 0);
  switch (mode) {
    case kEmitLegacy: return launch_select_mode<kEmitLegacy>(a, vec, rows, sm_count, stream);
    case kEmitTagged: return launch_select_mode<kEmitTagged>(a, vec, rows, sm_count, stream);
    case kEmitCarrier: return launch_select_mode<kEmitCarrier>(a, vec, rows, sm_count, stream);
    default: return launch_select_mode<kEmitPlain>(a, vec, rows, sm_count, stream);
  }
}

// Merge kernels are compiled per world size (1, 2 or 4 sources).
template <typename Kernel>
void launch_merge_one(Kernel kernel, const MergeArgs &a, int grid, cudaStream_t stream) {
  if (!a.pdl) {
    kernel<<<grid, 128, 0, stream>>>(a);
    return;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaLaunchKernelEx(&cfg, kernel, a);
}

template <int NS>
void launch_merge_ns(const MergeArgs &a, int kind, int grid, cudaStream_t stream) {
  if (kind == 2) launch_merge_one(merge_carrier_kernel<NS>, a, grid, stream);
  else if (kind == 1) launch_merge_one(merge_tagged_kernel<NS>, a, grid, stream);
  else launch_merge_one(merge_kernel<NS>, a, grid, stream);
}

cudaError_t launch_merge_kind(const MergeArgs &a, int kind, cudaStream_t stream) {
  const int items = a.T * a.heads_per_rank;
  if (items == 0) return cudaSuccess;
  const int grid = (items + 3) / 4;
  switch (a.world_size) {
    case 1: launch_merge_ns<1>(a, kind, grid, stream); break;
    case 2: launch_merge_ns<2>(a, kind, grid, stream); break;
    case 4: launch_merge_ns<4>(a, kind, grid, stream); break;
    default: return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t launch_merge_carrier(const MergeArgs &a, cudaStream_t stream) {
  return launch_merge_kind(a, 2, stream);
}

cudaError_t launch_merge(const MergeArgs &a, bool tagged, cudaStream_t stream) {
  return launch_merge_kind(a, tagged ? 1 : 0, stream);
}

}  // namespace icp
