// icp_score.cu - decode index scorer (msa_icp_decode_index_score_sharded) and
// the fused scorer + Top16 select (prepare_msa_icp_indexer, decode(pool=...),
// whose fused scorer leaves no score plane).
//
// What the scorer computes: for every request b, token j (position
// seq_len_b - dql + j), head h and plane column c of the request,
//   score_out[t][h][c] = max over the column's keys at positions <= the
//                        token's position of dot(deq(q[t,h,:]), deq(k[key,:]))
// (-inf when no key is visible), for c < round_up(columns, 4); the other
// columns are not written.  The fused variant computes the same column
// values and applies the Top16 rule of msa_icp_topk_select_publish to them
// directly.
//
// How (one persistent CTA per SM, 192 threads, warp-specialised):
//   warp 0     TMA producer: streams the 128-row K tiles of the CTA's share of
//              all requests' pages (each page read once per call) into a
//              ring of 16 KB shared-memory stages (10 for this scorer, 8 for
//              the fused one), and each request's 32 query rows
//              (4 * dql used) once, stored four times so that every TMEM lane
//              quarter receives all of them.  When a tile is two or four page
//              slices (world size 2 or 4), warp 6, a second producer, issues
//              every other tile: one warp alone cannot issue that many boxes
//              fast enough.
//   warp 1     MMA issuer (the whole warp waits; an elected lane issues):
//              per tile, 4 x tcgen05.mma kind::f8f6f4 with A = the
//              replicated queries (M = 128), B = the 128 keys of the tile
//              (N = 128), K = 32, into one of 4 fp32 TMEM accumulators.
//              All 4 heads and all dql tokens share one K tile.
//   warps 2-5  epilogue: tile i belongs to epilogue warp i % 4, which reads
//              its lane quarter of the accumulator (thread = query row,
//              registers = the tile's 128 key scores) with the reducing TMEM
//              load: it also returns each column's maximum over its keys,
//              the column value unless the causal limit cuts the column,
//              whose keys are then masked and folded by a register max tree.
//              Scorer: one plane store per (query row, column).
//              Fused: the column value goes into the row's running Top16
//              (forced ids kept aside); at the end of each request segment
//              every epilogue warp writes its lists to the workspace, and the
//              last CTA to finish a request merges all lists of that request.
// The tiles of all requests form one list that is cut into gridDim.x equal
// contiguous ranges, so every CTA streams the same number of K bytes.
// Products of two e4m3 values are exact in fp32; the MMA sums 128 of them in
// fp32.  The per-key arithmetic does not depend on where the key sits in the
// tile, so sharded and unsharded layouts give identical key scores.
#include <climits>

#include "icp_device.cuh"
#include "icp_fused.cuh"
#include "icp_internal.h"

namespace icp {

#ifdef ICP_TIMELINE
// Timeline build only: globaltimer stamps of each CTA's phases (slot
// meanings in include/icp_timeline.h), read back by icp_timeline_read.
constexpr int kTimelineCtas = 1024;
constexpr int kTimelineSlots = 24;
__device__ unsigned long long g_timeline[kTimelineCtas * kTimelineSlots];
#define ICP_STAMP(slot) (g_timeline[blockIdx.x * kTimelineSlots + (slot)] = globaltimer_ns())
// adds the ns spent in `wait` to a per-CTA sum (a slot that holds a total)
#define ICP_TIMED(slot, wait)                                              \
  do {                                                                     \
    const unsigned long long icp_t0_ = globaltimer_ns();                   \
    wait;                                                                  \
    g_timeline[blockIdx.x * kTimelineSlots + (slot)] += globaltimer_ns() - icp_t0_; \
  } while (0)
// the same inside a loop that the whole warp runs: lane 0 keeps the sum
#define ICP_TIMED_WARP(slot, wait)                                         \
  do {                                                                     \
    const unsigned long long icp_t0_ = globaltimer_ns();                   \
    wait;                                                                  \
    if ((threadIdx.x & 31) == 0)                                           \
      g_timeline[blockIdx.x * kTimelineSlots + (slot)] += globaltimer_ns() - icp_t0_; \
  } while (0)
#else
#define ICP_STAMP(slot) ((void)0)
#define ICP_TIMED(slot, wait) wait
#define ICP_TIMED_WARP(slot, wait) wait
#endif

namespace {

// Ring stages: 8 of 16 KB, or 10 for the plane scorer with one producer
// (more bytes in flight: 0.4 % faster on the large decode workloads, while
// the two-producer variant measured slower with 10)
constexpr int kStages = 8;
constexpr int kStagesPlane = 10;
constexpr int kStagesMax = 10;    // barriers are laid out for the deepest ring
template <bool FUSED, bool WIDE, int NPROD = 1>
struct RingStages {
  static constexpr int value = (FUSED || WIDE || NPROD > 1) ? kStages : kStagesPlane;
};
constexpr int kAcc = 4;                // one accumulator per epilogue warp
constexpr int kTileBytes = 128 * 128;  // 128 K rows x 128 fp8
constexpr int kQRows = 32;             // query rows staged per request (4 * dql <= 32)
constexpr int kQBytes = 4 * kQRows * 128;  // four copies -> the 128-row A operand
// prefill: a plan record's 4 * kPlanTokens distinct query rows, one TMA box
// that holds two 128-row A operands
constexpr int kQBytesWide = 4 * kPlanTokens * 128;
static_assert(4 * kPlanTokens == 256, "a record's query rows are two 128-row operands");
constexpr int kThreads = 192;
// prefill scorer: two sets of four epilogue warps, one per accumulator
constexpr int kEpiSetsWide = 2;
constexpr int kThreadsWide = 64 + 128 * kEpiSetsWide;
// NPROD 2: a second producer warp (warp 6) takes every other tile; used when
// a tile is two or four page slices (one TMA box each)
template <bool WIDE, int NPROD = 1>
struct BlockThreads {
  static constexpr int value = WIDE ? kThreadsWide : kThreads + 32 * (NPROD - 1);
};
constexpr uint32_t kAccCols = 128;     // N = 128 keys per accumulator
constexpr uint32_t kTmemCols = kAcc * kAccCols;
constexpr int kNumBars = 2 * kStagesMax + 2 * kAcc + 4 + 1;

// Shared-memory carve-up (offsets from a 1024-byte aligned base).
// The prefill scorer's two query slots are twice as large.
constexpr uint32_t kOffStages = 0;
template <bool FUSED, bool WIDE, int NPROD = 1>
struct Layout {
  static constexpr uint32_t q_bytes = WIDE ? kQBytesWide : kQBytes;
  static constexpr uint32_t off_q =
      kOffStages + RingStages<FUSED, WIDE, NPROD>::value * kTileBytes;
  static constexpr uint32_t off_bars = off_q + 2 * q_bytes;
  static constexpr uint32_t off_misc = off_bars + ((kNumBars * 8 + 127) / 128) * 128;
  static constexpr uint32_t off_lists = off_misc + 128;  // fused only
};
// fused epilogue: per warp 16 list keys x 32 lanes (u64) + 16 forced (id, score) x 32 lanes
constexpr uint32_t kWarpListBytes = 16 * 32 * 8 + 16 * 32 * 8;
constexpr uint32_t kListBytes = 4 * kWarpListBytes;   // 32 KB
constexpr uint32_t kFusedExtra = kListBytes;

template <bool FUSED, bool WIDE, int NPROD = 1>
struct PrefixOffset {
  static constexpr uint32_t value =
      FUSED ? Layout<FUSED, WIDE, NPROD>::off_lists + kFusedExtra
            : Layout<FUSED, WIDE, NPROD>::off_lists;
};

// Walks the CTA's tile range [g0, g1) request by request.
// The list is in units of work: a request with tiles weighs its tiles plus
// k leading units that hold no tile (the cost of starting a request), so a
// CTA whose range covers many short requests gets fewer tiles.
struct SegmentWalker {
  const int *prefix;  // prefix[b] = units of requests < b, prefix[batch] = total
  int batch;
  int g, g1, b, k;
  __device__ SegmentWalker(const int *p, int nb, int g0_, int g1_, int k_)
      : prefix(p), batch(nb), g(g0_), g1(g1_), b(0), k(k_) {
    int lo = 0, hi = nb;  // largest lo with prefix[lo] <= g0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= g) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  // Next segment: request rb, local tiles [t0, t1).  False when done.
  // Requests of which the range holds only leading units are skipped.
  __device__ bool next(int &rb, int &t0, int &t1) {
    for (;;) {
      if (g >= g1) return false;
      while (b < batch && prefix[b + 1] <= g) ++b;
      if (b >= batch) return false;
      const int end = min(g1, prefix[b + 1]);
      const int s0 = max(g, prefix[b] + k);  // first tile position in range
      g = end;
      ++b;
      if (s0 < end) {
        rb = b - 1;
        t0 = s0 - prefix[b - 1] - k;
        t1 = end - prefix[b - 1] - k;
        return true;
      }
    }
  }
};

// Leading units per request in the prefill scorer's work list (about the
// time a request's start costs a CTA there, in tiles); none for decode.
constexpr int kWideRequestUnits = 4;

__device__ __forceinline__ int page_slot_of(int c, int split) { return split ? (c >> 1) : c; }

// What the kernel needs of request b: a decode request (token rows
// b * dql .. + dql, its own block-table row and seq_len), or a record of a
// prefill plan (up to kPlanTokens = 64 consecutive tokens of a request's chunk).
struct ReqView {
  int seq_len;   // positions seen by the tokens: the last one is seq_len - 1
  int tok0;      // first token (index_q / plane rows tok0 * 4 ...)
  int bt_row;    // block-table row
  int ntok;      // tokens (queries of positions seq_len - ntok .. seq_len - 1)
  int full_len;  // the request's seq_len: sets the columns written
};

// Requests of this call; a plan's count is clamped to the capacity that the
// shared-memory prefix sums were sized for.
__device__ __forceinline__ int req_count(const ScoreArgs &a) {
  return a.vreq ? min(max(*a.vcount, 0), a.batch) : a.batch;
}

__device__ __forceinline__ int req_seq_len(const ScoreArgs &a, int b) {
  return a.vreq ? a.vreq[kPlanHeaderInts + kPlanRecordInts * b + 2] : a.seq_lens[b];
}

__device__ __forceinline__ ReqView req_view(const ScoreArgs &a, int b) {
  if (a.vreq) {
    const int *r = a.vreq + kPlanHeaderInts + kPlanRecordInts * b;
    return ReqView{r[2], r[0], r[1], r[3], r[4]};
  }
  const int sl = a.seq_lens[b];
  return ReqView{sl, b * a.dql, b, a.dql, sl};
}
__device__ __forceinline__ int row_off_of(int c, int split) { return split ? (c & 1) * 128 : 0; }

// Counts a request whose block table holds an entry outside [0, num_pages)
// once per call: fb is the first such column a producer warp met in its
// segment of request (or plan record) b.  The warp that met the request's
// first bad page counts it: no earlier page of the row may be bad, and for a
// plan record the preceding record of the same request (which covers a
// prefix of the same columns) must not reach that column.
__device__ __noinline__ void count_bad_entry(const ScoreArgs &a, int b, const ReqView &rv,
                                             const int32_t *btrow, int fb, int lane) {
  if (fb == INT_MAX || !a.errors) return;
  const ScoreGeom &g = a.g;
  const int slot = page_slot_of(fb, g.split);
  bool earlier = false;
  for (int i = lane; i < slot && !earlier; i += 32)
    earlier = (unsigned)btrow[i] >= (unsigned)a.num_pages;
  earlier = __any_sync(0xFFFFFFFFu, earlier);
  if (!earlier && a.vreq && b > 0) {
    const ReqView pv = req_view(a, b - 1);
    earlier = pv.bt_row == rv.bt_row && fb < units_of(pv.seq_len, a.page_size, g.split);
  }
  if (!earlier && lane == 0) atomicAdd(a.errors, 1);
}

// Per-lane running Top16 of one query row over the columns a warp has seen.
struct LaneTop {
  int cnt;                 // list entries used (<= 16)
  unsigned long long kmin; // smallest listed key once the list is full
  int fcnt;                // forced entries kept
  int nvp;                 // the row's num_valid_pages
};

__device__ __forceinline__ void lane_insert(LaneTop &s, unsigned long long *lk, int lane,
                                            unsigned long long key) {
  if (s.cnt < kTopK) {
    lk[s.cnt * 32 + lane] = key;
    if (++s.cnt == kTopK) {
      unsigned long long mn = lk[lane];
      for (int j = 1; j < kTopK; ++j) mn = min(mn, lk[j * 32 + lane]);
      s.kmin = mn;
    }
  } else if (key > s.kmin) {
    unsigned long long mn = ~0ull;
    bool replaced = false;
    for (int j = 0; j < kTopK; ++j) {
      unsigned long long x = lk[j * 32 + lane];
      if (!replaced && x == s.kmin) {
        lk[j * 32 + lane] = key;
        x = key;
        replaced = true;
      }
      mn = min(mn, x);
    }
    s.kmin = mn;
  }
}

// Epilogue of one tile for a warp.  taddr addresses the warp's lane quarter
// of the tile's accumulator: lane l holds query row rowq + l of the request
// (row = token j * 4 + head; rowq = 0, the queries being replicated in every
// quarter), columns 0..127 hold the tile's keys in order.  R keys feed one
// plane column, so the tile covers 128 / R columns.
template <int R, bool FUSED>
__device__ __forceinline__ void epilogue_tile(const ScoreArgs &a, uint32_t taddr, int lane,
                                              int rowq, int tok0, int ntok, int tl, int nunits,
                                              int seq_len, uint32_t tempty,
                                              LaneTop &lt, unsigned long long *lk, int *lfid,
                                              float *lfsc) {
  constexpr int CPT = 128 / R;
  // the tile in registers, and each column's maximum over its R keys from
  // the reducing load
  float v[128];
  float mx[CPT];
#pragma unroll
  for (int cc = 0; cc < CPT; ++cc) {
    if constexpr (R == 128) tmem_ld_max128(taddr, v, mx[0]);
    else if constexpr (R == 64) tmem_ld_max64(taddr + cc * R, v + cc * R, mx[cc]);
    else tmem_ld_max32(taddr + cc * R, v + cc * R, mx[cc]);
  }
  tmem_wait_ld();
  // the accumulator is in registers: hand it back to the MMA warp
  tc_fence_before();
  __syncwarp();
  if (lane == 0) mbar_arrive(tempty);

  const ScoreGeom &g = a.g;
  const int row = rowq + lane;                         // the lane's query row
  const long long pfirst = (long long)seq_len - ntok;  // position of token 0
  const long long p_lane = pfirst + (row >> 2);        // position of this row's token
  const bool row_ok = row < 4 * ntok;
#pragma unroll
  for (int cc = 0; cc < CPT; ++cc) {
    const int c = tl * CPT + cc;
    if (c >= nunits) break;
    float *vc = v + cc * R;
    const long long pos0 = g.split ? (long long)c * 128
                                   : (long long)c * a.page_size +
                                         (long long)a.rank * g.rows_per_page;
    float val = mx[cc];
    if (pos0 + R - 1 > pfirst) {
      // the column reaches past the first token: mask, then fold
#pragma unroll
      for (int i = 0; i < R; ++i)
        if (pos0 + i > p_lane) vc[i] = -INFINITY;
      max_tree3<R>(vc);
      val = vc[0];
    }
    val += 0.0f;  // + 0 folds -0 onto +0
    if (row_ok && c < a.cols) {
      if constexpr (!FUSED) {
        const long long prow = (long long)tok0 * 4 + row;
        a.score_out[prow * a.cols + c] = val;
      } else {
        const int id = c * a.index_scale + a.index_offset;
        if (id < lt.nvp) {
          if (forced_id(id, lt.nvp, a.init_blocks, a.local_blocks)) {
            if (lt.fcnt < kTopK) {
              lfid[lt.fcnt * 32 + lane] = id;
              lfsc[lt.fcnt * 32 + lane] = val;
              ++lt.fcnt;
            }
          } else {
            lane_insert(lt, lk, lane, make_key(val, id));
          }
        }
      }
    }
  }
}

// Epilogue of one tile of the prefill scorer for one warp: lane l holds
// query row rowq + l of the record (up to 256 distinct rows).  A column that
// reaches past the record's first token is masked with 32-bit compares.
// With release, the warp hands the accumulator back once its tile is in
// registers.
template <int R>
__device__ __forceinline__ void epilogue_tile_wide(const ScoreArgs &a, uint32_t ta, int lane,
                                                   int rowq, int tok0, int ntok, int tl,
                                                   int nunits, int seq_len, uint32_t tempty,
                                                   bool release) {
  constexpr int CPT = 128 / R;  // plane columns in the tile
  const ScoreGeom &g = a.g;
  const int row = rowq + lane;
  const long long pfirst = (long long)seq_len - ntok;  // position of token 0
  const long long p_lane = pfirst + (row >> 2);        // position of this row's token
  const bool row_ok = row < 4 * ntok;
  // The load also returns each column's maximum over its R keys: the plane
  // value of every column that no row's causal limit cuts.  A cut column
  // masks its keys in registers and folds them with a max tree.
  auto column = [&](int cc, float *vc, float mx) {
    const int c = tl * CPT + cc;
    const long long pos0 = g.split ? (long long)c * 128
                                   : (long long)c * a.page_size +
                                         (long long)a.rank * g.rows_per_page;
    if (pos0 + R - 1 > pfirst) {
      // keys i <= lim of the column are at or before the row's token
      const long long d = p_lane - pos0;
      const int lim = (int)(d < -1 ? -1 : (d > R - 1 ? R - 1 : d));
#pragma unroll
      for (int i = 0; i < R; ++i)
        if (i > lim) vc[i] = -INFINITY;
      max_tree3<R>(vc);
      mx = vc[0];
    }
    return mx;
  };
  auto store = [&](int cc, float val) {
    const int c = tl * CPT + cc;
    if (c < nunits && c < a.cols && row_ok)
      a.score_out[((long long)tok0 * 4 + row) * a.cols + c] = val + 0.0f;  // + 0 folds -0
  };
  auto hand_back = [&]() {
    if (release) {
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
    }
  };
  if constexpr (R == 128) {
    // the whole tile in registers with one wait
    float v[128];
    float mx;
    tmem_ld_max128(ta, v, mx);
    tmem_wait_ld();
    hand_back();
    store(0, column(0, v, mx));
  } else {
    // one column at a time (a wait each): the kernel's registers then stay
    // below the ten-warp limit without spills
    float val[CPT];
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) {
      float v[R];
      float mx;
      if constexpr (R == 64) tmem_ld_max64(ta + cc * R, v, mx);
      else tmem_ld_max32(ta + cc * R, v, mx);
      tmem_wait_ld();
      val[cc] = column(cc, v, mx);
    }
    hand_back();
#pragma unroll
    for (int cc = 0; cc < CPT; ++cc) store(cc, val[cc]);
  }
}

// WIDE: the prefill scorer.  A request (a plan record of up to 64 tokens)
// stages its 256 distinct query rows in one box: two 128-row A operands
// (row halves).  Its tiles go in pairs: two adjacent ring stages form one
// 256-row B operand.  Each row half of a pair is one item: an N = 256 MMA
// group (N = 128 for a segment's odd last tile; the second half only when
// the record has more than 32 tokens) into one of two 256-column
// accumulators, items alternating, so each key byte read serves 256 query
// rows at the N = 256 MMA rate.  The epilogue warps form two sets of four,
// set s owning accumulator s: it finishes every item of parity s, one tile
// after the other, each warp its lane quarter (8 of the half's 32 tokens),
// and the accumulator is free again after the set's four warps have read
// both tiles.  The two warps that share a scheduler thus work on different
// items.
template <bool FUSED, bool WIDE, int NPROD = 1, int RW = 0>
__global__ void __launch_bounds__(BlockThreads<WIDE, NPROD>::value, 1)
score_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq,
             const ScoreArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t *gb = smem_raw + (sb - raw);

  constexpr int NT = BlockThreads<WIDE, NPROD>::value;
  constexpr int kEpiThreads = WIDE ? 128 * kEpiSetsWide : 128;
  static_assert(NPROD == 1 || (!WIDE && !FUSED), "a second producer only for the plane scorer");
  static_assert(!WIDE || RW == 128 || RW == 64 || RW == 32, "prefill: RW = g.R, one kernel each");
  using L = Layout<FUSED, WIDE, NPROD>;
  constexpr int NS = RingStages<FUSED, WIDE, NPROD>::value;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const ScoreGeom g = a.g;

  auto bar_full = [&](int s) { return sb + L::off_bars + 8u * s; };
  auto bar_empty = [&](int s) { return sb + L::off_bars + 8u * (kStagesMax + s); };
  auto bar_tfull = [&](int i) { return sb + L::off_bars + 8u * (2 * kStagesMax + i); };
  auto bar_tempty = [&](int i) { return sb + L::off_bars + 8u * (2 * kStagesMax + kAcc + i); };
  auto bar_qfull = [&](int i) { return sb + L::off_bars + 8u * (2 * kStagesMax + 2 * kAcc + i); };
  auto bar_qempty = [&](int i) {
    return sb + L::off_bars + 8u * (2 * kStagesMax + 2 * kAcc + 2 + i);
  };
  const uint32_t bar_done = sb + L::off_bars + 8u * (2 * kStagesMax + 2 * kAcc + 4);

  // [0] TMEM base, [1] abort flag
  volatile int *misc = reinterpret_cast<volatile int *>(gb + L::off_misc);
  int *prefix = reinterpret_cast<int *>(gb + PrefixOffset<FUSED, WIDE, NPROD>::value);
  int *partial = prefix + a.batch + 1;  // NT / 32 scratch ints
  const int nbatch = req_count(a);      // <= a.batch

  if (threadIdx.x == 0) {
    ICP_STAMP(0);
    for (int s = 0; s < NS; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(bar_tfull(i), 1);
      mbar_init(bar_tempty(i), WIDE ? 4 : 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar_qfull(i), 1);
      mbar_init(bar_qempty(i), 1);
    }
    mbar_init(bar_done, 1);
    misc[1] = 0;
    fence_mbarrier_init();
  }
  if (warp == 0 && lane == 0) {
    prefetch_tensormap(&tmk);
    prefetch_tensormap(&tmq);
  }
  if (warp == 1) tmem_alloc(sb + L::off_misc, kTmemCols);

  // Tiles per request and their prefix sums (chunked block scan).
  {
    const int nb = nbatch;
    const int chunk = (nb + NT - 1) / NT;
    const int lo = threadIdx.x * chunk, hi = min(nb, lo + chunk);
    int sum = 0;
    for (int b = lo; b < hi; ++b) {
      const int u = units_of(req_seq_len(a, b), a.page_size, g.split);
      const int tiles = (u + g.cpt - 1) / g.cpt;
      sum += tiles + (WIDE && tiles > 0 ? kWideRequestUnits : 0);
    }
#ifdef ICP_TIMELINE
    if (threadIdx.x == 0 && sum >= 0) ICP_STAMP(15);
#endif
    // exclusive scan of the per-thread sums: shuffles inside each warp, then
    // the warp totals (NT / 32 of them) in shared memory
    int incl = sum;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) partial[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int w = 0; w < warp; ++w) base += partial[w];
    if (threadIdx.x == NT - 1) prefix[nb] = base + incl;
    int run = base + incl - sum;
    for (int b = lo; b < hi; ++b) {
      prefix[b] = run;
      const int u = units_of(req_seq_len(a, b), a.page_size, g.split);
      const int tiles = (u + g.cpt - 1) / g.cpt;
      run += tiles + (WIDE && tiles > 0 ? kWideRequestUnits : 0);
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = (uint32_t)misc[0];
  if (threadIdx.x == 0) ICP_STAMP(1);

  const long long total = prefix[nbatch];
  const int g0 = (int)(total * blockIdx.x / gridDim.x);
  const int g1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
  volatile int *abort_flag = misc + 1;

  if (warp == 0 || (NPROD == 2 && warp == 6)) {
    // ------------------------------------------------------------ producer
    // With two producers, producer pp issues the tiles whose place in the
    // CTA's tile sequence has parity pp; both walk every tile to keep the
    // ring's stage and phase, and producer 0 alone loads the queries.
    const int pp = NPROD == 2 && warp == 6 ? 1 : 0;
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t sphase = 0;
    uint32_t qph0 = 0, qph1 = 0;
    int qslot = 0;
    long long issued = 0;
    int last_qslot = -1;
    SegmentWalker walk(prefix, nbatch, g0, g1, WIDE ? kWideRequestUnits : 0);
    int b, t0, t1;
    bool ok = true;
#ifdef ICP_TIMELINE
    if (lane == 0 && walk.b >= 0) ICP_STAMP(18);
#endif
    if (a.pdl) {
      // Early start: the set-up above (barriers, TMEM, the tile prefix sums
      // from seq_lens) ran while the preceding kernel finished; every load
      // of the step's data comes after the wait.
      pdl_wait();
      if (lane == 0) ICP_STAMP(12);
    }
    while (ok && walk.next(b, t0, t1)) {
#ifdef ICP_TIMELINE
      if (lane == 0) g_timeline[blockIdx.x * kTimelineSlots + 23] += 1;  // segments
#endif
      const ReqView rv = req_view(a, b);
      const int nunits = units_of(rv.seq_len, a.page_size, g.split);
      const uint32_t qph = qslot ? qph1 : qph0;
#ifdef ICP_TIMELINE
      if (lane == 0 && issued == 0 && nunits >= 0) ICP_STAMP(16);
#endif
      if (pp == 0 && lane == 0) ok = mbar_wait(bar_qempty(qslot), qph ^ 1u, abort_flag);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
      if (!ok) break;
#ifdef ICP_TIMELINE
      if (lane == 0 && issued == 0) ICP_STAMP(17);
#endif
      if (pp == 0 && lane == 0) {
        mbar_arrive_expect_tx(bar_qfull(qslot), L::q_bytes);
        if constexpr (WIDE) {
          tma_load_2d(sb + L::off_q + qslot * L::q_bytes, &tmq, 0, rv.tok0 * 4, bar_qfull(qslot));
        } else {
          for (int r = 0; r < 4; ++r)
            tma_load_2d(sb + L::off_q + qslot * L::q_bytes + r * kQRows * 128, &tmq, 0, rv.tok0 * 4,
                        bar_qfull(qslot));
        }
      }
      last_qslot = qslot;
      if (qslot) qph1 ^= 1u; else qph0 ^= 1u;
      qslot ^= 1;
#ifdef ICP_TIMELINE
      if (lane == 0 && issued == 0) ICP_STAMP(13);
#endif
      const int cbeg = t0 * g.cpt;
      const int cend = min(t1 * g.cpt, nunits);
      const int32_t *btrow = a.block_table + (long long)rv.bt_row * a.bt_stride;
      // A table entry outside [0, num_pages) is replaced by num_pages, whose
      // rows lie past the end of the tensor map: the box reads as zeros.  The
      // lane notes the first such column it met (an entry is vetted when it
      // is first used, so the load stays in flight until then; at P256 with
      // world_size 1 a page feeds two columns and only the even one counts).
      int first_bad = INT_MAX;
      auto vet = [&](int pg, int c) {
        if ((unsigned)pg >= (unsigned)a.num_pages) {
          if (c < cend && !(g.split && (c & 1))) first_bad = min(first_bad, c);
          return a.num_pages;
        }
        return pg;
      };
      int grp = cbeg;
      int pg_cur = (cbeg + lane < cend) ? btrow[page_slot_of(cbeg + lane, g.split)] : 0;
      int pg_nxt = (cbeg + 32 + lane < cend) ? btrow[page_slot_of(cbeg + 32 + lane, g.split)] : 0;
      pg_cur = vet(pg_cur, cbeg + lane);
#ifdef ICP_TIMELINE
      if (lane == 0 && issued == 0 && pg_cur >= 0) ICP_STAMP(14);
#endif
      for (int tl = t0; tl < t1; ++tl) {
        const int c0 = tl * g.cpt;
        if (c0 >= grp + 32) {
          grp += 32;
          pg_cur = vet(pg_nxt, grp + lane);
          pg_nxt = (grp + 32 + lane < cend) ? btrow[page_slot_of(grp + 32 + lane, g.split)] : 0;
        }
        const int ncol = min(g.cpt, cend - c0);
        if (NPROD == 2 && (int)(issued & 1) != pp) {
          // the other producer's tile: only the ring position advances
          ++issued;
          if (++stage == NS) {
            stage = 0;
            sphase ^= 1u;
          }
          continue;
        }
        // WIDE: tiles go in pairs (t0, t0 + 1), ... into slots of two
        // adjacent stages, one barrier per slot; j is the tile in its pair
        const int j = WIDE ? ((tl - t0) & 1) : 0;
        if (j == 0) {
          if constexpr (NPROD == 2 || WIDE) {
            // the two-producer kernel (launches of 4 KB page slices) and the
            // prefill scorer: every lane waits, 0.823 against 0.798 of the
            // copy peak on the sharded workload, 0.744 against 0.738 of the
            // fp8 peak on the prefill window; the long single-producer
            // decode streams were slower so (multitoken 0.968 against 0.999)
            ICP_TIMED_WARP(19, ok = mbar_wait(bar_empty(stage), sphase ^ 1u, abort_flag));
            ok = __all_sync(0xFFFFFFFFu, ok);
          } else {
            if (lane == 0) ICP_TIMED(19, ok = mbar_wait(bar_empty(stage), sphase ^ 1u, abort_flag));
            ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
          }
          if (!ok) break;
        }
        const int p0 = __shfl_sync(0xFFFFFFFFu, pg_cur, (c0 - grp) & 31);
        const int p1 = __shfl_sync(0xFFFFFFFFu, pg_cur, (c0 - grp + 1) & 31);
        const int p2 = __shfl_sync(0xFFFFFFFFu, pg_cur, (c0 - grp + 2) & 31);
        const int p3 = __shfl_sync(0xFFFFFFFFu, pg_cur, (c0 - grp + 3) & 31);
        if (lane == 0) {
          const uint32_t bar = bar_full(stage);
          if (j == 0) {
            uint32_t bytes = (uint32_t)(ncol * g.R * 128);
            if (WIDE && tl + 1 < t1)
              bytes += (uint32_t)(min(g.cpt, cend - c0 - g.cpt) * g.R * 128);
            mbar_arrive_expect_tx(bar, bytes);
          }
          const uint32_t dst = WIDE ? sb + kOffStages + (stage * 2 + j) * kTileBytes
                                    : sb + kOffStages + stage * kTileBytes;
          for (int k = 0; k < ncol; ++k) {
            const int c = c0 + k;
            const int pg = k == 0 ? p0 : (k == 1 ? p1 : (k == 2 ? p2 : p3));
            const int y = pg * g.rows_per_page + row_off_of(c, g.split);
            tma_load_2d_hint(dst + k * g.R * 128, &tmk, 0, y, bar, pol);
          }
#ifdef ICP_TIMELINE
          if (issued == 0) ICP_STAMP(2);
          ICP_STAMP(3);
#endif
        }
        __syncwarp();
        if (!WIDE || j == 1 || tl + 1 == t1) {
          ++issued;
          if (++stage == (WIDE ? NS / 2 : NS)) {
            stage = 0;
            sphase ^= 1u;
          }
        }
      }
      if (ok && pp == 0)
        count_bad_entry(a, b, rv, btrow, __reduce_min_sync(0xFFFFFFFFu, first_bad), lane);
    }
    if (*abort_flag && lane == 0) {
      // let copies still in flight land before the CTA exits
      constexpr int nst = WIDE ? NS / 2 : NS;
      const long long first = issued > nst ? issued - nst : 0;
      for (long long n = first; n < issued; ++n)
        if (NPROD == 1 || (int)(n & 1) == pp)
          mbar_wait_drain(bar_full((int)(n % nst)), (uint32_t)((n / nst) & 1));
      if (pp == 0 && last_qslot >= 0)
        mbar_wait_drain(bar_qfull(last_qslot), (last_qslot ? qph1 : qph0) ^ 1u);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    // The whole warp runs the loop, every lane waits, and the lane
    // elect.sync picks issues each MMA and commit; the warp-uniform
    // descriptors then stay in uniform registers.  A lone issuing thread
    // was slower everywhere: the prefill window 54.6 against 52.0 us, the
    // batched decode scorer 0.785 against 0.825 of the copy peak.
    {
      const uint32_t idesc = idesc_f8_f32(128, (int)kAccCols);
#ifdef ICP_TIMELINE
      long long mma_tiles = 0;
#endif
      int stage = 0, acc = 0;
      uint32_t sphase = 0, aphase = 0;
      uint32_t qph0 = 0, qph1 = 0;
      int qslot = 0;
      SegmentWalker walk(prefix, nbatch, g0, g1, WIDE ? kWideRequestUnits : 0);
      int b, t0, t1;
      bool ok = true;
      while (ok && walk.next(b, t0, t1)) {
        ok = mbar_wait(bar_qfull(qslot), qslot ? qph1 : qph0, abort_flag);
        ok = __all_sync(0xFFFFFFFFu, ok);  // the lanes leave together
        if (!ok) break;
        const uint32_t qaddr = sb + L::off_q + qslot * L::q_bytes;
        if constexpr (WIDE) {
          // a pair of tiles is one 256-row B operand; each of the record's
          // row halves (the second only past 32 tokens) is one item: an
          // N = 256 MMA group (N = 128 for a segment's odd last tile) into
          // one of two 256-column accumulators, items alternating
          const int nh = req_view(a, b).ntok > kPlanTokens / 2 ? 2 : 1;
          for (int tl = t0; ok && tl < t1; tl += 2) {
            const int np = min(2, t1 - tl);
            ICP_TIMED_WARP(20, ok = mbar_wait(bar_full(stage), sphase, abort_flag));
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            const uint32_t kaddr = sb + kOffStages + stage * 2 * kTileBytes;
            const uint32_t id = np == 2 ? idesc_f8_f32(128, 2 * (int)kAccCols) : idesc;
            for (int h = 0; h < nh; ++h) {
              // a sleeping wait: a warp polling here took issue slots from
              // the epilogue warps on its scheduler (51.4 against 49.3 us)
              ICP_TIMED_WARP(21, ok = mbar_wait(bar_tempty(acc), aphase ^ 1u, abort_flag));
              ok = __all_sync(0xFFFFFFFFu, ok);
              if (!ok) break;
              tc_fence_after();
              const uint32_t d = tmem_base + (uint32_t)acc * (2 * kAccCols);
              const uint32_t qh = qaddr + (uint32_t)h * (128 * 128);
              // K steps of 32 bytes advance both start addresses by 2 (16-byte units)
              const uint64_t da = smem_desc_sw128(qh), db = smem_desc_sw128(kaddr);
#pragma unroll
              for (int k = 0; k < 4; ++k)
                mma_f8_elect(d, da + 2u * k, db + 2u * k, id, k > 0 ? 1u : 0u);
              mma_commit_elect(bar_tfull(acc));
              if (++acc == 2) {
                acc = 0;
                aphase ^= 1u;
              }
            }
            if (!ok) break;
            mma_commit_elect(bar_empty(stage));
#ifdef ICP_TIMELINE
            if (mma_tiles++ == 0 && lane == 0) ICP_STAMP(4);
            if (lane == 0) ICP_STAMP(5);
#endif
            if (++stage == NS / 2) {
              stage = 0;
              sphase ^= 1u;
            }
          }
        } else {
          for (int tl = t0; tl < t1; ++tl) {
            ok = mbar_wait(bar_full(stage), sphase, abort_flag) &&
                 mbar_wait(bar_tempty(acc), aphase ^ 1u, abort_flag);
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t kaddr = sb + kOffStages + stage * kTileBytes;
            const uint32_t d = tmem_base + (uint32_t)acc * kAccCols;
            // K steps of 32 bytes advance both start addresses by 2 (16-byte units)
            const uint64_t da = smem_desc_sw128(qaddr), db = smem_desc_sw128(kaddr);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8_elect(d, da + 2u * k, db + 2u * k, idesc, k > 0 ? 1u : 0u);
            mma_commit_elect(bar_empty(stage));
            mma_commit_elect(bar_tfull(acc));
#ifdef ICP_TIMELINE
            if (mma_tiles++ == 0 && lane == 0) ICP_STAMP(4);
            if (lane == 0) ICP_STAMP(5);
#endif
            if (++stage == NS) {
              stage = 0;
              sphase ^= 1u;
            }
            if (++acc == kAcc) {
              acc = 0;
              aphase ^= 1u;
            }
          }
        }
        if (!ok) break;
        mma_commit_elect(bar_qempty(qslot));
        if (qslot) qph1 ^= 1u; else qph0 ^= 1u;
        qslot ^= 1;
      }
      if (*abort_flag) {
        // every MMA issued so far must finish before TMEM is released
        mma_commit_elect(bar_done);
        mbar_wait_drain(bar_done, 0);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;      // TMEM lane quarter this warp may access
    const int e = warp - 2;      // owns tiles i with i % 4 == e, accumulator e
    const int et = threadIdx.x - 64;
    if (a.pdl) pdl_wait();       // no global write before the preceding kernel is done
    for (int b = blockIdx.x; b < nbatch; b += gridDim.x) {
      const ReqView rv = req_view(a, b);
      const int u = units_of(rv.seq_len, a.page_size, g.split);
      const int wcols = (units_of(rv.full_len, a.page_size, g.split) + 3) & ~3;
      if (wcols > a.cols && et == 0 && a.errors) atomicAdd(a.errors, 1);  // plane too narrow
      const int rows = 4 * rv.ntok;
      if constexpr (!FUSED) {
        // columns [units, round_up(the request's units, 4)) of the rows this
        // CTA owns: padding, or blocks past every one of the rows' tokens
        const int npad = min(wcols, a.cols) - min(u, a.cols);
        for (int k = et; k < npad * rows; k += kEpiThreads) {
          const int r = k / npad, c = u + k % npad;
          a.score_out[((long long)rv.tok0 * 4 + r) * a.cols + c] = -INFINITY;
        }
      } else if (et == 0) {
        // where the merge kernel finds this request's partial lists
        ReqInfo in;
        in.total = (int)total;
        in.nunits = u;
        if (prefix[b + 1] > prefix[b]) {
          in.i0 = cta_of(total, gridDim.x, prefix[b]);
          in.i1 = cta_of(total, gridDim.x, prefix[b + 1] - 1);
        } else {
          in.i0 = 0;
          in.i1 = -1;
        }
        reinterpret_cast<ReqInfo *>(a.ws_counters)[b] = in;
        (void)rows;
      }
    }
    uint32_t aphase = 0;
    int idx = 0;
    int pi = 0;          // WIDE: the CTA's (tile pair, row half) item counter
    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)e * kAccCols;
    unsigned long long *lk = nullptr;
    int *lfid = nullptr;
    float *lfsc = nullptr;
    if constexpr (FUSED) {
      uint8_t *wl = gb + L::off_lists + e * kWarpListBytes;
      lk = reinterpret_cast<unsigned long long *>(wl);
      lfid = reinterpret_cast<int *>(wl + 16 * 32 * 8);
      lfsc = reinterpret_cast<float *>(wl + 16 * 32 * 8 + 16 * 32 * 4);
    }
    SegmentWalker walk(prefix, nbatch, g0, g1, WIDE ? kWideRequestUnits : 0);
    int b, t0, t1;
    bool ok = true;
    while (walk.next(b, t0, t1)) {
      if (!FUSED && !ok) break;
      const ReqView rv = req_view(a, b);
      const int seq_len = rv.seq_len;
      const int nunits = units_of(seq_len, a.page_size, g.split);
      LaneTop lt;
      lt.cnt = 0;
      lt.kmin = 0;
      lt.fcnt = 0;
      lt.nvp = 0;
      if constexpr (FUSED) {
        if (lane < 4 * rv.ntok) lt.nvp = a.nvp[rv.tok0 + (lane >> 2)];
#pragma unroll
        for (int j = 0; j < kTopK; ++j) lk[j * 32 + lane] = 0ull;
      }
      if constexpr (WIDE) {
        // every (tile pair, row half) item: pi counts the CTA's items as the
        // MMA thread does, item pi sits in accumulator pi & 1, and set s
        // takes the items of accumulator s, the pair's tiles in turn, for
        // this warp's lane quarter (tokens 32 h + 8 q .. 32 h + 8 q + 7)
        const int set = (warp - 2) >> 2;
        const int nh = rv.ntok > kPlanTokens / 2 ? 2 : 1;
        for (int tl = t0; ok && tl < t1; tl += 2) {
          const int np = min(2, t1 - tl);
          for (int h = 0; ok && h < nh; ++h, ++pi) {
            if ((pi & 1) != set) continue;
            const int acc = set;
            const uint32_t wph = (uint32_t)(pi >> 1) & 1u;
            // every lane waits (no lane-0 branch and broadcast)
#ifdef ICP_TIMELINE
            if (warp == 2 && lane == 0) ICP_TIMED(22, ok = mbar_wait(bar_tfull(acc), wph, abort_flag));
            else ok = mbar_wait(bar_tfull(acc), wph, abort_flag);
#else
            ok = mbar_wait(bar_tfull(acc), wph, abort_flag);
#endif
            ok = __all_sync(0xFFFFFFFFu, ok);
            if (!ok) break;
            tc_fence_after();
            const uint32_t tj = tmem_base + ((uint32_t)(q * 32) << 16) +
                                (uint32_t)acc * (2 * kAccCols);
            const int rowq = h * 128 + q * 32;
            // the second tile (if any) hands the accumulator back
            for (int j = 0; j < np; ++j)
              epilogue_tile_wide<(WIDE ? RW : 128)>(a, tj + (uint32_t)j * kAccCols, lane, rowq,
                                                    rv.tok0, rv.ntok, tl + j, nunits, seq_len,
                                                    bar_tempty(acc), j == np - 1);
#ifdef ICP_TIMELINE
            if (warp == 2 && lane == 0) {
              if (pi == 0) ICP_STAMP(6);
              ICP_STAMP(10);
            }
#endif
          }
        }
      } else {
        // first tile of this segment that belongs to this warp
        int tl = t0 + ((e - idx) % 4 + 4) % 4;
        const int seg_tiles = t1 - t0;
        idx += seg_tiles;
        for (; ok && tl < t1; tl += 4) {
          // every lane waits (a lane-0 wait and broadcast was slower: the
          // batched decode scorer 0.763 against 0.785 of the copy peak)
          ok = mbar_wait(bar_tfull(e), aphase, abort_flag);
          ok = __all_sync(0xFFFFFFFFu, ok);
          if (!ok) break;
          tc_fence_after();
          if (g.R == 128)
            epilogue_tile<128, FUSED>(a, taddr, lane, 0, rv.tok0, rv.ntok, tl, nunits, seq_len,
                                      bar_tempty(e), lt, lk, lfid, lfsc);
          else if (g.R == 64)
            epilogue_tile<64, FUSED>(a, taddr, lane, 0, rv.tok0, rv.ntok, tl, nunits, seq_len,
                                     bar_tempty(e), lt, lk, lfid, lfsc);
          else
            epilogue_tile<32, FUSED>(a, taddr, lane, 0, rv.tok0, rv.ntok, tl, nunits, seq_len,
                                     bar_tempty(e), lt, lk, lfid, lfsc);
          aphase ^= 1u;
#ifdef ICP_TIMELINE
          if (lane == 0) {
            if (aphase == 1u && idx == seg_tiles && tl - t0 < 4) ICP_STAMP(6 + e);
            ICP_STAMP(10);
          }
#endif
        }
      }
      if constexpr (FUSED) {
        // publish this warp's lists of the segment, then count the segment's
        // tiles; the CTA that completes the request merges it
        const int pidx = (blockIdx.x + b) * 4 + e;
        if (lane < 4 * rv.ntok) {
          PartialRec *pr = partial_rec(a, pidx, lane);
          unsigned long long mxk = 0;
#pragma unroll
          for (int j = 0; j < kTopK; ++j) {
            const unsigned long long x = lk[j * 32 + lane];
            pr->keys[j] = x;
            mxk = x > mxk ? x : mxk;
          }
          pr->max = mxk;
          pr->fcount = lt.fcnt;
          for (int j = 0; j < lt.fcnt; ++j) {
            pr->fid[j] = lfid[j * 32 + lane];
            pr->fsc[j] = lfsc[j * 32 + lane];
          }
        }
      }
    }
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag && a.errors) atomicAdd(a.errors, 1);
  if (threadIdx.x == 0) ICP_STAMP(11);
}

template <bool FUSED, bool WIDE = false, int NPROD = 1>
size_t smem_bytes_for(int batch) {
  static_assert(PrefixOffset<FUSED, WIDE, NPROD>::value % 16 == 0, "prefix alignment");
  return 1024 + PrefixOffset<FUSED, WIDE, NPROD>::value +
         sizeof(int) * (size_t)(batch + 1 + kThreadsWide / 32);
}

}  // namespace


size_t score_smem_bytes(int batch) { return smem_bytes_for<false>(batch); }

cudaError_t score_prepare(int device) {
  (void)device;
  cudaError_t e = cudaFuncSetAttribute(score_kernel<false, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)smem_bytes_for<false>(kMaxBatchDevice));
  if (e != cudaSuccess) return e;
  // the prefill scorer: one kernel per page-slice height, each with a
  // single epilogue (a run-time choice among three raised its register peak)
  for (auto k : {score_kernel<false, true, 1, 128>, score_kernel<false, true, 1, 64>,
                 score_kernel<false, true, 1, 32>}) {
    e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)smem_bytes_for<false, true>(kMaxBatchDevice));
    if (e != cudaSuccess) return e;
  }
  e = cudaFuncSetAttribute(score_kernel<false, false, 2>,
                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                           (int)smem_bytes_for<false, false, 2>(kMaxBatchDevice));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(score_kernel<true, false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)smem_bytes_for<true>(kMaxBatchDevice));
}

cudaError_t launch_score(const CUtensorMap &tmk, const CUtensorMap &tmq, const ScoreArgs &a,
                         int grid, cudaStream_t stream) {
  if (a.wide) {
    const size_t smem = smem_bytes_for<false, true>(a.batch);
    if (a.g.R == 128)
      score_kernel<false, true, 1, 128><<<grid, kThreadsWide, smem, stream>>>(tmk, tmq, a);
    else if (a.g.R == 64)
      score_kernel<false, true, 1, 64><<<grid, kThreadsWide, smem, stream>>>(tmk, tmq, a);
    else
      score_kernel<false, true, 1, 32><<<grid, kThreadsWide, smem, stream>>>(tmk, tmq, a);
    return cudaGetLastError();
  }
  // a tile of two or four page slices is as many TMA boxes: two producer
  // warps issue them
  const bool two = a.g.cpt >= 2;
  if (!a.pdl) {
    if (two)
      score_kernel<false, false, 2><<<grid, BlockThreads<false, 2>::value,
                                      smem_bytes_for<false, false, 2>(a.batch), stream>>>(tmk,
                                                                                          tmq, a);
    else
      score_kernel<false, false><<<grid, kThreads, smem_bytes_for<false>(a.batch), stream>>>(
          tmk, tmq, a);
    return cudaGetLastError();
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(two ? BlockThreads<false, 2>::value : kThreads);
  cfg.dynamicSmemBytes = two ? smem_bytes_for<false, false, 2>(a.batch)
                            : smem_bytes_for<false>(a.batch);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return two ? cudaLaunchKernelEx(&cfg, score_kernel<false, false, 2>, tmk, tmq, a)
             : cudaLaunchKernelEx(&cfg, score_kernel<false, false>, tmk, tmq, a);
}

cudaError_t launch_score_select(const CUtensorMap &tmk, const CUtensorMap &tmq, ScoreArgs a,
                                int grid, cudaStream_t stream) {
  // (a second producer made the fused scorer slower on the sharded layout)
  grid = grid > kFusedMaxGrid ? kFusedMaxGrid : grid;
  score_kernel<true, false><<<grid, kThreads, smem_bytes_for<true>(a.batch), stream>>>(tmk, tmq,
                                                                                       a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return launch_fused_merge(a, grid, stream);
}

}  // namespace icp

#ifdef ICP_TIMELINE
extern "C" int icp_timeline_read(unsigned long long *dst, int ctas, int clear) {
  if (!dst || ctas < 0 || ctas > icp::kTimelineCtas) return 1;
  const size_t n = (size_t)ctas * icp::kTimelineSlots * sizeof(unsigned long long);
  if (cudaMemcpyFromSymbol(dst, icp::g_timeline, n) != cudaSuccess) return 2;
  if (clear) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, icp::g_timeline) != cudaSuccess ||
        cudaMemset(p, 0, sizeof(icp::g_timeline)) != cudaSuccess || cudaDeviceSynchronize())
      return 2;
  }
  return 0;
}
#endif
