// icp_score.cu - decode index scorer (msa_icp_decode_index_score_sharded).
//
// What it computes: for every request b, token j (position
// seq_len_b - dql + j), head h and plane column c of the request,
//   score_out[t][h][c] = max over the column's keys at positions <= the
//                        token's position of dot(deq(q[t,h,:]), deq(k[key,:]))
// (-inf when no key is visible), for c < round_up(columns, 4); the other
// columns are not written.
//
// How (one persistent CTA per SM, 192 threads, warp-specialised):
//   warp 0     TMA producer: streams the 128-row K tiles of the CTA's share of
//              all requests' pages (each page read once per call) into an
//              8-stage shared-memory ring, and each request's queries once.
//   warp 1     MMA issuer: per tile, 4 x tcgen05.mma kind::f8f6f4 (M=128 keys,
//              N = 16 or 32 query rows, K = 32) into an fp32 TMEM accumulator.
//              All 4 heads and all dql tokens share one K tile.
//   warps 2-5  epilogue: tcgen05.ld of the accumulator (thread = key, registers
//              = query rows), causal mask, max over the column's keys by a
//              transposed warp butterfly (plus shared memory across warps when a
//              column spans several warps), and the plane store.
// The tiles of all requests form one list that is cut into gridDim.x equal
// contiguous ranges, so every CTA streams the same number of K bytes.
// Products of two e4m3 values are exact in fp32; the MMA sums 128 of them in
// fp32.  The per-key arithmetic does not depend on where the key sits in the
// tile, so sharded and unsharded layouts give identical key scores.
#include "icp_device.cuh"
#include "icp_internal.h"

namespace icp {
namespace {

constexpr int kStages = 8;
constexpr int kAcc = 8;
constexpr int kTileBytes = 128 * 128;  // 128 K rows x 128 fp8
constexpr int kQBytes = 32 * 128;      // up to 32 query rows x 128 fp8
constexpr int kThreads = 192;
constexpr uint32_t kTmemCols = 256;    // kAcc accumulators of up to 32 columns
constexpr int kNumBars = 2 * kStages + 2 * kAcc + 4 + 1;

// Shared-memory carve-up (offsets from a 1024-byte aligned base).
constexpr uint32_t kOffStages = 0;
constexpr uint32_t kOffQ = kOffStages + kStages * kTileBytes;
constexpr uint32_t kOffBars = kOffQ + 2 * kQBytes;
constexpr uint32_t kOffMisc = kOffBars + ((kNumBars * 8 + 127) / 128) * 128;
constexpr uint32_t kOffRed = kOffMisc + 128;
constexpr uint32_t kOffPrefix = kOffRed + 2 * 4 * 32 * 4;

__device__ __forceinline__ int units_of(int seq_len, int page_size, int split) {
  const int u = split ? 128 : page_size;
  return seq_len <= 0 ? 0 : (seq_len + u - 1) / u;
}

// Walks the CTA's tile range [g0, g1) request by request.
struct SegmentWalker {
  const int *prefix;  // prefix[b] = tiles of requests < b, prefix[batch] = total
  int batch;
  int g, g1, b;
  __device__ SegmentWalker(const int *p, int nb, int g0_, int g1_)
      : prefix(p), batch(nb), g(g0_), g1(g1_), b(0) {
    // largest b with prefix[b] <= g0
    int lo = 0, hi = nb;  // invariant: prefix[lo] <= g0
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= g) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  // Next segment: request rb, local tiles [t0, t1).  False when done.
  __device__ bool next(int &rb, int &t0, int &t1) {
    if (g >= g1) return false;
    while (b < batch && prefix[b + 1] <= g) ++b;
    if (b >= batch) return false;
    rb = b;
    t0 = g - prefix[b];
    t1 = min(g1, prefix[b + 1]) - prefix[b];
    g = prefix[b] + t1;
    ++b;
    return true;
  }
};

__device__ __forceinline__ int page_slot_of(int c, int split) { return split ? (c >> 1) : c; }
__device__ __forceinline__ int row_off_of(int c, int split) { return split ? (c & 1) * 128 : 0; }

// Max over the 32 lanes of the warp for each of N values, done as a
// transposed butterfly: each exchange halves the values a lane keeps, so the
// whole reduction costs about N shuffles per lane.  On return v[0] of lane l
// holds the maximum for value index l (N = 32) or l >> 1 (N = 16).
template <int N>
__device__ __forceinline__ void warp_transpose_max(float (&v)[N], int lane) {
  static_assert(N == 16 || N == 32, "N");
#pragma unroll
  for (int o = 16, n = N; o >= 1; o >>= 1) {
    if (n > 1) {
      const bool upper = (lane & o) != 0;
      const int h = n >> 1;
#pragma unroll
      for (int i = 0; i < h; ++i) {
        const float send = upper ? v[i] : v[i + h];
        const float keep = upper ? v[i + h] : v[i];
        const float got = __shfl_xor_sync(0xFFFFFFFFu, send, o);
        v[i] = fmaxf(keep, got);
      }
      n = h;
    } else {
      v[0] = fmaxf(v[0], __shfl_xor_sync(0xFFFFFFFFu, v[0], o));
    }
  }
}

__device__ __forceinline__ void named_bar_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

template <int NQ>
__device__ __forceinline__ void epilogue_tile(const ScoreArgs &a, uint32_t taddr, int q, int lane,
                                              int b, int tl, int nunits, int seq_len,
                                              float *red_buf, int par) {
  float v[NQ];
  {
    float lo[16];
    tmem_ld16(taddr, lo);
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = lo[i];
    if constexpr (NQ == 32) {
      float hi[16];
      tmem_ld16(taddr + 16, hi);
#pragma unroll
      for (int i = 0; i < 16; ++i) v[16 + i] = hi[i];
    }
  }
  tmem_wait_ld();
  (void)b;
  const ScoreGeom &g = a.g;
  const int cc = (q * 32) / g.R;
  const int c = tl * g.cpt + cc;
  const int i = (q * 32) % g.R + lane;
  const long long pos0 = g.split ? (long long)c * 128
                                 : (long long)c * a.page_size + (long long)a.rank * g.rows_per_page;
  const long long pos = pos0 + i;
  const long long pfirst = (long long)seq_len - a.dql;  // position of token 0
  if (pos > pfirst) {
#pragma unroll
    for (int r = 0; r < NQ; ++r)
      if (pos > pfirst + (r >> 2)) v[r] = -INFINITY;
  }
  warp_transpose_max<NQ>(v, lane);
  float m = v[0];
  const int wpc = g.R >> 5;  // warps per column
  bool writer = true;
  if (wpc > 1) {
    red_buf[(par * 4 + q) * 32 + lane] = m;
    named_bar_sync(1, 128);
    writer = (q % wpc) == 0;
    if (writer) {
      for (int w = 1; w < wpc; ++w) m = fmaxf(m, red_buf[(par * 4 + q + w) * 32 + lane]);
    }
  }
  if (writer && c < nunits && c < a.cols) {
    const int row = (NQ == 32) ? lane : (lane >> 1);
    const bool holder = (NQ == 32) || ((lane & 1) == 0);
    if (holder && row < 4 * a.dql) {
      const long long prow = (long long)b * a.dql * 4 + row;
      a.score_out[prow * a.cols + c] = m + 0.0f;  // + 0 folds -0 onto +0
    }
  }
}

__global__ void __launch_bounds__(kThreads, 1)
score_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmq,
             const ScoreArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t *gb = smem_raw + (sb - raw);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const ScoreGeom g = a.g;

  auto bar_full = [&](int s) { return sb + kOffBars + 8u * s; };
  auto bar_empty = [&](int s) { return sb + kOffBars + 8u * (kStages + s); };
  auto bar_tfull = [&](int i) { return sb + kOffBars + 8u * (2 * kStages + i); };
  auto bar_tempty = [&](int i) { return sb + kOffBars + 8u * (2 * kStages + kAcc + i); };
  auto bar_qfull = [&](int i) { return sb + kOffBars + 8u * (2 * kStages + 2 * kAcc + i); };
  auto bar_qempty = [&](int i) { return sb + kOffBars + 8u * (2 * kStages + 2 * kAcc + 2 + i); };
  const uint32_t bar_done = sb + kOffBars + 8u * (2 * kStages + 2 * kAcc + 4);

  volatile int *misc = reinterpret_cast<volatile int *>(gb + kOffMisc);  // [0] tmem, [1] abort
  float *red_buf = reinterpret_cast<float *>(gb + kOffRed);
  int *prefix = reinterpret_cast<int *>(gb + kOffPrefix);
  int *partial = prefix + a.batch + 1;  // kThreads scratch ints

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(bar_full(s), 1);
      mbar_init(bar_empty(s), 1);
    }
    for (int i = 0; i < kAcc; ++i) {
      mbar_init(bar_tfull(i), 1);
      mbar_init(bar_tempty(i), 4);
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
  if (warp == 1) tmem_alloc(sb + kOffMisc, kTmemCols);

  // Tiles per request and their prefix sums (chunked block scan).
  {
    const int nb = a.batch;
    const int chunk = (nb + kThreads - 1) / kThreads;
    const int lo = threadIdx.x * chunk, hi = min(nb, lo + chunk);
    int sum = 0;
    for (int b = lo; b < hi; ++b) {
      const int u = units_of(a.seq_lens[b], a.page_size, g.split);
      sum += (u + g.cpt - 1) / g.cpt;
    }
    partial[threadIdx.x] = sum;
    __syncthreads();
    if (threadIdx.x == 0) {
      int run = 0;
      for (int i = 0; i < kThreads; ++i) {
        const int x = partial[i];
        partial[i] = run;
        run += x;
      }
      prefix[nb] = run;
    }
    __syncthreads();
    int run = partial[threadIdx.x];
    for (int b = lo; b < hi; ++b) {
      prefix[b] = run;
      const int u = units_of(a.seq_lens[b], a.page_size, g.split);
      run += (u + g.cpt - 1) / g.cpt;
    }
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = (uint32_t)misc[0];

  const long long total = prefix[a.batch];
  const int g0 = (int)(total * blockIdx.x / gridDim.x);
  const int g1 = (int)(total * (blockIdx.x + 1) / gridDim.x);
  volatile int *abort_flag = misc + 1;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint64_t pol = policy_evict_first();
    int stage = 0;
    uint32_t sphase = 0;
    uint32_t qph[2] = {0u, 0u};
    int qslot = 0;
    long long issued = 0;
    int last_qslot = -1;
    SegmentWalker walk(prefix, a.batch, g0, g1);
    int b, t0, t1;
    bool ok = true;
    while (ok && walk.next(b, t0, t1)) {
      const int nunits = units_of(a.seq_lens[b], a.page_size, g.split);
      if (lane == 0) ok = mbar_wait(bar_qempty(qslot), qph[qslot] ^ 1u, abort_flag);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(bar_qfull(qslot), (uint32_t)(g.nq * 128));
        tma_load_2d(sb + kOffQ + qslot * kQBytes, &tmq, 0, b * a.dql * 4, bar_qfull(qslot));
      }
      last_qslot = qslot;
      qph[qslot] ^= 1u;
      qslot ^= 1;
      const int cbeg = t0 * g.cpt;
      const int cend = min(t1 * g.cpt, nunits);
      const int32_t *btrow = a.block_table + (long long)b * a.bt_stride;
      int grp = cbeg;
      int pg_cur = (cbeg + lane < cend) ? btrow[page_slot_of(cbeg + lane, g.split)] : 0;
      int pg_nxt = (cbeg + 32 + lane < cend) ? btrow[page_slot_of(cbeg + 32 + lane, g.split)] : 0;
      for (int tl = t0; tl < t1; ++tl) {
        const int c0 = tl * g.cpt;
        if (c0 >= grp + 32) {
          grp += 32;
          pg_cur = pg_nxt;
          pg_nxt = (grp + 32 + lane < cend) ? btrow[page_slot_of(grp + 32 + lane, g.split)] : 0;
        }
        const int ncol = min(g.cpt, cend - c0);
        if (lane == 0) ok = mbar_wait(bar_empty(stage), sphase ^ 1u, abort_flag);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
        if (!ok) break;
        int pages[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) pages[k] = __shfl_sync(0xFFFFFFFFu, pg_cur, (c0 - grp + k) & 31);
        if (lane == 0) {
          const uint32_t bar = bar_full(stage);
          mbar_arrive_expect_tx(bar, (uint32_t)(ncol * g.R * 128));
          const uint32_t dst = sb + kOffStages + stage * kTileBytes;
          for (int k = 0; k < ncol; ++k) {
            const int c = c0 + k;
            const int y = pages[k] * g.rows_per_page + row_off_of(c, g.split);
            tma_load_2d_hint(dst + k * g.R * 128, &tmk, 0, y, bar, pol);
          }
        }
        __syncwarp();
        ++issued;
        if (++stage == kStages) {
          stage = 0;
          sphase ^= 1u;
        }
      }
    }
    if (*abort_flag && lane == 0) {
      // let copies still in flight land before the CTA exits
      const long long first = issued > kStages ? issued - kStages : 0;
      for (long long n = first; n < issued; ++n)
        mbar_wait_drain(bar_full((int)(n % kStages)), (uint32_t)((n / kStages) & 1));
      if (last_qslot >= 0) mbar_wait_drain(bar_qfull(last_qslot), qph[last_qslot] ^ 1u);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    const uint32_t idesc = idesc_f8_f32(128, g.nq);
    int stage = 0, acc = 0;
    uint32_t sphase = 0, aphase = 0;
    uint32_t qph[2] = {0u, 0u};
    int qslot = 0;
    SegmentWalker walk(prefix, a.batch, g0, g1);
    int b, t0, t1;
    bool ok = true;
    while (ok && walk.next(b, t0, t1)) {
      if (lane == 0) ok = mbar_wait(bar_qfull(qslot), qph[qslot], abort_flag);
      ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
      if (!ok) break;
      const uint32_t qaddr = sb + kOffQ + qslot * kQBytes;
      for (int tl = t0; tl < t1; ++tl) {
        if (lane == 0) {
          ok = mbar_wait(bar_full(stage), sphase, abort_flag) &&
               mbar_wait(bar_tempty(acc), aphase ^ 1u, abort_flag);
          if (ok) {
            tc_fence_after();
            const uint32_t kaddr = sb + kOffStages + stage * kTileBytes;
            const uint32_t d = tmem_base + (uint32_t)(acc * g.nq);
#pragma unroll
            for (int k = 0; k < 4; ++k)
              mma_f8(d, smem_desc_sw128(kaddr + 32 * k), smem_desc_sw128(qaddr + 32 * k), idesc,
                     k > 0 ? 1u : 0u);
            mma_commit(bar_empty(stage));
            mma_commit(bar_tfull(acc));
          }
        }
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
        if (!ok) break;
        if (++stage == kStages) {
          stage = 0;
          sphase ^= 1u;
        }
        if (++acc == kAcc) {
          acc = 0;
          aphase ^= 1u;
        }
      }
      if (!ok) break;
      if (lane == 0) mma_commit(bar_qempty(qslot));
      __syncwarp();
      qph[qslot] ^= 1u;
      qslot ^= 1;
    }
    if (*abort_flag && lane == 0) {
      // every MMA issued so far must finish before TMEM is released
      mma_commit(bar_done);
      mbar_wait_drain(bar_done, 0);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    const int et = threadIdx.x - 64;
    // padding columns [units, round_up(units, 4)) of the requests this CTA owns
    for (int b = blockIdx.x; b < a.batch; b += gridDim.x) {
      const int u = units_of(a.seq_lens[b], a.page_size, g.split);
      const int wcols = (u + 3) & ~3;
      if (wcols > a.cols && et == 0 && a.errors) atomicAdd(a.errors, 1);  // plane too narrow
      const int npad = min(wcols, a.cols) - min(u, a.cols);
      const int rows = 4 * a.dql;
      for (int k = et; k < npad * rows; k += 128) {
        const int r = k / npad, c = u + k % npad;
        a.score_out[((long long)b * a.dql * 4 + r) * a.cols + c] = -INFINITY;
      }
    }
    int acc = 0, par = 0;
    uint32_t aphase = 0;
    SegmentWalker walk(prefix, a.batch, g0, g1);
    int b, t0, t1;
    bool ok = true;
    while (ok && walk.next(b, t0, t1)) {
      const int seq_len = a.seq_lens[b];
      const int nunits = units_of(seq_len, a.page_size, g.split);
      for (int tl = t0; tl < t1; ++tl) {
        if (lane == 0) ok = mbar_wait(bar_tfull(acc), aphase, abort_flag);
        ok = __shfl_sync(0xFFFFFFFFu, ok, 0) != 0;
        if (!ok) break;
        tc_fence_after();
        const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(acc * g.nq);
        if (g.nq == 32)
          epilogue_tile<32>(a, taddr, q, lane, b, tl, nunits, seq_len, red_buf, par);
        else
          epilogue_tile<16>(a, taddr, q, lane, b, tl, nunits, seq_len, red_buf, par);
        // epilogue_tile has read the accumulator (tcgen05.wait::ld inside)
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_tempty(acc));
        par ^= 1;
        if (++acc == kAcc) {
          acc = 0;
          aphase ^= 1u;
        }
      }
    }
    (void)et;
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, kTmemCols);
  }
  if (threadIdx.x == 0 && *abort_flag && a.errors) atomicAdd(a.errors, 1);
}

}  // namespace

size_t score_smem_bytes(int batch) {
  return 1024 + kOffPrefix + sizeof(int) * (size_t)(batch + 1 + kThreads);
}

cudaError_t score_prepare(int device) {
  (void)device;
  return cudaFuncSetAttribute(score_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              (int)score_smem_bytes(4096));
}

cudaError_t launch_score(const CUtensorMap &tmk, const CUtensorMap &tmq, const ScoreArgs &a,
                         int grid, cudaStream_t stream) {
  const size_t smem = score_smem_bytes(a.batch);
  score_kernel<<<grid, kThreads, smem, stream>>>(tmk, tmq, a);
  return cudaGetLastError();
}

}  // namespace icp
