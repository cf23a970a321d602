// icp_fused.cu - second kernel of the fused scorer + Top16 select: merges
// the partial Top16 lists the scorer's epilogue warps wrote per request
// segment into each row's final Top16 (prepare_msa_icp_indexer,
// decode(pool=...): the fused chain leaves no score plane).
#include "icp_device.cuh"
#include "icp_fused.cuh"
#include "icp_internal.h"

namespace icp {
namespace {

// Final Top16 of one (token, head) row from the partial lists that the
// epilogue warps of every CTA covering the token's request wrote, plus the
// request's padding columns [units, round_up(units, 4)), which hold -inf.
// One warp per row; the lists holding the m largest entries are found from
// the lists' maxima (tau = the m-th largest maximum), so at most m * 16
// candidates are read.
__global__ void __launch_bounds__(128)
fused_merge_kernel(const ScoreArgs a, const ReqInfo *info, int grid_a) {
  __shared__ unsigned long long s_mx[4][4 * kFusedMaxGrid];
  __shared__ unsigned long long s_cand[4][kTopK * 16 + 8];
  __shared__ int s_fid[4][kTopK];
  __shared__ float s_fsc[4][kTopK];
  __shared__ int s_flist[4][kTopK];   // lists holding forced entries, in list order
  __shared__ int s_ffirst[4][kTopK];  // slot of each such list's first forced entry
  __shared__ unsigned long long s_sel[4][kTopK];  // the m largest candidates by rank
  __shared__ int s_win[4][kTopK];                 // winner lists by rank
  // wait for the fused scorer (programmatic dependent launch)
  asm volatile("griddepcontrol.wait;" ::: "memory");

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.x * 4 + warp;   // t * 4 + h
  const int T = a.batch * a.dql;
  if (row >= T * 4) return;
  const int t = row >> 2, h = row & 3;
  const int b = t / a.dql;
  const int r = (t - b * a.dql) * 4 + h;   // query row inside the request
  unsigned long long *mx = s_mx[warp];
  unsigned long long *cand = s_cand[warp];
  int *fbuf_id = s_fid[warp];
  float *fbuf_sc = s_fsc[warp];
  int *flist = s_flist[warp];
  int *ffirst = s_ffirst[warp];

  const ReqInfo in = info[b];
  const long long total = in.total;
  const int G = grid_a;
  const int i0 = in.i0;
  const int P = in.i1 >= in.i0 ? (in.i1 - in.i0 + 1) * 4 : 0;
  const int nunits = in.nunits;
  const int wcols = min((nunits + 3) & ~3, a.cols);
  const int nvp = a.nvp[t];
  auto pidx_of = [&](int k) { return (i0 + (k >> 2) + b) * 4 + (k & 3); };
  // a CTA in [i0, i1] with an empty tile range never wrote lists for b
  auto part_valid = [&](int k) {
    const int i = i0 + (k >> 2);
    return total * i / G < total * (i + 1) / G;
  };

  // one pass over the lists: each list's maximum (to the shared cache),
  // and the lists holding forced entries (every forced id was seen by
  // exactly one list) with the slot of their first entry, in list order
  int nfl = 0, nfe = 0;  // lists with forced entries, forced entries so far
  for (int k0 = 0; k0 < P; k0 += 32) {
    const int k = k0 + lane;
    unsigned long long mxk = 0;
    int fc = 0;
    if (k < P && part_valid(k)) {
      const PartialRec *pr = partial_rec(a, pidx_of(k), r);
      mxk = __ldcg(&pr->max);
      fc = __ldcg(&pr->fcount);
    }
    if (k < P) mx[k] = mxk;
    int incl = fc;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xFFFFFFFFu, incl, o);
      if (lane >= o) incl += y;
    }
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, fc > 0);
    if (fc > 0) {
      const int pos = nfl + __popc(bal & ((1u << lane) - 1u));
      if (pos < kTopK) {
        flist[pos] = k;
        ffirst[pos] = nfe + incl - fc;
      }
    }
    nfl += __popc(bal);
    nfe += __shfl_sync(0xFFFFFFFFu, incl, 31);
  }
  nfl = min(nfl, kTopK);
  const int nf_lists = min(nfe, kTopK);
  // forced ids among the padding columns (no key: score -inf) come after
  int nf = nf_lists;
  for (int c = nunits; c < wcols; ++c) {
    const int id = c * a.index_scale + a.index_offset;
    if (id < nvp && forced_id(id, nvp, a.init_blocks, a.local_blocks) && nf < kTopK) {
      if (lane == 0) {
        fbuf_id[nf] = id;
        fbuf_sc[nf] = -INFINITY;
      }
      ++nf;
    }
  }
  const int m = kTopK - nf;
  __syncwarp();
  // tau = m-th largest list maximum; the lists holding keys >= tau are
  // exactly the m lists with the largest maxima (the winners).  Up to 32
  // lists: every lane ranks its list's maximum against the others (the
  // maxima are distinct keys); more lists: rounds of a warp maximum.
  unsigned long long prev = ~0ull, tau = 0;
  int found = 0, my_winner = -1;
  if (m > 0 && P <= 32) {
    const unsigned long long x = lane < P ? mx[lane] : 0ull;
    int rank = 0;
#pragma unroll 8
    for (int j = 0; j < 32; ++j) rank += __shfl_sync(0xFFFFFFFFu, x, j) > x ? 1 : 0;
    const bool win = x != 0ull && rank < m;
    found = __popc(__ballot_sync(0xFFFFFFFFu, win));
    if (win) s_win[warp][rank] = lane;
    const unsigned lastm = __ballot_sync(0xFFFFFFFFu, x != 0ull && rank == m - 1);
    tau = found < m ? 1ull : __shfl_sync(0xFFFFFFFFu, x, lastm ? __ffs(lastm) - 1 : 0);
    __syncwarp();
    if (lane < found) my_winner = s_win[warp][lane];
    __syncwarp();
  }
  for (int rd = 0; P > 32 && rd < m; ++rd) {
    unsigned long long local = 0;
    int lidx = -1;
    for (int k = lane; k < P; k += 32) {
      const unsigned long long x = mx[k];
      if (x < prev && x > local) {
        local = x;
        lidx = k;
      }
    }
    const unsigned long long w = warp_max_key(local);
    if (w == 0) break;
    const int src = __ffs(__ballot_sync(0xFFFFFFFFu, local == w)) - 1;
    const int widx = __shfl_sync(0xFFFFFFFFu, lidx, src);
    if (lane == rd) my_winner = widx;
    prev = w;
    tau = w;
    ++found;
  }
  if (P > 32 && found < m) tau = 1;  // fewer than m lists hold entries: take all of them
  // one round of loads: forced entry `lane` (lane < nf_lists) from its list,
  // and every winner's 16 keys (lane L reads entries L, L + 32, ... of the
  // found * 16 keys)
  int f_id = 0;
  float f_sc = -INFINITY;
  if (lane < nf_lists) {
    int li = 0;
    while (li + 1 < nfl && ffirst[li + 1] <= lane) ++li;
    const PartialRec *pr = partial_rec(a, pidx_of(flist[li]), r);
    f_id = __ldcg(&pr->fid[lane - ffirst[li]]);
    f_sc = __ldcg(&pr->fsc[lane - ffirst[li]]);
  }
  unsigned long long kv[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int q = lane + 32 * j;
    const int wi = q >> 4;
    const int k = __shfl_sync(0xFFFFFFFFu, my_winner, wi & 31);
    kv[j] = (wi < found) ? __ldcg(&partial_rec(a, pidx_of(k), r)->keys[q & 15]) : 0ull;
  }
  if (lane < nf_lists) {
    fbuf_id[lane] = f_id;
    fbuf_sc[lane] = f_sc;
  }
  int nc = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const bool keep = kv[j] != 0 && kv[j] >= tau;
    const unsigned bal = __ballot_sync(0xFFFFFFFFu, keep);
    if (keep) cand[nc + __popc(bal & ((1u << lane) - 1u))] = kv[j];
    nc += __popc(bal);
  }
  for (int c = nunits; c < wcols; ++c) {
    const int id = c * a.index_scale + a.index_offset;
    if (id < nvp && !forced_id(id, nvp, a.init_blocks, a.local_blocks)) {
      const unsigned long long key = make_key(-INFINITY, id);
      if (key >= tau) {
        if (lane == 0) cand[nc] = key;
        ++nc;
      }
    }
  }
  __syncwarp();
  // the m largest candidates; lane nf + rd receives the rd-th.  Up to 64
  // candidates: each is placed by its rank (the keys are distinct); more:
  // rounds of a warp maximum.
  unsigned long long mine = 0;
  int nch = 0;
  if (nc <= 64) {
    for (int j = lane; j < nc; j += 32) {
      const unsigned long long c = cand[j];
      int rank = 0;
      for (int i = 0; i < nc; ++i) rank += cand[i] > c ? 1 : 0;
      if (rank < m) s_sel[warp][rank] = c;
    }
    nch = min(nc, max(m, 0));
    __syncwarp();
    if (lane >= nf && lane < nf + nch) mine = s_sel[warp][lane - nf];
  }
  unsigned long long cl[9];
  unsigned long long lmax = 0;
#pragma unroll
  for (int j = 0; j < 9; ++j) {
    const int k = lane + 32 * j;
    cl[j] = (nc > 64 && k < nc) ? cand[k] : 0ull;
    lmax = cl[j] > lmax ? cl[j] : lmax;
  }
  for (int rd = 0; nc > 64 && rd < m; ++rd) {
    const unsigned long long w = warp_max_key(lmax);
    if (w == 0) break;
    if (lane == nf + rd) mine = w;
    ++nch;
    if (lmax == w) {
      lmax = 0;
#pragma unroll
      for (int j = 0; j < 9; ++j) {
        if (cl[j] == w) cl[j] = 0;
        lmax = cl[j] > lmax ? cl[j] : lmax;
      }
    }
  }
  const int n = nf + nch;
  int my_id = 0x7FFFFFFF;
  float my_sc = -INFINITY;
  if (lane < nf) {
    my_id = fbuf_id[lane];
    my_sc = fbuf_sc[lane];
  } else if (lane < n) {
    my_id = key_id(mine);
    my_sc = unord_float((uint32_t)(mine >> 32));
  }
  int out_id;
  float out_sc;
  sort_by_id_16(lane, n, my_id, my_sc, out_id, out_sc, fbuf_id, fbuf_sc);
  if (lane < kTopK) {
    const long long o = (long long)row * kTopK + lane;
    a.out_scores[o] = out_sc;
    a.out_ids[o] = out_id;
  }
}

}  // namespace

size_t fused_workspace_bytes(int batch, int dql) {
  const size_t counters = ((size_t)batch * sizeof(ReqInfo) + 255) / 256 * 256;
  const size_t records =
      (size_t)(kFusedMaxGrid + batch) * 4 * (size_t)(4 * dql) * sizeof(PartialRec);
  return counters + records;
}

cudaError_t launch_fused_merge(const ScoreArgs &a, int grid_a, cudaStream_t stream) {
  // the merge kernel starts early and waits on griddepcontrol for the scorer
  const int rows = a.batch * a.dql * 4;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((rows + 3) / 4));
  cfg.blockDim = dim3(128);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  const ReqInfo *info = reinterpret_cast<const ReqInfo *>(a.ws_counters);
  return cudaLaunchKernelEx(&cfg, fused_merge_kernel, a, info, grid_a);
}

}  // namespace icp
