"""Helpers for the GPU parity tests: run the CUDA path through the C ABI
binding, run the oracle on the same seeded inputs, compare."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from sparse_attention_block_gb300 import workloads as W

SENTINEL_BITS = 0x7FC0DEAD  # a NaN payload no kernel writes


def icp():
    from sparse_attention_block_gb300 import icp as _icp
    return _icp


def sentinel_plane(T, cols, device="cuda"):
    return torch.full((T, 4, cols), SENTINEL_BITS, dtype=torch.int32, device=device).view(
        torch.float32)


def gpu_score(q, k, bt, sl, *, cols, rank, world_size, page_size, dql, maxdql=None,
              errors=None):
    """Runs icp_score on device tensors; returns the plane (device, float32)."""
    T = sl.shape[0] * dql
    out = sentinel_plane(T, cols, q.device)
    icp().icp_score(q, k, bt, sl, out, rank=rank, world_size=world_size, page_size=page_size,
                    decode_query_len=dql, max_decode_query_len=maxdql or dql, errors=errors)
    return out


def oracle_plane(q, k, bt, sl, *, cols, rank, world_size, page_size, dql):
    """Exact plane (float64, NaN where not written) and |q.k| scale plane."""
    c = lambda t: t.cpu().numpy() if isinstance(t, torch.Tensor) else np.asarray(t)
    return oracle.score(c(q), c(k), c(bt), c(sl), cols=cols, rank=rank, world_size=world_size,
                        page_size=page_size, decode_query_len=dql, fill=np.nan)


def assert_plane_matches(gpu_plane, exact, absplane, what=""):
    """Tolerance |gpu - exact| <= 1e-5 * sum|q_i k_i| + 1e-7 on written entries
    (-inf exact), and the sentinel bit pattern untouched elsewhere."""
    g = gpu_plane.cpu().numpy() if isinstance(gpu_plane, torch.Tensor) else gpu_plane
    written = ~np.isnan(exact)
    gbits = g.view(np.int32)
    untouched = gbits[~written]
    assert np.all(untouched == SENTINEL_BITS), f"{what}: a column outside the contract was written"
    gw = g[written].astype(np.float64)
    ew = exact[written]
    aw = absplane[written]
    e_inf = np.isneginf(ew)
    g_inf = np.isneginf(gw)
    bad_inf = np.nonzero(e_inf != g_inf)[0]
    assert bad_inf.size == 0, f"{what}: -inf mismatch at {bad_inf[:10]} (gpu {gw[bad_inf[:5]]}, " \
                              f"exact {ew[bad_inf[:5]]})"
    fin = ~e_inf
    assert np.all(np.isfinite(gw[fin])), f"{what}: non-finite GPU score"
    err = np.abs(gw[fin] - ew[fin])
    tol = 1e-5 * aw[fin] + 1e-7
    ratio = err / tol
    worst = int(np.argmax(ratio)) if ratio.size else 0
    assert ratio.size == 0 or ratio.max() <= 1.0, (
        f"{what}: score error {err[worst]:.3e} exceeds tolerance {tol[worst]:.3e} "
        f"(gpu {gw[fin][worst]!r}, exact {ew[fin][worst]!r}); max err/tol {ratio.max():.3f}")
    return float(ratio.max()) if ratio.size else 0.0


def to_dev(inp: W.DecodeInputs, device="cuda"):
    return (inp.index_q.to(device), inp.index_k.to(device), inp.block_table.to(device),
            inp.seq_lens.to(device), inp.num_valid_pages.to(device))


def gpu_select(plane, nvp, *, init, local, scale=1, offset=0):
    T = plane.shape[0]
    s = torch.empty((T, 4, 16), dtype=torch.float32, device=plane.device)
    i = torch.empty((T, 4, 16), dtype=torch.int32, device=plane.device)
    icp().icp_top16_select(plane, nvp, s, i, init_blocks=init, local_blocks=local,
                           index_scale=scale, index_offset=offset)
    return s, i


def assert_select_equal(gs, gi, os_, oi, what=""):
    gs = gs.cpu().numpy() if isinstance(gs, torch.Tensor) else gs
    gi = gi.cpu().numpy() if isinstance(gi, torch.Tensor) else gi
    bad = np.nonzero(np.any(gi != oi, axis=-1).reshape(-1))[0]
    assert bad.size == 0, f"{what}: ids differ in {bad.size} rows, first {bad[:5]}: " \
                          f"gpu {gi.reshape(-1, 16)[bad[0]]} oracle {oi.reshape(-1, 16)[bad[0]]}"
    assert np.array_equal(gs.view(np.int32), os_.view(np.int32)), f"{what}: scores differ"


def exact_selection_agrees(exact_plane, absplane, gpu_ids, nvp, init, local, scale=1, offset=0):
    """The GPU's Top16 ids against the selection of the exact plane.

    Each GPU score lies within tol = 1e-5 * sum|q_i k_i| + 1e-7 of its exact
    value (-inf exactly).  Where every free block the exact plane selects
    stays above every free block it rejects by the two blocks' tolerances
    (min over selected of exact - tol > max over rejected of exact + tol), no
    admissible rounding can change the selected set, so the ids must be
    equal; rows whose cut is within those tolerances are not decided by the
    plane and are skipped.  Rows with at most 16 valid ids, or no free slot
    left to fill, have a unique answer and are always checked.  Returns
    (rows checked, rows skipped)."""
    e32 = np.where(np.isnan(exact_plane), -np.inf, exact_plane).astype(np.float32)
    _, ei = oracle.select(e32, nvp, init_blocks=init, local_blocks=local, index_scale=scale,
                          index_offset=offset)
    T, H, K = exact_plane.shape
    ids_all = np.arange(K, dtype=np.int64) * scale + offset
    checked = skipped = 0
    for t in range(T):
        n = int(nvp[t])
        valid = ids_all < n
        forced = valid & ((ids_all < init) | (ids_all >= n - local))
        free_cols = np.nonzero(valid & ~forced)[0]
        m = 16 - int(forced.sum())
        if n <= 16 or int(valid.sum()) <= 16 or m <= 0 or free_cols.size <= m:
            for h in range(H):
                assert np.array_equal(gpu_ids[t, h], ei[t, h]), (t, h, gpu_ids[t, h], ei[t, h])
            checked += H
            continue
        fid = ids_all[free_cols]
        for h in range(H):
            e = exact_plane[t, h, free_cols]
            assert not np.isnan(e).any(), "a valid column of the exact plane is not written"
            tol = 1e-5 * np.nan_to_num(absplane[t, h, free_cols], nan=0.0) + 1e-7
            order = np.lexsort((fid, -e))
            sel, rej = order[:m], order[m:]
            lo = e[sel] - tol[sel]
            hi = e[rej] + tol[rej]
            if np.isneginf(e[sel[-1]]) or lo.min() > hi.max():
                assert np.array_equal(gpu_ids[t, h], ei[t, h]), (t, h, gpu_ids[t, h], ei[t, h])
                checked += 1
            else:
                skipped += 1
    return checked, skipped
