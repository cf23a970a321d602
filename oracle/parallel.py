"""Runs the oracle over several host cores (test infrastructure).

The CPU baseline runs the oracle as it is, request by request:
- the score plane of the request (``score``), one per shard;
- its Top16 published into legacy receive rows (``publish``);
- the owner merge (``merge``).

This module computes nothing of its own. ``decode_request`` is that chain
for one request. ``ParallelChain`` runs it over the requests of a batch in
worker processes started with ``spawn``. ``PlanePool`` gives the tests the
oracle's exact score plane of a whole full-size batch the same way, one
request (or one slice of a prefill chunk) per task.  The batch's arrays (the
index-K shards above all) sit in shared memory, so no worker copies them.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import time
from multiprocessing import shared_memory

import numpy as np

from . import merge, publish, score, score_chunks


def decode_request(q, shards, bt, sl, nvp, b, *, cols, world_size, page_size, decode_query_len,
                   init_blocks, local_blocks):
    """The oracle's chain (score, select + publish, merge) for request b."""
    ws, dql = world_size, decode_query_len
    hpr = 4 // ws
    qb = q[b * dql:(b + 1) * dql]
    nv = nvp[b * dql:(b + 1) * dql]
    cap = dql
    recv = [np.zeros((3 * ws * hpr * cap, 33), np.int32) for _ in range(ws)]
    for rank in range(ws):
        plane, _ = score(qb, shards[rank], bt[b:b + 1], sl[b:b + 1], cols=cols, rank=rank,
                         world_size=ws, page_size=page_size, decode_query_len=dql,
                         fill=-np.inf)
        scale, offset = (1, 0) if (page_size == 128 or ws == 1) else (2, rank * 2 // ws)
        publish(plane.astype(np.float32), nv, recv, slot=0, rank=rank, world_size=ws,
                heads_per_rank=hpr, capacity=cap, force_begin_blocks=init_blocks,
                force_end_blocks=local_blocks, index_scale=scale, index_offset=offset)
    outs = []
    for owner in range(ws):
        outs.append(merge(recv[owner], nv, T=dql, slot=0, owner=owner, world_size=ws,
                          heads_per_rank=hpr, capacity=cap, init_blocks=init_blocks,
                          local_blocks=local_blocks))
    return outs


# ------------------------------------------------------------------ workers
_W = {}


def _attach(desc):
    """Worker start: numpy views of the shared arrays described by desc."""
    shms, arrays = [], {}
    for name, (shm_name, shape, dtype) in desc["arrays"].items():
        shm = shared_memory.SharedMemory(name=shm_name)
        shms.append(shm)
        arrays[name] = np.ndarray(shape, dtype=np.dtype(dtype), buffer=shm.buf)
    _W["shms"] = shms
    _W["arrays"] = arrays
    _W["params"] = desc["params"]
    _W["nshards"] = desc["nshards"]


def _run(reqs):
    a, p = _W["arrays"], _W["params"]
    shards = [a[f"shard{r}"] for r in range(_W["nshards"])]
    t0 = time.perf_counter()
    for b in reqs:
        decode_request(a["q"], shards, a["bt"], a["sl"], a["nvp"], b, **p)
    return time.perf_counter() - t0


class ParallelChain:
    """Worker processes that run decode_request over a batch held in shared
    memory.  Use as a context manager; workers = os.cpu_count() by default."""

    def __init__(self, q, shards, bt, sl, nvp, params, workers=None):
        self.workers = workers or os.cpu_count() or 1
        self._shms = []
        desc = {"arrays": {}, "params": dict(params), "nshards": len(shards)}
        named = {"q": q, "bt": bt, "sl": sl, "nvp": nvp}
        named.update({f"shard{r}": s for r, s in enumerate(shards)})
        for name, arr in named.items():
            arr = np.ascontiguousarray(arr)
            shm = shared_memory.SharedMemory(create=True, size=max(arr.nbytes, 1))
            np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)[...] = arr
            self._shms.append(shm)
            desc["arrays"][name] = (shm.name, arr.shape, arr.dtype.str)
        ctx = mp.get_context("spawn")
        self._pool = ctx.Pool(self.workers, initializer=_attach, initargs=(desc,))
        # every worker loads the oracle library before anything is timed
        self._pool.map(_run, [[] for _ in range(self.workers)], chunksize=1)

    def time(self, requests):
        """Wall seconds for the chain over `requests`, split evenly over the
        workers (every request once)."""
        reqs = list(requests)
        parts = [reqs[i::self.workers] for i in range(self.workers)]
        t0 = time.perf_counter()
        self._pool.map(_run, parts, chunksize=1)
        return time.perf_counter() - t0

    def close(self):
        self._pool.close()
        self._pool.join()
        for shm in self._shms:
            shm.close()
            shm.unlink()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


# ---------------------------------------------------------------- planes
def _plane_task(task):
    """One request's rows of the exact plane (oracle.score on its own
    block-table row), or one slice of a prefill chunk (oracle.score_chunks
    on the tokens j0 .. j1 - 1 of request b's chunk of n tokens, which sit at
    positions seq_len - n + j0 .. seq_len - n + j1 - 1: a window of its own
    whose request length ends at the last of them)."""
    a = _W["arrays"]
    k = a[f"shard{task['k']}"]
    b = task["b"]
    if task["kind"] == "decode":
        dql = task["dql"]
        plane, absplane = score(a["q"][b * dql:(b + 1) * dql], k, a["bt"][b:b + 1],
                                a["sl"][b:b + 1], cols=task["cols"], rank=task["rank"],
                                world_size=task["world_size"], page_size=task["page_size"],
                                decode_query_len=dql, fill=np.nan)
        return task, plane, absplane
    j0, j1, n, q0 = task["j0"], task["j1"], task["n"], task["q0"]
    L = int(a["sl"][b])
    plane, absplane = score_chunks(a["q"][q0 + j0:q0 + j1], k, a["bt"][b:b + 1],
                                   np.array([L - n + j1], np.int32),
                                   np.array([0, j1 - j0], np.int32), cols=task["cols"], rank=0,
                                   world_size=1, page_size=task["page_size"], fill=np.nan)
    return task, plane, absplane


class PlanePool:
    """The oracle's exact score planes of a batch, computed by spawned worker
    processes over the batch held in shared memory.

    q: uint8 [T, 4, 128]; ks: list of index-K arrays (the shards of a sharded
    cache, or the whole cache); bt: int32 [B, W]; sl: int32 [B].
    """

    def __init__(self, q, ks, bt, sl, workers=None):
        self.workers = workers or os.cpu_count() or 1
        self._shms = []
        desc = {"arrays": {}, "params": {}, "nshards": len(ks)}
        named = {"q": q, "bt": bt, "sl": sl, "nvp": np.zeros(1, np.int32)}
        named.update({f"shard{r}": kk for r, kk in enumerate(ks)})
        for name, arr in named.items():
            arr = np.ascontiguousarray(arr)
            shm = shared_memory.SharedMemory(create=True, size=max(arr.nbytes, 1))
            np.ndarray(arr.shape, dtype=arr.dtype, buffer=shm.buf)[...] = arr
            self._shms.append(shm)
            desc["arrays"][name] = (shm.name, arr.shape, arr.dtype.str)
        self.sl = np.asarray(sl)
        self.T_rows = np.asarray(q).shape[0]
        ctx = mp.get_context("spawn")
        self._pool = ctx.Pool(self.workers, initializer=_attach, initargs=(desc,))

    def decode_plane(self, *, k, cols, rank, world_size, page_size, decode_query_len,
                     requests=None):
        """Exact plane float64 [B * dql, 4, cols] (NaN where not written) and
        its |q.k| scale plane, as oracle.score over the whole batch would
        give them, computed request by request (a request's rows depend only
        on its own block-table row and seq_len)."""
        dql = decode_query_len
        B = len(self.sl)
        reqs = range(B) if requests is None else requests
        # longest requests first, so that the pool ends together
        order = sorted(reqs, key=lambda b: -int(self.sl[b]))
        tasks = [dict(kind="decode", k=k, b=b, cols=cols, rank=rank, world_size=world_size,
                      page_size=page_size, dql=dql) for b in order]
        plane = np.full((B * dql, 4, cols), np.nan)
        absplane = np.full((B * dql, 4, cols), np.nan)
        for task, p, ab in self._pool.imap_unordered(_plane_task, tasks, chunksize=1):
            b = task["b"]
            plane[b * dql:(b + 1) * dql] = p
            absplane[b * dql:(b + 1) * dql] = ab
        return plane, absplane

    def window_slices(self, qo_indptr, *, cols, page_size, piece=128, k=0):
        """Exact rows of a prefill window (oracle.score_chunks), in slices of
        at most `piece` tokens of each request's chunk.  Yields
        (b, j0, j1, plane [j1 - j0, 4, cols], absplane): the slice's tokens
        are window rows qo[b] + j0 .. qo[b] + j1 - 1, and the slice is scored
        as a window whose request length ends at its last token, so only the
        columns that length reaches are written (NaN elsewhere)."""
        qo = np.asarray(qo_indptr)
        tasks = []
        for b in range(len(self.sl)):
            n = int(qo[b + 1] - qo[b])
            for j0 in range(0, n, piece):
                tasks.append(dict(kind="window", k=k, b=b, j0=j0, j1=min(n, j0 + piece), n=n,
                                  q0=int(qo[b]), cols=cols, page_size=page_size))
        tasks.sort(key=lambda t: -(int(self.sl[t["b"]]) - t["n"] + t["j1"]))
        for task, p, ab in self._pool.imap_unordered(_plane_task, tasks, chunksize=1):
            yield task["b"], task["j0"], task["j1"], p, ab

    def close(self):
        self._pool.close()
        self._pool.join()
        for shm in self._shms:
            shm.close()
            shm.unlink()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
