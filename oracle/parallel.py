"""Times the oracle's decode chain over several host cores (test infrastructure).

The CPU baseline runs the oracle as it is, request by request:
- the score plane of the request (``score``), one per shard;
- its Top16 published into legacy receive rows (``publish``);
- the owner merge (``merge``).

This module computes nothing of its own. ``decode_request`` is that chain
for one request. ``ParallelChain`` runs it over the requests of a batch in
worker processes started with ``spawn``. The batch's arrays (the index-K
shards above all) sit in shared memory, so no worker copies them.
"""
from __future__ import annotations

import multiprocessing as mp
import os
import time
from multiprocessing import shared_memory

import numpy as np

from . import merge, publish, score


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
