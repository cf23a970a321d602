"""Parity at the full workload sizes, in the launch configuration bench.py
times (one icp_score / icp_publish_rows / icp_merge per shard, and
icp_score_select), on inputs drawn on the GPU by the seeded recipe.

- Score plane: every request of every workload (every shard rank of the
  sharded one, and its unsharded plane) against the oracle's exact plane,
  every written entry, tolerance 1e-5 * sum|q k| + 1e-7; the sentinel
  elsewhere.  The oracle runs request by request over the host cores
  (oracle.parallel.PlanePool).
- Top16 / publish / merge: every row, bit-exact against the oracle's select
  run on the GPU's own plane; merged lists equal the unsharded Top16; the
  fused path equals the chain.
- Exact selection: every row whose cut the exact plane decides (see
  gpu_util.exact_selection_agrees) has the exact plane's ids.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle.parallel import PlanePool
from sparse_attention_block_gb300 import workloads as W

from gpu_util import (assert_plane_matches, assert_select_equal, exact_selection_agrees,
                      gpu_score, gpu_select, icp)

pytestmark = pytest.mark.gpu

# rows whose Top16 cut lies within the scores' tolerance are not decided by
# the plane; on these workloads they are rare
MIN_DECIDED = 0.97


def _host(*ts):
    return [t.cpu().numpy() for t in ts]


def _assert_decided(checked, skipped, what):
    total = checked + skipped
    print(f"{what}: exact selection checked on {checked} of {total} rows")
    assert checked >= MIN_DECIDED * total, f"{what}: only {checked} of {total} rows decided"


@pytest.mark.parametrize("name", ["batched", "multitoken", "longctx"])
def test_unsharded_workload_full_size(name):
    spec = W.DECODE_SPECS[name]
    inp = W.make_decode_inputs(spec, seed=0, device="cuda")
    q, k, bt, sl, nvp = inp.index_q, inp.index_k, inp.block_table, inp.seq_lens, \
        inp.num_valid_pages
    T = inp.T
    dql = spec.decode_query_len
    cols = icp().icp_score_columns(int(sl.max()), spec.page_size, 1)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    plane = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=spec.page_size,
                      dql=dql, maxdql=spec.max_decode_query_len, errors=errors)
    # publish + merge as in the bench step (ws 1: one owner with all four heads)
    recv = torch.zeros((icp().recv_rows(1, 4, T), 33), dtype=torch.int32, device="cuda")
    bases = torch.tensor([recv.data_ptr()], dtype=torch.int64, device="cuda")
    icp().icp_publish_rows(plane, nvp, bases, errors, slot=1, rank=0, world_size=1,
                           heads_per_rank=4, capacity=T, force_begin_blocks=spec.init_blocks,
                           force_end_blocks=spec.local_blocks, spin_limit=1 << 22)
    ms = torch.empty((T, 4, 16), dtype=torch.float32, device="cuda")
    mi = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    icp().icp_merge(recv, nvp, ms, mi, errors, T=T, slot=1, world_size=1, heads_per_rank=4,
                    capacity=T, init_blocks=spec.init_blocks, local_blocks=spec.local_blocks,
                    spin_limit=1 << 22)
    # fused
    work = torch.empty((icp().icp_score_select_workspace_bytes(spec.batch, dql),),
                       dtype=torch.uint8, device="cuda")
    fs = torch.empty((T, 4, 16), dtype=torch.float32, device="cuda")
    fi = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    icp().icp_score_select(q, k, bt, sl, nvp, fs, fi, work, cols=cols, rank=0, world_size=1,
                           page_size=spec.page_size, decode_query_len=dql,
                           max_decode_query_len=spec.max_decode_query_len,
                           init_blocks=spec.init_blocks, local_blocks=spec.local_blocks,
                           errors=errors)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0
    gp, hn = _host(plane, nvp)
    # every row: oracle select on the GPU plane
    os_, oi = oracle.select(gp, hn, init_blocks=spec.init_blocks,
                            local_blocks=spec.local_blocks)
    assert_select_equal(ms, mi, os_, oi, f"{name} merged")
    assert_select_equal(fs, fi, os_, oi, f"{name} fused")
    # every published row carries the oracle's row; the merge freed them all
    ref = [np.zeros(tuple(recv.shape), np.int32)]
    oracle.publish(gp, hn, ref, slot=1, rank=0, world_size=1, heads_per_rank=4, capacity=T,
                   force_begin_blocks=spec.init_blocks, force_end_blocks=spec.local_blocks)
    got = recv.cpu().numpy()
    assert np.array_equal(got[:, :32], ref[0][:, :32]), f"{name}: published rows differ"
    assert not got[:, 32].any(), f"{name}: a ready flag was not cleared by the merge"
    # every request's plane against the exact plane
    hq, hk, hbt, hsl = _host(q, k, bt, sl)
    with PlanePool(hq, [hk], hbt, hsl) as pool:
        ex, ab = pool.decode_plane(k=0, cols=cols, rank=0, world_size=1,
                                   page_size=spec.page_size, decode_query_len=dql)
    assert_plane_matches(gp, ex, ab, f"{name} plane, all {spec.batch} requests")
    checked, skipped = exact_selection_agrees(ex, ab, mi.cpu().numpy(), hn, spec.init_blocks,
                                              spec.local_blocks)
    _assert_decided(checked, skipped, name)


def test_sharded_workload_full_size():
    spec = W.SHARDED
    inp = W.make_decode_inputs(spec, seed=0, device="cuda")
    ws, hpr, T, cap = spec.world_size, 4 // spec.world_size, inp.T, spec.capacity
    q, bt, sl, nvp = inp.index_q, inp.block_table, inp.seq_lens, inp.num_valid_pages
    dql = spec.decode_query_len
    cols = icp().icp_score_columns(int(sl.max()), spec.page_size, ws)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    recv = [torch.zeros((icp().recv_rows(ws, hpr, cap), 33), dtype=torch.int32, device="cuda")
            for _ in range(ws)]
    bases = torch.tensor([r.data_ptr() for r in recv], dtype=torch.int64, device="cuda")
    planes = []
    for rank in range(ws):
        p = gpu_score(q, inp.shards[rank], bt, sl, cols=cols, rank=rank, world_size=ws,
                      page_size=spec.page_size, dql=dql, errors=errors)
        icp().icp_publish_rows(p, nvp, bases, errors, slot=2, rank=rank, world_size=ws,
                               heads_per_rank=hpr, capacity=cap,
                               force_begin_blocks=spec.init_blocks,
                               force_end_blocks=spec.local_blocks, spin_limit=1 << 22)
        planes.append(p)
    torch.cuda.synchronize()
    hn = nvp.cpu().numpy()
    hplanes = [p.cpu().numpy() for p in planes]
    ref = [np.zeros((icp().recv_rows(ws, hpr, cap), 33), np.int32) for _ in range(ws)]
    for rank in range(ws):
        oracle.publish(hplanes[rank], hn, ref, slot=2, rank=rank, world_size=ws,
                       heads_per_rank=hpr, capacity=cap, force_begin_blocks=spec.init_blocks,
                       force_end_blocks=spec.local_blocks)
    for owner in range(ws):
        assert np.array_equal(recv[owner].cpu().numpy(), ref[owner]), f"owner {owner} rows"
    merged_i = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    merged_s = torch.empty((T, 4, 16), dtype=torch.float32, device="cuda")
    for owner in range(ws):
        s = torch.empty((T, hpr, 16), dtype=torch.float32, device="cuda")
        i = torch.empty((T, hpr, 16), dtype=torch.int32, device="cuda")
        icp().icp_merge(recv[owner], nvp, s, i, errors, T=T, slot=2, world_size=ws,
                        heads_per_rank=hpr, capacity=cap, init_blocks=spec.init_blocks,
                        local_blocks=spec.local_blocks, spin_limit=1 << 22)
        merged_s[:, owner * hpr:(owner + 1) * hpr] = s
        merged_i[:, owner * hpr:(owner + 1) * hpr] = i
    # the unsharded plane of the same cache, selected on the GPU
    up = gpu_score(q, inp.index_k, bt, sl, cols=cols, rank=0, world_size=1,
                   page_size=spec.page_size, dql=dql)
    us, ui = gpu_select(up, nvp, init=spec.init_blocks, local=spec.local_blocks)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0
    assert torch.equal(merged_i, ui), "merged ids differ from the unsharded Top16"
    assert torch.equal(merged_s.view(torch.int32), us.view(torch.int32))
    for owner in range(ws):
        s, i, missing = oracle.merge(ref[owner], hn, T=T, slot=2, owner=owner, world_size=ws,
                                     heads_per_rank=hpr, capacity=cap,
                                     init_blocks=spec.init_blocks,
                                     local_blocks=spec.local_blocks)
        assert missing == 0
        assert np.array_equal(i, merged_i[:, owner * hpr:(owner + 1) * hpr].cpu().numpy())
    # every shard plane and the unsharded plane against the exact planes
    hq, hbt, hsl = _host(q, bt, sl)
    ks = [s.cpu().numpy() for s in inp.shards] + [inp.index_k.cpu().numpy()]
    with PlanePool(hq, ks, hbt, hsl) as pool:
        for rank in range(ws):
            ex, ab = pool.decode_plane(k=rank, cols=cols, rank=rank, world_size=ws,
                                       page_size=spec.page_size, decode_query_len=dql)
            assert_plane_matches(hplanes[rank], ex, ab, f"sharded plane of rank {rank}")
        ex, ab = pool.decode_plane(k=ws, cols=cols, rank=0, world_size=1,
                                   page_size=spec.page_size, decode_query_len=dql)
    assert_plane_matches(up, ex, ab, "unsharded plane of the sharded workload")
    checked, skipped = exact_selection_agrees(ex, ab, merged_i.cpu().numpy(), hn,
                                              spec.init_blocks, spec.local_blocks)
    _assert_decided(checked, skipped, "sharded (merged lists)")
