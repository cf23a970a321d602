"""Parity at the full workload sizes, in the launch configuration bench.py
times (one icp_score / icp_publish_rows / icp_merge per shard, and
icp_score_select), on inputs drawn on the GPU by the seeded recipe.

- Score plane: sampled requests (first, longest, one more) against the
  oracle's exact plane, every written entry, tolerance 1e-5 * sum|q k| + 1e-7.
- Top16 / publish / merge: every row, bit-exact against the oracle's select
  run on the GPU's own plane; merged lists equal the unsharded Top16; the
  fused path equals the chain.
- Exact selection: on the sampled rows, wherever the gap at the Top16 cut is
  above twice the tolerance, the ids equal the exact plane's selection.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_block_gb300 import workloads as W

from gpu_util import (assert_plane_matches, assert_select_equal, exact_selection_agrees,
                      gpu_score, gpu_select, icp)

pytestmark = pytest.mark.gpu


def _sub_request(inp, b, shard=None):
    """The request's own pages as a small pool, for the oracle."""
    spec = inp.spec
    L = int(inp.seq_lens[b])
    npages = (L + spec.page_size - 1) // spec.page_size
    pages = inp.block_table[b, :npages].long().cpu()
    src = inp.index_k if shard is None else shard
    k = src[pages.to(src.device)].cpu().numpy()
    bt = np.arange(npages, dtype=np.int32)[None, :]
    dql = spec.decode_query_len
    q = inp.index_q[b * dql:(b + 1) * dql].cpu().numpy()
    return q, k, bt, np.array([L], np.int32)


def _sample(inp):
    sl = inp.seq_lens.cpu()
    picks = {0, int(torch.argmax(sl)), len(sl) // 2}
    return sorted(picks)


def _check_plane_samples(inp, plane, cols, rank=0, shard=None, world_size=None):
    spec = inp.spec
    dql = spec.decode_query_len
    ws = spec.world_size if world_size is None else world_size
    gp = plane.cpu().numpy()
    for b in _sample(inp):
        q, k, bt, sl = _sub_request(inp, b, shard)
        ex, ab = oracle.score(q, k, bt, sl, cols=cols, rank=rank, world_size=ws,
                              page_size=spec.page_size, decode_query_len=dql, fill=np.nan)
        rows = gp[b * dql:(b + 1) * dql]
        assert_plane_matches(rows, ex, ab, f"{spec.name} request {b} rank {rank}")
        if shard is None:
            nvp = inp.num_valid_pages[b * dql:(b + 1) * dql].cpu().numpy()
            gs, gi = oracle.select(rows, nvp, init_blocks=spec.init_blocks,
                                   local_blocks=spec.local_blocks)
            n = exact_selection_agrees(ex, ab, gi, nvp, spec.init_blocks, spec.local_blocks)
            assert n > 0


@pytest.mark.parametrize("name", ["batched", "multitoken", "longctx"])
def test_unsharded_workload_full_size(name):
    spec = W.DECODE_SPECS[name]
    inp = W.make_decode_inputs(spec, seed=0, device="cuda")
    q, k, bt, sl, nvp = inp.index_q, inp.index_k, inp.block_table, inp.seq_lens, \
        inp.num_valid_pages
    T = inp.T
    cols = icp().icp_score_columns(int(sl.max()), spec.page_size, 1)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    plane = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=spec.page_size,
                      dql=spec.decode_query_len, maxdql=spec.max_decode_query_len,
                      errors=errors)
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
    work = torch.empty((icp().icp_score_select_workspace_bytes(spec.batch,
                                                               spec.decode_query_len),),
                       dtype=torch.uint8, device="cuda")
    fs = torch.empty((T, 4, 16), dtype=torch.float32, device="cuda")
    fi = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    icp().icp_score_select(q, k, bt, sl, nvp, fs, fi, work, cols=cols, rank=0, world_size=1,
                           page_size=spec.page_size, decode_query_len=spec.decode_query_len,
                           max_decode_query_len=spec.max_decode_query_len,
                           init_blocks=spec.init_blocks, local_blocks=spec.local_blocks,
                           errors=errors)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0
    # every row: oracle select on the GPU plane
    os_, oi = oracle.select(plane.cpu().numpy(), nvp.cpu().numpy(),
                            init_blocks=spec.init_blocks, local_blocks=spec.local_blocks)
    assert_select_equal(ms, mi, os_, oi, f"{name} merged")
    assert_select_equal(fs, fi, os_, oi, f"{name} fused")
    # publish rows carry the same lists
    got = recv.cpu().numpy()
    for t in range(0, T, max(1, T // 64)):
        for h in range(4):
            row = got[oracle.recv_row(1, 0, 1, 4, h, T, t)]
            assert row[32] == 0                            # freed by the merge
            assert np.array_equal(row[16:32], oi[t, h])
    # sampled requests against the exact plane
    _check_plane_samples(inp, plane, cols)


def test_sharded_workload_full_size():
    spec = W.SHARDED
    inp = W.make_decode_inputs(spec, seed=0, device="cuda")
    ws, hpr, T, cap = spec.world_size, 4 // spec.world_size, inp.T, spec.capacity
    q, bt, sl, nvp = inp.index_q, inp.block_table, inp.seq_lens, inp.num_valid_pages
    cols = icp().icp_score_columns(int(sl.max()), spec.page_size, ws)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    recv = [torch.zeros((icp().recv_rows(ws, hpr, cap), 33), dtype=torch.int32, device="cuda")
            for _ in range(ws)]
    bases = torch.tensor([r.data_ptr() for r in recv], dtype=torch.int64, device="cuda")
    planes = []
    for rank in range(ws):
        p = gpu_score(q, inp.shards[rank], bt, sl, cols=cols, rank=rank, world_size=ws,
                      page_size=spec.page_size, dql=spec.decode_query_len, errors=errors)
        icp().icp_publish_rows(p, nvp, bases, errors, slot=2, rank=rank, world_size=ws,
                               heads_per_rank=hpr, capacity=cap,
                               force_begin_blocks=spec.init_blocks,
                               force_end_blocks=spec.local_blocks, spin_limit=1 << 22)
        planes.append(p)
    torch.cuda.synchronize()
    ref = [np.zeros((icp().recv_rows(ws, hpr, cap), 33), np.int32) for _ in range(ws)]
    for rank in range(ws):
        oracle.publish(planes[rank].cpu().numpy(), nvp.cpu().numpy(), ref, slot=2, rank=rank,
                       world_size=ws, heads_per_rank=hpr, capacity=cap,
                       force_begin_blocks=spec.init_blocks, force_end_blocks=spec.local_blocks)
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
                   page_size=spec.page_size, dql=spec.decode_query_len)
    us, ui = gpu_select(up, nvp, init=spec.init_blocks, local=spec.local_blocks)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0
    assert torch.equal(merged_i, ui), "merged ids differ from the unsharded Top16"
    assert torch.equal(merged_s.view(torch.int32), us.view(torch.int32))
    for owner in range(ws):
        s, i, missing = oracle.merge(ref[owner], nvp.cpu().numpy(), T=T, slot=2, owner=owner,
                                     world_size=ws, heads_per_rank=hpr, capacity=cap,
                                     init_blocks=spec.init_blocks,
                                     local_blocks=spec.local_blocks)
        assert missing == 0
        assert np.array_equal(i, merged_i[:, owner * hpr:(owner + 1) * hpr].cpu().numpy())
    # shard planes and the unsharded plane against the oracle on sampled requests
    _check_plane_samples(inp, planes[1], cols, rank=1, shard=inp.shards[1])
    _check_plane_samples(inp, up, cols, world_size=1)
