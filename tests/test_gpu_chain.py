"""Publish into legacy receive rows and owner merge (CUDA) against the oracle,
the sharded-merge == unsharded invariant on the GPU, and the bounded waits."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_block_gb300 import workloads as W

from gpu_util import gpu_score, gpu_select, icp, to_dev

pytestmark = pytest.mark.gpu


def _recv(ws, hpr, cap, n_owner):
    rows = 3 * ws * hpr * cap
    bufs = [torch.zeros((rows, 33), dtype=torch.int32, device="cuda") for _ in range(n_owner)]
    bases = torch.tensor([b.data_ptr() for b in bufs], dtype=torch.int64, device="cuda")
    return bufs, bases


def _run_sharded(inp, spec, cols, slot, bufs, bases, errors, init, local):
    """4 shard scorers + 4 publishes on one GPU; returns the shard planes."""
    ws = spec.world_size
    hpr = 4 // ws
    q, _, bt, sl, nvp = to_dev(inp)
    planes = []
    for rank in range(ws):
        shard = inp.shards[rank].cuda()
        p = gpu_score(q, shard, bt, sl, cols=cols, rank=rank, world_size=ws,
                      page_size=spec.page_size, dql=spec.decode_query_len, errors=errors)
        scale, offset = (1, 0) if spec.page_size == 128 else (2, rank * 2 // ws)
        icp().icp_publish_rows(p, nvp, bases, errors, slot=slot, rank=rank, world_size=ws,
                               heads_per_rank=hpr, capacity=spec.capacity or inp.T,
                               force_begin_blocks=init, force_end_blocks=local,
                               spin_limit=1 << 20, index_scale=scale, index_offset=offset)
        planes.append(p)
    return planes


def _merge_all(inp, spec, slot, bufs, errors, init, local):
    ws = spec.world_size
    hpr = 4 // ws
    T = inp.T
    nvp = inp.num_valid_pages.cuda()
    out_s = torch.empty((T, 4, 16), dtype=torch.float32, device="cuda")
    out_i = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    for owner in range(ws):
        s = torch.empty((T, hpr, 16), dtype=torch.float32, device="cuda")
        i = torch.empty((T, hpr, 16), dtype=torch.int32, device="cuda")
        icp().icp_merge(bufs[owner], nvp, s, i, errors, T=T, slot=slot, world_size=ws,
                        heads_per_rank=hpr, capacity=spec.capacity or T, init_blocks=init,
                        local_blocks=local, spin_limit=1 << 20)
        out_s[:, owner * hpr:(owner + 1) * hpr] = s
        out_i[:, owner * hpr:(owner + 1) * hpr] = i
    return out_s, out_i


@pytest.mark.parametrize("page_size,ws", [(128, 4), (128, 2), (256, 2), (256, 4)])
def test_sharded_chain_matches_oracle_and_unsharded(page_size, ws):
    spec = W.DecodeSpec("chain", batch=6, page_size=page_size, world_size=ws, decode_query_len=2,
                        max_decode_query_len=2, init_blocks=1, local_blocks=3,
                        seq_range=(300, 9000), capacity=16)
    inp = W.make_decode_inputs(spec, seed=page_size + ws)
    hpr = 4 // ws
    cols = W.columns_for(spec, int(inp.seq_lens.max()))
    bufs, bases = _recv(ws, hpr, spec.capacity, ws)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    for step in range(4):     # slots rotate; rows are freed by the merge and reused
        slot = step % 3
        planes = _run_sharded(inp, spec, cols, slot, bufs, bases, errors, 1, 3)
        torch.cuda.synchronize()
        # publish rows == oracle publish on the GPU's own planes
        ref = [np.zeros((3 * ws * hpr * spec.capacity, 33), np.int32) for _ in range(ws)]
        for rank in range(ws):
            scale, offset = (1, 0) if page_size == 128 else (2, rank * 2 // ws)
            oracle.publish(planes[rank].cpu().numpy(), inp.num_valid_pages.numpy(), ref,
                           slot=slot, rank=rank, world_size=ws, heads_per_rank=hpr,
                           capacity=spec.capacity, force_begin_blocks=1, force_end_blocks=3,
                           index_scale=scale, index_offset=offset)
        for owner in range(ws):
            got = bufs[owner].cpu().numpy()
            rows = slice(slot * ws * hpr * spec.capacity, (slot + 1) * ws * hpr * spec.capacity)
            assert np.array_equal(got[rows], ref[owner][rows]), f"owner {owner} rows differ"
        ms, mi = _merge_all(inp, spec, slot, bufs, errors, 1, 3)
        torch.cuda.synchronize()
        assert int(errors.item()) == 0
        for b in bufs:
            assert int(b[:, 32].sum().item()) == 0      # all rows free again
        # unsharded GPU plane (one column per B128 block) + select == merged
        q, k, bt, sl, nvp = to_dev(inp)
        full_spec_cols = W.columns_for(
            W.DecodeSpec("u", batch=1, page_size=page_size, world_size=1, decode_query_len=2,
                         max_decode_query_len=2, init_blocks=0, local_blocks=0, seq_lens=(1,)),
            int(inp.seq_lens.max()))
        up = gpu_score(q, k, bt, sl, cols=full_spec_cols, rank=0, world_size=1,
                       page_size=page_size, dql=2)
        us, ui = gpu_select(up, nvp, init=1, local=3)
        torch.cuda.synchronize()
        assert torch.equal(mi, ui), "merged ids differ from the unsharded Top16"
        assert torch.equal(ms.view(torch.int32), us.view(torch.int32))
        # and the oracle's merge of the oracle's rows gives the same lists
        for owner in range(ws):
            s, i, missing = oracle.merge(ref[owner], inp.num_valid_pages.numpy(), T=inp.T,
                                         slot=slot, owner=owner, world_size=ws,
                                         heads_per_rank=hpr, capacity=spec.capacity,
                                         init_blocks=1, local_blocks=3)
            assert missing == 0
            assert np.array_equal(i, mi[:, owner * hpr:(owner + 1) * hpr].cpu().numpy())


def test_publish_times_out_on_an_occupied_row_without_trapping():
    T, K, ws, hpr, cap = 3, 200, 1, 4, 4
    plane = torch.randn((T, 4, K), device="cuda")
    nvp = torch.full((T,), K, dtype=torch.int32, device="cuda")
    bufs, bases = _recv(ws, hpr, cap, 1)
    occupied = oracle.recv_row(1, 0, ws, hpr, 2, cap, 1)
    bufs[0][occupied] = 77
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    icp().icp_publish_rows(plane, nvp, bases, errors, slot=1, rank=0, world_size=ws,
                           heads_per_rank=hpr, capacity=cap, force_begin_blocks=1,
                           force_end_blocks=1, spin_limit=1000)
    torch.cuda.synchronize()
    assert int(errors.item()) == 1
    got = bufs[0].cpu().numpy()
    assert np.all(got[occupied] == 77)                    # left alone
    flags = got[:, 32].copy()
    flags[occupied] = 0
    assert int(flags.sum()) == T * 4 - 1                   # every other row published


def test_merge_reports_a_source_that_never_published():
    T, ws, hpr, cap = 2, 2, 2, 2
    bufs, bases = _recv(ws, hpr, cap, ws)
    nvp = torch.full((T,), 50, dtype=torch.int32, device="cuda")
    plane = torch.randn((T, 4, 50), device="cuda")
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    icp().icp_publish_rows(plane, nvp, bases, errors, slot=0, rank=0, world_size=ws,
                           heads_per_rank=hpr, capacity=cap, force_begin_blocks=0,
                           force_end_blocks=0, spin_limit=1000)
    s = torch.empty((T, hpr, 16), dtype=torch.float32, device="cuda")
    i = torch.empty((T, hpr, 16), dtype=torch.int32, device="cuda")
    icp().icp_merge(bufs[0], nvp, s, i, errors, T=T, slot=0, world_size=ws, heads_per_rank=hpr,
                    capacity=cap, init_blocks=0, local_blocks=0, spin_limit=1000)
    torch.cuda.synchronize()
    assert int(errors.item()) == T * hpr                   # rank 1's rows never arrived
    ref_s, ref_i = oracle.select(plane.cpu().numpy(), nvp.cpu().numpy(), init_blocks=0,
                                 local_blocks=0)
    assert np.array_equal(i.cpu().numpy(), ref_i[:, :hpr])


def test_chain_under_programmatic_dependent_launch():
    # scorer and publish both launched with enable_pdl: the publish waits on
    # the scorer before reading the plane, so the rows equal the oracle's
    spec = W.DecodeSpec("pdl", batch=9, page_size=128, world_size=2, decode_query_len=2,
                        max_decode_query_len=2, init_blocks=1, local_blocks=3,
                        seq_range=(300, 20000), capacity=18)
    inp = W.make_decode_inputs(spec, seed=77)
    ws, hpr = 2, 2
    cols = W.columns_for(spec, int(inp.seq_lens.max()))
    bufs, bases = _recv(ws, hpr, spec.capacity, ws)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, _, bt, sl, nvp = to_dev(inp)
    for step in range(3):
        slot = step % 3
        planes = []
        for rank in range(ws):
            shard = inp.shards[rank].cuda()
            p = torch.empty((inp.T, 4, cols), device="cuda")
            icp().icp_score(q, shard, bt, sl, p, rank=rank, world_size=ws, page_size=128,
                            decode_query_len=2, max_decode_query_len=2, enable_pdl=True,
                            errors=errors)
            icp().icp_publish_rows(p, nvp, bases, errors, slot=slot, rank=rank, world_size=ws,
                                   heads_per_rank=hpr, capacity=spec.capacity,
                                   force_begin_blocks=1, force_end_blocks=3,
                                   spin_limit=1 << 20, enable_pdl=True)
            planes.append(p)
        torch.cuda.synchronize()
        ref = [np.zeros((3 * ws * hpr * spec.capacity, 33), np.int32) for _ in range(ws)]
        for rank in range(ws):
            oracle.publish(planes[rank].cpu().numpy(), inp.num_valid_pages.numpy(), ref,
                           slot=slot, rank=rank, world_size=ws, heads_per_rank=hpr,
                           capacity=spec.capacity, force_begin_blocks=1, force_end_blocks=3)
        rows = slice(slot * ws * hpr * spec.capacity, (slot + 1) * ws * hpr * spec.capacity)
        for owner in range(ws):
            assert np.array_equal(bufs[owner].cpu().numpy()[rows], ref[owner][rows])
        _merge_all(inp, spec, slot, bufs, errors, 1, 3)
        torch.cuda.synchronize()
        assert int(errors.item()) == 0


def test_whole_chain_under_programmatic_dependent_launch():
    # scorer, publish and owner merge all launched with enable_pdl, back to
    # back with no synchronisation in between: every kernel waits on its
    # predecessor before reading, so the merged lists equal the oracle's
    # merge of the oracle's rows of the same planes
    spec = W.DecodeSpec("pdl3", batch=7, page_size=128, world_size=2, decode_query_len=2,
                        max_decode_query_len=2, init_blocks=1, local_blocks=3,
                        seq_range=(300, 20000), capacity=14)
    inp = W.make_decode_inputs(spec, seed=78)
    ws, hpr, T = 2, 2, inp.T
    cols = W.columns_for(spec, int(inp.seq_lens.max()))
    bufs, bases = _recv(ws, hpr, spec.capacity, ws)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    q, _, bt, sl, nvp = to_dev(inp)
    shards = [s.cuda() for s in inp.shards]
    for step in range(3):
        slot = step % 3
        planes, outs = [], []
        for rank in range(ws):
            p = torch.empty((T, 4, cols), device="cuda")
            icp().icp_score(q, shards[rank], bt, sl, p, rank=rank, world_size=ws, page_size=128,
                            decode_query_len=2, max_decode_query_len=2, enable_pdl=True,
                            errors=errors)
            icp().icp_publish_rows(p, nvp, bases, errors, slot=slot, rank=rank, world_size=ws,
                                   heads_per_rank=hpr, capacity=spec.capacity,
                                   force_begin_blocks=1, force_end_blocks=3,
                                   spin_limit=1 << 20, enable_pdl=True)
            planes.append(p)
        for owner in range(ws):
            s = torch.empty((T, hpr, 16), dtype=torch.float32, device="cuda")
            i = torch.empty((T, hpr, 16), dtype=torch.int32, device="cuda")
            icp().icp_merge(bufs[owner], nvp, s, i, errors, T=T, slot=slot, world_size=ws,
                            heads_per_rank=hpr, capacity=spec.capacity, init_blocks=1,
                            local_blocks=3, spin_limit=1 << 20, enable_pdl=True)
            outs.append((s, i))
        torch.cuda.synchronize()
        assert int(errors.item()) == 0
        ref = [np.zeros((3 * ws * hpr * spec.capacity, 33), np.int32) for _ in range(ws)]
        for rank in range(ws):
            oracle.publish(planes[rank].cpu().numpy(), inp.num_valid_pages.numpy(), ref,
                           slot=slot, rank=rank, world_size=ws, heads_per_rank=hpr,
                           capacity=spec.capacity, force_begin_blocks=1, force_end_blocks=3)
        for owner in range(ws):
            ms, mi, missing = oracle.merge(ref[owner], inp.num_valid_pages.numpy(), T=T,
                                           slot=slot, owner=owner, world_size=ws,
                                           heads_per_rank=hpr, capacity=spec.capacity,
                                           init_blocks=1, local_blocks=3)
            assert missing == 0
            s, i = outs[owner]
            np.testing.assert_array_equal(i.cpu().numpy(), mi)
            np.testing.assert_array_equal(s.cpu().numpy().view(np.int32), ms.view(np.int32))
