"""Tagged receive rows (msa_icp_topk_select_publish, tagged mode) on the GPU:
rows and generation counters bit-exact against the oracle's tagged publish on
the GPU planes, the tagged merge equal to the unsharded Top16 over several
steps with slot rotation, and a bounded wait for rows that never arrive."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_block_gb300 import workloads as W

from gpu_util import gpu_score, gpu_select, icp, to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("page_size,ws", [(128, 4), (256, 2), (128, 1)])
def test_tagged_chain_over_steps(page_size, ws):
    spec = W.DecodeSpec("tag", batch=5, page_size=page_size, world_size=ws, decode_query_len=2,
                        max_decode_query_len=2, init_blocks=2, local_blocks=2,
                        seq_range=(300, 7000), capacity=12)
    inp = W.make_decode_inputs(spec, seed=40 + ws)
    hpr, T, cap = 4 // ws, inp.T, spec.capacity
    q, k, bt, sl, nvp = to_dev(inp)
    cols = W.columns_for(spec, int(inp.seq_lens.max()))
    rows = icp().recv_rows(ws, hpr, cap)
    recv = [torch.zeros((rows, 32), dtype=torch.int64, device="cuda") for _ in range(ws)]
    bases = torch.tensor([r.data_ptr() for r in recv], dtype=torch.int64, device="cuda")
    gens = [torch.zeros((3, 4, cap), dtype=torch.int32, device="cuda") for _ in range(ws)]
    expect = [torch.zeros((3, ws, hpr, cap), dtype=torch.int32, device="cuda") for _ in range(ws)]
    ref_recv = [np.zeros((rows, 32), np.int64) for _ in range(ws)]
    ref_gens = [np.zeros((3, 4, cap), np.int32) for _ in range(ws)]
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    rp = page_size // ws
    shards = [inp.index_k[:, r * rp:(r + 1) * rp].contiguous().cuda() for r in range(ws)]
    unsharded_cols = W.columns_for(
        W.DecodeSpec("u", batch=1, page_size=page_size, world_size=1, decode_query_len=2,
                     max_decode_query_len=2, init_blocks=0, local_blocks=0, seq_lens=(1,)),
        int(inp.seq_lens.max()))
    up = gpu_score(q, k, bt, sl, cols=unsharded_cols, rank=0, world_size=1,
                   page_size=page_size, dql=2)
    us, ui = gpu_select(up, nvp, init=2, local=2)
    for step in range(5):
        slot = step % 3
        for rank in range(ws):
            p = gpu_score(q, shards[rank], bt, sl, cols=cols, rank=rank, world_size=ws,
                          page_size=page_size, dql=2)
            scale, off = (2, rank * 2 // ws) if (page_size == 256 and ws > 1) else (1, 0)
            icp().icp_publish_rows_tagged(p, nvp, bases, gens[rank], slot=slot, rank=rank,
                                          world_size=ws, heads_per_rank=hpr, capacity=cap,
                                          force_begin_blocks=2, force_end_blocks=2,
                                          index_scale=scale, index_offset=off)
            torch.cuda.synchronize()
            oracle.publish_tagged(p.cpu().numpy(), inp.num_valid_pages.numpy(), ref_recv,
                                  ref_gens[rank], slot=slot, rank=rank, world_size=ws,
                                  heads_per_rank=hpr, capacity=cap, force_begin_blocks=2,
                                  force_end_blocks=2, index_scale=scale, index_offset=off)
            assert np.array_equal(gens[rank].cpu().numpy(), ref_gens[rank])
        for owner in range(ws):
            assert np.array_equal(recv[owner].cpu().numpy(), ref_recv[owner]), f"owner {owner}"
        ms = torch.empty((T, 4, 16), dtype=torch.float32, device="cuda")
        mi = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
        for owner in range(ws):
            s = torch.empty((T, hpr, 16), dtype=torch.float32, device="cuda")
            i = torch.empty((T, hpr, 16), dtype=torch.int32, device="cuda")
            icp().icp_merge_tagged(recv[owner], expect[owner], nvp, s, i, errors, T=T, slot=slot,
                                   world_size=ws, heads_per_rank=hpr, capacity=cap,
                                   init_blocks=2, local_blocks=2, spin_limit=1 << 20)
            ms[:, owner * hpr:(owner + 1) * hpr] = s
            mi[:, owner * hpr:(owner + 1) * hpr] = i
        torch.cuda.synchronize()
        assert int(errors.item()) == 0
        assert torch.equal(mi, ui), f"step {step}: tagged merge differs from unsharded Top16"
        assert torch.equal(ms.view(torch.int32), us.view(torch.int32))


def test_tagged_merge_reports_rows_that_never_arrive():
    T, ws, hpr, cap = 3, 2, 2, 4
    recv = torch.zeros((icp().recv_rows(ws, hpr, cap), 32), dtype=torch.int64, device="cuda")
    expect = torch.zeros((3, ws, hpr, cap), dtype=torch.int32, device="cuda")
    nvp = torch.full((T,), 40, dtype=torch.int32, device="cuda")
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    s = torch.empty((T, hpr, 16), dtype=torch.float32, device="cuda")
    i = torch.empty((T, hpr, 16), dtype=torch.int32, device="cuda")
    icp().icp_merge_tagged(recv, expect, nvp, s, i, errors, T=T, slot=1, world_size=ws,
                           heads_per_rank=hpr, capacity=cap, init_blocks=1, local_blocks=1,
                           spin_limit=1000)
    torch.cuda.synchronize()
    assert int(errors.item()) == T * hpr * ws
    assert torch.all(i == -1)
    assert torch.all(expect[1, :, :, :T] == 1) and torch.all(expect[0] == 0)
