"""icp_score_select (fused scorer + Top16, CUDA) against icp_score followed by
icp_top16_select on the same inputs (bit for bit), and against the oracle's
select on the GPU plane."""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_block_gb300 import workloads as W

from gpu_util import assert_select_equal, gpu_score, gpu_select, icp, to_dev

pytestmark = pytest.mark.gpu


def _spec(page_size, ws, dql, seq_lens, init=1, local=2, maxdql=None):
    return W.DecodeSpec("f", batch=len(seq_lens), page_size=page_size, world_size=ws,
                        decode_query_len=dql, max_decode_query_len=maxdql or dql,
                        init_blocks=init, local_blocks=local, seq_lens=tuple(seq_lens))


def gpu_fused(q, k, bt, sl, nvp, *, cols, rank, ws, ps, dql, init, local, maxdql=None,
              errors=None):
    B = sl.shape[0]
    T = B * dql
    wsz = icp().icp_score_select_workspace_bytes(B, dql)
    work = torch.full((wsz,), 0xA5, dtype=torch.uint8, device=q.device)  # garbage on purpose
    s = torch.empty((T, 4, 16), dtype=torch.float32, device=q.device)
    i = torch.empty((T, 4, 16), dtype=torch.int32, device=q.device)
    icp().icp_score_select(q, k, bt, sl, nvp, s, i, work, cols=cols, rank=rank, world_size=ws,
                           page_size=ps, decode_query_len=dql,
                           max_decode_query_len=maxdql or dql, init_blocks=init,
                           local_blocks=local, errors=errors)
    return s, i


def _compare(inp, spec, rank=0, shard=None, cols=None, nvp=None, what=""):
    q, k, bt, sl, nv = to_dev(inp)
    if shard is not None:
        k = shard.cuda()
    if nvp is not None:
        nv = nvp.cuda()
    ws, ps, dql = spec.world_size, spec.page_size, spec.decode_query_len
    cols = cols or W.columns_for(spec, int(inp.seq_lens.max()))
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    fs, fi = gpu_fused(q, k, bt, sl, nv, cols=cols, rank=rank, ws=ws, ps=ps, dql=dql,
                       init=spec.init_blocks, local=spec.local_blocks,
                       maxdql=spec.max_decode_query_len, errors=errors)
    plane = gpu_score(q, k, bt, sl, cols=cols, rank=rank, world_size=ws, page_size=ps, dql=dql,
                      maxdql=spec.max_decode_query_len)
    scale, offset = (2, rank * 2 // ws) if (ps == 256 and ws > 1) else (1, 0)
    ss, si = gpu_select(plane, nv, init=spec.init_blocks, local=spec.local_blocks, scale=scale,
                        offset=offset)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0
    assert torch.equal(fi, si), f"{what}: fused ids differ from score + select"
    assert torch.equal(fs.view(torch.int32), ss.view(torch.int32)), f"{what}: fused scores differ"
    os_, oi = oracle.select(plane.cpu().numpy(), nv.cpu().numpy(), init_blocks=spec.init_blocks,
                            local_blocks=spec.local_blocks, index_scale=scale,
                            index_offset=offset)
    assert_select_equal(fs, fi, os_, oi, what)


def test_fused_tiny_workload():
    inp = W.make_decode_inputs(W.TINY, seed=0)
    _compare(inp, W.TINY, what="tiny")


@pytest.mark.parametrize("page_size,ws", [(128, 1), (128, 2), (128, 4), (256, 1), (256, 2),
                                          (256, 4)])
@pytest.mark.parametrize("dql", [1, 4, 8])
def test_fused_layouts_ragged(page_size, ws, dql):
    lens = [1, 5, 128, 129, 700, 2049, 5000, 9000]
    spec = _spec(page_size, ws, dql, lens, init=2, local=3)
    inp = W.make_decode_inputs(spec, seed=dql + ws)
    rp = page_size // ws
    for rank in range(ws):
        shard = inp.index_k[:, rank * rp:(rank + 1) * rp].contiguous()
        _compare(inp, spec, rank=rank, shard=shard, what=f"P{page_size} ws{ws} r{rank} dql{dql}")


def test_fused_many_requests_and_empty_ones():
    rng = np.random.default_rng(3)
    lens = rng.integers(1, 3000, 400).tolist()
    lens[5] = 0
    lens[77] = 0
    spec = _spec(128, 1, 2, lens, init=1, local=4)
    inp = W.make_decode_inputs(spec, seed=3)
    _compare(inp, spec, what="400 requests")


def test_fused_one_request_spanning_every_cta():
    spec = _spec(128, 1, 8, [300_000], init=4, local=8)
    inp = W.make_decode_inputs(spec, seed=8)
    _compare(inp, spec, what="one long request")


def test_fused_fewer_valid_pages_and_forced_everything():
    spec = _spec(128, 1, 2, [4000, 2500, 900], init=8, local=8)
    inp = W.make_decode_inputs(spec, seed=12)
    # requests have 32, 20 and 8 B128 blocks; num_valid_pages stays within them
    for nv in ([1, 2, 16, 17, 7, 8], [5, 16, 3, 20, 8, 8], [32, 17, 20, 1, 2, 3]):
        _compare(inp, spec, nvp=torch.tensor(nv, dtype=torch.int32), what=f"nvp {nv}")


def test_fused_plane_width_larger_than_needed():
    spec = _spec(256, 1, 4, [3000, 200, 7000], init=2, local=4, maxdql=8)
    inp = W.make_decode_inputs(spec, seed=21)
    _compare(inp, spec, cols=W.columns_for(spec, 7000) + 20, what="wide plane")


def test_fused_twice_in_a_row_reuses_the_workspace():
    inp = W.make_decode_inputs(W.BATCHED, seed=4, batch=20)
    q, k, bt, sl, nv = to_dev(inp)
    cols = W.columns_for(W.BATCHED, int(inp.seq_lens.max()))
    B, dql = 20, 1
    wsz = icp().icp_score_select_workspace_bytes(B, dql)
    work = torch.empty((wsz,), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(2):
        s = torch.empty((B, 4, 16), dtype=torch.float32, device="cuda")
        i = torch.empty((B, 4, 16), dtype=torch.int32, device="cuda")
        icp().icp_score_select(q, k, bt, sl, nv, s, i, work, cols=cols, rank=0, world_size=1,
                               page_size=128, decode_query_len=1, max_decode_query_len=1,
                               init_blocks=1, local_blocks=4)
        outs.append((s, i))
    torch.cuda.synchronize()
    assert torch.equal(outs[0][1], outs[1][1])
    assert torch.equal(outs[0][0].view(torch.int32), outs[1][0].view(torch.int32))
