"""icp_score_select_noalloc: the fused scorer + Top16 select for callers that
cannot allocate device memory when they call (fixed device pools, CUDA graph
recording, latency-critical paths).  Its scratch is the library's fixed
device array instead of a caller workspace.

The test calls it through the C ABI twice in a row, on different inputs, and
checks each result against icp_score_select with an ordinary workspace: ids
and score bits must be identical (the tolerance every Top16 test here uses).
It also checks that a batch needing more scratch than the fixed array is
refused.  The file is named so that pytest collects it last.
"""
import pytest
import torch

from sparse_attention_block_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _icp():
    from sparse_attention_block_gb300 import icp
    return icp


def _run_both(inp, spec):
    icp = _icp()
    dev = torch.device("cuda")
    q, k, bt, sl, nvp = (inp.index_q.to(dev), inp.index_k.to(dev), inp.block_table.to(dev),
                         inp.seq_lens.to(dev), inp.num_valid_pages.to(dev))
    B, dql = sl.shape[0], spec.decode_query_len
    T = B * dql
    cols = icp.icp_score_columns(int(inp.seq_lens.max()), spec.page_size, spec.world_size)
    kw = dict(cols=cols, rank=0, world_size=1, page_size=spec.page_size, decode_query_len=dql,
              max_decode_query_len=spec.max_decode_query_len, init_blocks=spec.init_blocks,
              local_blocks=spec.local_blocks)
    errors = torch.zeros(1, dtype=torch.int32, device=dev)
    ns = torch.empty((T, 4, 16), dtype=torch.float32, device=dev)
    ni = torch.empty((T, 4, 16), dtype=torch.int32, device=dev)
    icp.icp_score_select_noalloc(q, k, bt, sl, nvp, ns, ni, errors=errors, **kw)
    work = torch.empty((icp.icp_score_select_workspace_bytes(B, dql),), dtype=torch.uint8,
                       device=dev)
    ws_ = torch.empty((T, 4, 16), dtype=torch.float32, device=dev)
    wi = torch.empty((T, 4, 16), dtype=torch.int32, device=dev)
    icp.icp_score_select(q, k, bt, sl, nvp, ws_, wi, work, errors=errors, **kw)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0
    return (ns, ni), (ws_, wi)


def test_noalloc_matches_the_workspace_entry_point_on_two_calls_in_a_row():
    spec = W.MULTITOKEN
    first = W.make_decode_inputs(spec, seed=31, batch=24)
    second = W.make_decode_inputs(spec, seed=32, batch=40)
    for inp in (first, second):
        (ns, ni), (ws_, wi) = _run_both(inp, spec)
        assert torch.equal(ni, wi), "ids differ from icp_score_select"
        assert torch.equal(ns.view(torch.int32), ws_.view(torch.int32)), "scores differ"
        assert int((ni >= 0).sum()) > 0


def test_noalloc_refuses_a_batch_beyond_its_fixed_scratch():
    icp = _icp()
    B, dql = 1024, 8
    assert icp.icp_score_select_workspace_bytes(B, dql) > icp.NOALLOC_SCRATCH_BYTES
    dev = torch.device("cuda")
    q = torch.zeros((B * dql, 4, 128), dtype=torch.uint8, device=dev)
    k = torch.zeros((4, 128, 128), dtype=torch.uint8, device=dev)
    bt = torch.zeros((B, 1), dtype=torch.int32, device=dev)
    sl = torch.full((B,), 10, dtype=torch.int32, device=dev)
    nvp = torch.ones((B * dql,), dtype=torch.int32, device=dev)
    s = torch.empty((B * dql, 4, 16), dtype=torch.float32, device=dev)
    i = torch.empty((B * dql, 4, 16), dtype=torch.int32, device=dev)
    with pytest.raises(icp.IcpError) as e:
        icp.icp_score_select_noalloc(q, k, bt, sl, nvp, s, i, cols=4, rank=0, world_size=1,
                                     page_size=128, decode_query_len=dql,
                                     max_decode_query_len=dql, init_blocks=1, local_blocks=2)
    assert e.value.status == icp.ERR_INVALID_ARG
