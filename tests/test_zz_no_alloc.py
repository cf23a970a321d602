"""icp_score_select_noalloc: the fused scorer + Top16 select for callers that
cannot allocate device memory when they call (fixed device pools, CUDA graph
recording, latency-critical paths).  Its scratch is the library's fixed
device array instead of a caller workspace.

The test calls it through the C ABI twice in a row, on different inputs: first
the largest multi-token batch the fixed scratch takes (294 requests of 4
tokens), then 40 requests of 8 tokens.  Each result must equal
icp_score_select with an ordinary workspace bit for bit (the tolerance every
Top16 test here uses), and its ids must equal the selection of the oracle's
exact plane wherever that plane decides the cut.  A batch one request past the
limit must be refused.  The file is named so that pytest collects it last.
"""
import dataclasses

import pytest
import torch

from sparse_attention_block_gb300 import workloads as W

pytestmark = pytest.mark.gpu


def _icp():
    from sparse_attention_block_gb300 import icp
    return icp


def _largest_batch(dql):
    icp = _icp()
    B = 1
    while icp.icp_score_select_workspace_bytes(B + 1, dql) <= icp.NOALLOC_SCRATCH_BYTES:
        B += 1
    return B


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
    return cols, (ns, ni), (ws_, wi)


def _against_the_oracle(inp, spec, cols, ids):
    from gpu_util import exact_selection_agrees
    from oracle.parallel import PlanePool
    hq, hk, hbt, hsl, hn = (t.cpu().numpy() for t in (inp.index_q, inp.index_k,
                                                      inp.block_table, inp.seq_lens,
                                                      inp.num_valid_pages))
    with PlanePool(hq, [hk], hbt, hsl) as pool:
        ex, ab = pool.decode_plane(k=0, cols=cols, rank=0, world_size=1,
                                   page_size=spec.page_size,
                                   decode_query_len=spec.decode_query_len)
    checked, skipped = exact_selection_agrees(ex, ab, ids.cpu().numpy(), hn, spec.init_blocks,
                                              spec.local_blocks)
    assert checked >= 0.97 * (checked + skipped), (checked, skipped)


def test_noalloc_matches_the_workspace_entry_point_and_the_oracle_on_two_calls_in_a_row():
    # multi-token decode draws (P256, init 2, local 4), with shorter contexts
    # so that the oracle's exact planes stay quick
    at_limit = dataclasses.replace(W.MULTITOKEN, batch=_largest_batch(4),
                                   seq_range=(300, 20000))
    eight = dataclasses.replace(W.MULTITOKEN, batch=40, decode_query_len=8,
                                seq_range=(1000, 60000))
    assert at_limit.batch == 294
    for spec, seed in ((at_limit, 31), (eight, 32)):
        inp = W.make_decode_inputs(spec, seed=seed)
        cols, (ns, ni), (ws_, wi) = _run_both(inp, spec)
        assert torch.equal(ni, wi), "ids differ from icp_score_select"
        assert torch.equal(ns.view(torch.int32), ws_.view(torch.int32)), "scores differ"
        assert int((ni >= 0).sum()) > 0
        _against_the_oracle(inp, spec, cols, ni)


@pytest.mark.parametrize("dql", [4, 8])
def test_noalloc_refuses_the_first_batch_beyond_its_fixed_scratch(dql):
    icp = _icp()
    B = _largest_batch(dql) + 1
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
