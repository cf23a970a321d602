"""The scorer and the fused scorer + select at the documented limits, against
the oracle: the widest plane (cols = 8192, a request of 1,048,576 tokens at
page size 128) and the largest batch (4096 requests per call).

msa_icp_decode_index_score_sharded bounds score_out's columns by 8192; the
library's batch limit ICP_MAX_BATCH is 4096 requests.
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


def _fused(inp, spec, cols):
    T = inp.T
    dev = inp.index_q.device
    fs = torch.empty((T, 4, 16), dtype=torch.float32, device=dev)
    fi = torch.empty((T, 4, 16), dtype=torch.int32, device=dev)
    work = torch.empty((icp().icp_score_select_workspace_bytes(len(inp.seq_lens),
                                                               spec.decode_query_len),),
                       dtype=torch.uint8, device=dev)
    errors = torch.zeros(1, dtype=torch.int32, device=dev)
    icp().icp_score_select(inp.index_q, inp.index_k, inp.block_table, inp.seq_lens,
                           inp.num_valid_pages, fs, fi, work, cols=cols, rank=0, world_size=1,
                           page_size=spec.page_size, decode_query_len=spec.decode_query_len,
                           max_decode_query_len=spec.max_decode_query_len,
                           init_blocks=spec.init_blocks, local_blocks=spec.local_blocks,
                           errors=errors)
    return fs, fi, errors


def _check(spec, seed):
    inp = W.make_decode_inputs(spec, seed=seed, device="cuda")
    cols = icp().icp_score_columns(int(inp.seq_lens.max()), spec.page_size, 1)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    plane = gpu_score(inp.index_q, inp.index_k, inp.block_table, inp.seq_lens, cols=cols,
                      rank=0, world_size=1, page_size=spec.page_size,
                      dql=spec.decode_query_len, maxdql=spec.max_decode_query_len,
                      errors=errors)
    s, i = gpu_select(plane, inp.num_valid_pages, init=spec.init_blocks,
                      local=spec.local_blocks)
    fs, fi, ferr = _fused(inp, spec, cols)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0 and int(ferr.item()) == 0
    gp, hn = plane.cpu().numpy(), inp.num_valid_pages.cpu().numpy()
    os_, oi = oracle.select(gp, hn, init_blocks=spec.init_blocks,
                            local_blocks=spec.local_blocks)
    assert_select_equal(s, i, os_, oi, f"{spec.name} select")
    assert_select_equal(fs, fi, os_, oi, f"{spec.name} fused")
    hq, hk, hbt, hsl = (t.cpu().numpy() for t in (inp.index_q, inp.index_k, inp.block_table,
                                                  inp.seq_lens))
    with PlanePool(hq, [hk], hbt, hsl) as pool:
        ex, ab = pool.decode_plane(k=0, cols=cols, rank=0, world_size=1,
                                   page_size=spec.page_size,
                                   decode_query_len=spec.decode_query_len)
    assert_plane_matches(gp, ex, ab, spec.name)
    checked, skipped = exact_selection_agrees(ex, ab, i.cpu().numpy(), hn, spec.init_blocks,
                                              spec.local_blocks)
    assert checked >= 0.97 * (checked + skipped)
    return cols


def test_the_widest_plane():
    spec = W.DecodeSpec("widest", batch=3, page_size=128, world_size=1, decode_query_len=2,
                        max_decode_query_len=2, init_blocks=2, local_blocks=5, planted=0.01,
                        seq_lens=(8192 * 128, 300, 8192 * 128 - 129))
    assert _check(spec, seed=41) == 8192


def test_the_largest_batch():
    spec = W.DecodeSpec("largest", batch=4096, page_size=256, world_size=1,
                        decode_query_len=1, max_decode_query_len=1, init_blocks=1,
                        local_blocks=3, seq_range=(1, 2600))
    _check(spec, seed=42)
