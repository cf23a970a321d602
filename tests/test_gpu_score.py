"""icp_score (CUDA, through the C ABI) against the oracle, element by element.

Tolerance (per written plane entry): |gpu - exact| <= 1e-5 * S + 1e-7, S the
largest sum_i |q_i k_i| among the column's visible keys; -inf entries match
exactly; entries outside each request's written columns keep a sentinel.
"""
import numpy as np
import pytest
import torch

from sparse_attention_block_gb300 import workloads as W

from gpu_util import assert_plane_matches, gpu_score, oracle_plane, to_dev

pytestmark = pytest.mark.gpu


def _case(page_size, world_size, dql, seq_lens, seed=0, maxdql=None):
    spec = W.DecodeSpec("case", batch=len(seq_lens), page_size=page_size, world_size=world_size,
                        decode_query_len=dql, max_decode_query_len=maxdql or dql,
                        init_blocks=1, local_blocks=2, seq_lens=tuple(seq_lens))
    return spec, W.make_decode_inputs(spec, seed=seed)


def test_tiny_workload_full_plane():
    inp = W.make_decode_inputs(W.TINY, seed=0)
    q, k, bt, sl, _ = to_dev(inp)
    cols = W.columns_for(W.TINY, 2500)
    gp = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=128, dql=1)
    torch.cuda.synchronize()
    ex, ab = oracle_plane(inp.index_q, inp.index_k, inp.block_table, inp.seq_lens, cols=cols,
                          rank=0, world_size=1, page_size=128, dql=1)
    assert_plane_matches(gp, ex, ab, "tiny")


RAGGED = [1, 2, 127, 128, 129, 255, 256, 257, 1000, 3001, 5000]


@pytest.mark.parametrize("page_size,world_size", [(128, 1), (128, 2), (128, 4), (256, 1),
                                                  (256, 2), (256, 4)])
@pytest.mark.parametrize("dql", [1, 3, 8])
def test_layouts_ragged_lengths(page_size, world_size, dql):
    spec, inp = _case(page_size, world_size, dql, RAGGED, seed=dql)
    rp = page_size // world_size
    cols = W.columns_for(spec, max(RAGGED)) + 8   # extra columns must stay untouched
    q = inp.index_q.cuda()
    bt = inp.block_table.cuda()
    sl = inp.seq_lens.cuda()
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    for rank in range(world_size):
        shard = inp.index_k[:, rank * rp:(rank + 1) * rp].contiguous()
        gp = gpu_score(q, shard.cuda(), bt, sl, cols=cols, rank=rank, world_size=world_size,
                       page_size=page_size, dql=dql, errors=errors)
        torch.cuda.synchronize()
        ex, ab = oracle_plane(inp.index_q, shard, inp.block_table, inp.seq_lens, cols=cols,
                              rank=rank, world_size=world_size, page_size=page_size, dql=dql)
        assert_plane_matches(gp, ex, ab, f"P{page_size} ws{world_size} rank{rank} dql{dql}")
    assert int(errors.item()) == 0


def test_max_decode_query_len_padding_rows_do_not_leak():
    # dql 2 with max 8: the MMA tile holds 32 query rows, only 8 belong to a request
    spec, inp = _case(128, 1, 2, [700, 20, 1300], seed=5, maxdql=8)
    q, k, bt, sl, _ = to_dev(inp)
    cols = W.columns_for(spec, 1300)
    gp = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=128, dql=2, maxdql=8)
    torch.cuda.synchronize()
    ex, ab = oracle_plane(inp.index_q, inp.index_k, inp.block_table, inp.seq_lens, cols=cols,
                          rank=0, world_size=1, page_size=128, dql=2)
    assert_plane_matches(gp, ex, ab, "dql2/max8")


def test_block_table_with_row_stride_and_zero_length_requests():
    spec, inp = _case(128, 1, 1, [0, 300, 0, 129], seed=3)
    q, k, _, sl, _ = to_dev(inp)
    wide = torch.full((4, 11), -5, dtype=torch.int32)
    wide[:, :inp.block_table.shape[1]] = inp.block_table
    bt = wide.cuda()[:, :inp.block_table.shape[1] + 2]   # row stride 11, non-contiguous view
    cols = 8
    gp = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=128, dql=1)
    torch.cuda.synchronize()
    ex, ab = oracle_plane(inp.index_q, inp.index_k, inp.block_table, inp.seq_lens, cols=cols,
                          rank=0, world_size=1, page_size=128, dql=1)
    assert_plane_matches(gp, ex, ab, "strided table")


@pytest.mark.parametrize("page_size", [128, 256])
def test_block_table_entries_outside_the_pool_read_as_zero_keys(page_size):
    # entries past the pool and below 0 inside each request's pages: the
    # tensor map fills those rows with zeros, so the plane must equal the
    # oracle's plane with the entries pointing at an all-zero page
    spec, inp = _case(page_size, 1, 2, [700, 300], seed=5)
    num_pages = inp.index_k.shape[0]
    bt = inp.block_table.clone()
    bt[0, 1] = num_pages + 7
    bt[0, 2] = num_pages
    bt[1, 0] = -2
    kz = torch.cat([inp.index_k, torch.zeros((1,) + tuple(inp.index_k.shape[1:]),
                                             dtype=torch.uint8)])
    bz = bt.clone()
    bz[0, 1] = bz[0, 2] = bz[1, 0] = num_pages
    q, k, _, sl, _ = to_dev(inp)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    cols = W.columns_for(spec, 700)
    gp = gpu_score(q, k, bt.cuda(), sl, cols=cols, rank=0, world_size=1, page_size=page_size,
                   dql=2, errors=errors)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0
    ex, ab = oracle_plane(inp.index_q, kz, bz, inp.seq_lens, cols=cols, rank=0, world_size=1,
                          page_size=page_size, dql=2)
    assert_plane_matches(gp, ex, ab, f"pages outside the pool, P{page_size}")


def test_extreme_fp8_values_stay_within_tolerance():
    # max-magnitude and subnormal codes; sums of 128 products of 448 * 448
    spec = W.DecodeSpec("x", batch=2, page_size=128, world_size=1, decode_query_len=2,
                        max_decode_query_len=2, init_blocks=0, local_blocks=0,
                        seq_lens=(300, 1000))
    inp = W.make_decode_inputs(spec, seed=11)
    g = torch.Generator().manual_seed(11)
    codes = torch.tensor([0x7E, 0xFE, 0x01, 0x81, 0x00, 0x80, 0x38, 0xB8], dtype=torch.uint8)
    pick = torch.randint(0, len(codes), inp.index_k.shape, generator=g)
    inp.index_k.copy_(codes[pick])
    pickq = torch.randint(0, len(codes), inp.index_q.shape, generator=g)
    inp.index_q.copy_(codes[pickq])
    q, k, bt, sl, _ = to_dev(inp)
    cols = 8
    gp = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=128, dql=2)
    torch.cuda.synchronize()
    ex, ab = oracle_plane(inp.index_q, inp.index_k, inp.block_table, inp.seq_lens, cols=cols,
                          rank=0, world_size=1, page_size=128, dql=2)
    assert_plane_matches(gp, ex, ab, "extreme codes")


def test_many_requests_spread_over_all_ctas():
    rng = np.random.default_rng(4)
    lens = rng.integers(1, 4000, 300).tolist()
    spec, inp = _case(128, 1, 1, lens, seed=4)
    q, k, bt, sl, _ = to_dev(inp)
    cols = W.columns_for(spec, max(lens))
    gp = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=128, dql=1)
    torch.cuda.synchronize()
    ex, ab = oracle_plane(inp.index_q, inp.index_k, inp.block_table, inp.seq_lens, cols=cols,
                          rank=0, world_size=1, page_size=128, dql=1)
    assert_plane_matches(gp, ex, ab, "300 requests")


def test_repeated_calls_are_deterministic():
    inp = W.make_decode_inputs(W.BATCHED, seed=2, batch=8)
    q, k, bt, sl, _ = to_dev(inp)
    cols = W.columns_for(W.BATCHED, int(inp.seq_lens.max()))
    a = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=128, dql=1)
    b = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=128, dql=1)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_early_start_under_programmatic_dependent_launch_changes_nothing():
    # the scorer launched with enable_pdl right after other kernels (here a
    # merge and a select) gives the same plane as a plain launch
    inp = W.make_decode_inputs(W.MULTITOKEN, seed=6, batch=12)
    q, k, bt, sl, nvp = to_dev(inp)
    spec = W.MULTITOKEN
    cols = W.columns_for(spec, int(inp.seq_lens.max()))
    from gpu_util import icp, sentinel_plane
    ref = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=256, dql=4, maxdql=8)
    T = inp.T
    for _ in range(3):
        plane = sentinel_plane(T, cols)
        # a preceding merge (triggers its dependents early) and a select
        recv = torch.zeros((icp().recv_rows(1, 4, T), 33), dtype=torch.int32, device="cuda")
        errors = torch.zeros(1, dtype=torch.int32, device="cuda")
        s = torch.empty((T, 4, 16), device="cuda")
        i = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
        icp().icp_merge(recv, nvp, s, i, errors, T=T, slot=0, world_size=1, heads_per_rank=4,
                        capacity=T, init_blocks=1, local_blocks=1, spin_limit=100)
        icp().icp_score(q, k, bt, sl, plane, rank=0, world_size=1, page_size=256,
                        decode_query_len=4, max_decode_query_len=8, enable_pdl=True)
        torch.cuda.synchronize()
        assert torch.equal(plane.view(torch.int32), ref.view(torch.int32))
