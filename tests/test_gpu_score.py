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


def _bad_table_case(page_size):
    """Requests whose block tables hold entries outside the pool: request 0
    two of them, request 1 one, request 3 two far apart (so that different
    CTAs read them); request 2 none.  Returns the case, the bad table, the
    oracle's reading of it (the entries point at an extra all-zero page) and
    the number of requests holding a bad entry."""
    seq_lens = [700, 300, 500, 20000]
    spec, inp = _case(page_size, 1, 2, seq_lens, seed=5)
    num_pages = inp.index_k.shape[0]
    bt = inp.block_table.clone()
    far = (100, 140) if page_size == 128 else (40, 70)
    bad = [(0, 1, num_pages + 7), (0, 2, num_pages), (1, 0, -2), (3, far[0], -1),
           (3, far[1], 1 << 30)]
    for b, j, v in bad:
        bt[b, j] = v
    kz = torch.cat([inp.index_k, torch.zeros((1,) + tuple(inp.index_k.shape[1:]),
                                             dtype=torch.uint8)])
    bz = bt.clone()
    for b, j, _ in bad:
        bz[b, j] = num_pages
    return spec, inp, bt, kz, bz, len({b for b, _, _ in bad})


@pytest.mark.parametrize("page_size", [128, 256])
@pytest.mark.parametrize("pdl", [False, True])
def test_block_table_entries_outside_the_pool_are_counted_and_read_as_zero_keys(page_size, pdl):
    # the tensor map fills those rows with zeros, so the plane must equal the
    # oracle's plane with the entries pointing at an all-zero page; errors
    # counts each request that holds such an entry once
    from gpu_util import icp, sentinel_plane
    spec, inp, bt, kz, bz, nbad = _bad_table_case(page_size)
    q, k, _, sl, _ = to_dev(inp)
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    cols = W.columns_for(spec, int(inp.seq_lens.max()))
    gp = sentinel_plane(inp.T, cols)
    icp().icp_score(q, k, bt.cuda(), sl, gp, rank=0, world_size=1, page_size=page_size,
                    decode_query_len=2, max_decode_query_len=2, enable_pdl=pdl, errors=errors)
    torch.cuda.synchronize()
    assert int(errors.item()) == nbad
    ex, ab = oracle_plane(inp.index_q, kz, bz, inp.seq_lens, cols=cols, rank=0, world_size=1,
                          page_size=page_size, dql=2)
    assert_plane_matches(gp, ex, ab, f"pages outside the pool, P{page_size}")


@pytest.mark.parametrize("page_size", [128, 256])
def test_fused_path_counts_block_table_entries_outside_the_pool(page_size):
    from gpu_util import gpu_select, icp
    spec, inp, bt, _, _, nbad = _bad_table_case(page_size)
    q, k, _, sl, nvp = to_dev(inp)
    btd = bt.cuda()
    cols = W.columns_for(spec, int(inp.seq_lens.max()))
    T = inp.T
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    work = torch.empty((icp().icp_score_select_workspace_bytes(4, 2),), dtype=torch.uint8,
                       device="cuda")
    fs = torch.empty((T, 4, 16), device="cuda")
    fi = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    icp().icp_score_select(q, k, btd, sl, nvp, fs, fi, work, cols=cols, rank=0, world_size=1,
                           page_size=page_size, decode_query_len=2, max_decode_query_len=2,
                           init_blocks=1, local_blocks=2, errors=errors)
    torch.cuda.synchronize()
    assert int(errors.item()) == nbad
    gp = gpu_score(q, k, btd, sl, cols=cols, rank=0, world_size=1, page_size=page_size, dql=2)
    s, i = gpu_select(gp, nvp, init=1, local=2)
    torch.cuda.synchronize()
    assert torch.equal(fi, i) and torch.equal(fs.view(torch.int32), s.view(torch.int32))


def test_prefill_window_counts_a_request_with_bad_entries_once():
    # request 0's 150-token chunk is three plan records that all read its
    # early pages; request 1's bad page is reached only by its later records
    from gpu_util import icp, sentinel_plane
    seq_lens, chunks = [3000, 9000], [150, 130]
    spec = W.DecodeSpec("w", batch=2, page_size=128, world_size=1, decode_query_len=1,
                        max_decode_query_len=1, init_blocks=1, local_blocks=3,
                        seq_lens=tuple(seq_lens))
    inp = W.make_decode_inputs(spec, seed=8)
    num_pages = inp.index_k.shape[0]
    bt = inp.block_table.clone()
    bt[0, 3] = -4
    bt[0, 20] = num_pages
    last = (9000 - 130 + 64) // 128 + 1            # past the first record's last column
    bt[1, last] = num_pages + 1
    T = sum(chunks)
    g = torch.Generator().manual_seed(8)
    q = (0.5 * torch.randn((T, 4, 128), generator=g) + 1.5 * inp.u).to(
        torch.float8_e4m3fn).view(torch.uint8)
    qo = torch.tensor([0, chunks[0], T], dtype=torch.int32, device="cuda")
    cols = W.columns_for(spec, max(seq_lens))
    plan = torch.empty((icp().icp_prefill_plan_words(2, T),), dtype=torch.int32, device="cuda")
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    icp().icp_prefill_plan(qo, inp.seq_lens.cuda(), plan, T=T, errors=errors)
    gp = sentinel_plane(T, cols)
    icp().icp_prefill_score(q.cuda(), inp.index_k.cuda(), bt.cuda(), plan, gp, rank=0,
                            world_size=1, page_size=128, errors=errors)
    torch.cuda.synchronize()
    assert int(errors.item()) == 2
    import oracle
    kz = torch.cat([inp.index_k, torch.zeros((1, 128, 128), dtype=torch.uint8)])
    bz = bt.clone()
    bz[0, 3] = bz[0, 20] = bz[1, last] = num_pages
    ex, ab = oracle.score_chunks(q.numpy(), kz.numpy(), bz.numpy(), inp.seq_lens.numpy(),
                                 qo.cpu().numpy(), cols=cols, rank=0, world_size=1,
                                 page_size=128)
    assert_plane_matches(gp, ex, ab, "prefill window with pages outside the pool")


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
