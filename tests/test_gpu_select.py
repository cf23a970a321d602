"""icp_top16_select (CUDA) against the oracle's select run on the same plane:
ids and score bits must be identical."""
import pytest
import torch

import oracle
from sparse_attention_block_gb300 import workloads as W

from gpu_util import assert_select_equal, gpu_select

pytestmark = pytest.mark.gpu


def _check(plane, nvp, init, local, scale=1, offset=0, what=""):
    p = plane.cuda()
    n = nvp.cuda()
    gs, gi = gpu_select(p, n, init=init, local=local, scale=scale, offset=offset)
    torch.cuda.synchronize()
    os_, oi = oracle.select(plane.numpy(), nvp.numpy(), init_blocks=init, local_blocks=local,
                            index_scale=scale, index_offset=offset)
    assert_select_equal(gs, gi, os_, oi, what)


def test_standalone_plane_full_size():
    plane, nvp = W.make_select_plane(seed=0)
    _check(plane, nvp, W.SELECT_INIT, W.SELECT_LOCAL, what="[256,4,12284]")


@pytest.mark.parametrize("K", [1, 3, 16, 17, 100, 1024, 1025, 4096, 4097, 12287])
def test_widths_across_kernel_variants(K):
    plane, nvp = W.make_select_plane(T=8, K=K, seed=K)
    nvp = torch.tensor([1, 2, 16, 17, max(1, K // 2), K, K + 5, 1 << 30], dtype=torch.int32)
    for init, local in [(0, 0), (1, 2), (4, 8), (16, 0), (0, 16)]:
        _check(plane, nvp, init, local, what=f"K={K} init={init} local={local}")


def test_all_equal_and_minus_inf_rows():
    T, K = 4, 3000
    plane = torch.zeros((T, 4, K))
    plane[1] = -float("inf")
    plane[2, :, ::7] = 1.0
    plane[3] = torch.randn(4, K).round()            # heavy ties
    nvp = torch.tensor([K, K, K, 40], dtype=torch.int32)
    _check(plane, nvp, 1, 2, what="ties")


def test_adversarial_candidates_in_one_stripe():
    # the best values all sit in the columns of one thread's stripe
    for NT, K in [(128, 1024), (256, 4096), (512, 12287)]:
        plane = torch.randn((2, 4, K))
        cols = torch.arange(0, K, NT)
        plane[:, :, cols] = 100.0 + torch.arange(cols.numel()).float()
        plane[1, :, cols] = 100.0                    # tied as well
        nvp = torch.tensor([K, K], dtype=torch.int32)
        _check(plane, nvp, 2, 3, what=f"stripe NT={NT}")


def test_index_scale_and_offset():
    plane, _ = W.make_select_plane(T=6, K=2000, seed=9)
    nvp = torch.tensor([1, 10, 33, 500, 4000, 4001], dtype=torch.int32)
    for scale, offset in [(2, 0), (2, 1), (3, 2)]:
        _check(plane, nvp, 2, 4, scale=scale, offset=offset, what=f"scale {scale} off {offset}")


def test_signed_zero_and_duplicates():
    plane = torch.zeros((2, 4, 600))
    plane[0, :, :300] = -0.0
    plane[1] = torch.randn(4, 600)
    plane[1, :, 300:] = plane[1, :, :300]
    nvp = torch.tensor([600, 600], dtype=torch.int32)
    _check(plane, nvp, 3, 3, what="zeros")


def test_select_on_gpu_plane_of_batched_workload():
    from gpu_util import gpu_score, to_dev
    inp = W.make_decode_inputs(W.BATCHED, seed=1, batch=16)
    q, k, bt, sl, nvp = to_dev(inp)
    cols = W.columns_for(W.BATCHED, int(inp.seq_lens.max()))
    plane = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=128, dql=1)
    gs, gi = gpu_select(plane, nvp, init=1, local=4)
    torch.cuda.synchronize()
    os_, oi = oracle.select(plane.cpu().numpy(), inp.num_valid_pages.numpy(), init_blocks=1,
                            local_blocks=4)
    assert_select_equal(gs, gi, os_, oi, "batched plane")


def test_candidate_overflow_takes_the_exact_fallback():
    # Rows up to 2048 columns are read by one warp with float4 loads, lane l
    # owning columns 4 * (l + 32 j) .. + 3.  Making every column of lanes
    # 0..15 larger than the rest leaves about 16 * 64 keys above the
    # threshold, more than the per-warp candidate buffer, which exercises the
    # exact fallback selection.
    K = 2048
    plane = torch.randn((3, 4, K))
    lanes = torch.arange(16)
    cols = (4 * (lanes[:, None, None] + 32 * torch.arange(K // 128)[None, :, None])
            + torch.arange(4)[None, None, :]).reshape(-1)
    plane[:, :, cols] = 100.0 + torch.rand(cols.numel())
    plane[1, :, cols] = 100.0                       # and all tied
    nvp = torch.tensor([K, K, K // 2], dtype=torch.int32)
    for init, local in [(0, 0), (2, 3)]:
        _check(plane, nvp, init, local, what=f"overflow init={init} local={local}")


def test_long_rows_with_concentrated_maxima():
    # the same concentration on rows long enough for the CTA-per-row kernel
    K = 12284
    plane = torch.randn((3, 4, K))
    cols = torch.arange(0, K, 256)
    plane[:, :, cols] = 100.0 + torch.rand(cols.numel())
    plane[1, :, cols] = 100.0
    nvp = torch.tensor([K, K, K // 3], dtype=torch.int32)
    _check(plane, nvp, 2, 3, what="long rows")


def test_long_row_candidate_overflow_in_one_warp_slice():
    # Rows longer than 2048 columns are split over 4 warps; warp w owns the
    # float4 chunks w * 32 + lane + 128 j.  Large values over all of warp 0's
    # chunks overflow that warp's candidate buffer (exact fallback path).
    K = 12284
    plane = torch.randn((2, 4, K))
    f = (torch.arange(32)[:, None] + 128 * torch.arange(K // 512 + 1)[None, :]).reshape(-1)
    f = f[4 * f + 3 < K]
    cols = (4 * f[:, None] + torch.arange(4)[None, :]).reshape(-1)
    plane[:, :, cols] = 50.0 + torch.rand(cols.numel())
    plane[1, :, cols] = 50.0
    nvp = torch.tensor([K, 9000], dtype=torch.int32)
    for init, local in [(0, 0), (3, 4)]:
        _check(plane, nvp, init, local, what=f"warp-slice overflow init={init} local={local}")


@pytest.mark.parametrize("K", [4, 128, 204, 252, 256])
def test_short_rows_many_per_warp(K):
    # rows of at most 256 columns stay in registers and each warp takes a
    # row after another (5000 tokens: more rows than the grid's warps)
    plane, nvp = W.make_select_plane(T=1300, K=K, seed=K + 7)
    for init, local in [(1, 4), (0, 0), (4, 8)]:
        _check(plane, nvp, init, local, what=f"short K={K} init={init} local={local}")


def test_short_rows_candidate_overflow_and_ties():
    # all-equal and heavily tied short rows overflow the 128-key candidate
    # buffer, which takes the exact fallback
    T, K = 6, 256
    plane = torch.zeros((T, 4, K))
    plane[1] = 7.0
    plane[2, :, ::2] = 3.0
    plane[3] = torch.randn(4, K).round()
    plane[4] = -float("inf")
    plane[5, :, :200] = 1.0
    nvp = torch.tensor([K, K, K, 100, K, 230], dtype=torch.int32)
    for init, local in [(0, 0), (2, 3)]:
        _check(plane, nvp, init, local, what=f"short ties init={init} local={local}")


def test_many_full_length_rows():
    # 2048 rows of 12284 columns, more rows than the long-row kernel keeps
    # resident at once, with num_valid_pages at K and just below it
    T, K = 512, 12284
    plane, _ = W.make_select_plane(T=T, K=K, seed=21)
    nvp = torch.full((T,), K, dtype=torch.int32)
    nvp[::5] = K - 3
    _check(plane, nvp, 4, 8, what="many full rows")


def test_long_rows_with_empty_short_and_overlong_valid_ranges():
    # 5200 rows of 2052 columns with num_valid_pages from none (and negative)
    # through 16 and 17 (the all-kept boundary) to past K
    T, K = 1300, 2052
    plane, _ = W.make_select_plane(T=T, K=K, seed=22)
    g = torch.Generator().manual_seed(22)
    nvp = torch.randint(-3, K + 40, (T,), generator=g, dtype=torch.int32)
    nvp[::7] = 0
    nvp[1::7] = 16
    nvp[2::7] = 17
    for init, local in [(1, 3), (0, 0)]:
        _check(plane, nvp, init, local, what=f"valid ranges init={init} local={local}")


def test_long_rows_fewer_than_the_sms():
    # a handful of long rows: fewer CTAs than SMs
    for T in (1, 3):
        plane, nvp = W.make_select_plane(T=T, K=8192, seed=23 + T)
        _check(plane, nvp, 2, 2, what=f"T={T}")
