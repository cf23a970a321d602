"""Prefill window path (CUDA, through the C ABI) against the oracle.

Plan -> icp_prefill_score (plane within the scorer tolerance, untouched
columns kept) -> icp_prefill_select (carrier rows bit-exact against the
oracle's carrier of the GPU's own plane) -> exchange on the host ->
icp_prefill_merge (bit-exact; sharded merges equal the unsharded Top16).
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_block_gb300 import workloads as W

from gpu_util import SENTINEL_BITS, assert_plane_matches, icp, sentinel_plane

pytestmark = pytest.mark.gpu


def _window(seq_lens, chunks, page_size=128, world_size=1, seed=0):
    """Seeded window: request b contributes its newest chunks[b] tokens."""
    spec = W.DecodeSpec("w", batch=len(seq_lens), page_size=page_size, world_size=world_size,
                        decode_query_len=1, max_decode_query_len=1, init_blocks=1,
                        local_blocks=3, seq_lens=tuple(seq_lens))
    inp = W.make_decode_inputs(spec, seed=seed)
    qo = torch.tensor(np.concatenate([[0], np.cumsum(chunks)]), dtype=torch.int32)
    T = int(qo[-1])
    g = torch.Generator().manual_seed(seed + 100)
    qf = 0.5 * torch.randn((T, 4, 128), generator=g) + 1.5 * inp.u
    q = qf.to(torch.float8_e4m3fn).view(torch.uint8)
    pos = np.concatenate([np.arange(L - n, L) for L, n in zip(seq_lens, chunks)]).astype(np.int64)
    nvp = torch.tensor((pos + 1 + 127) // 128, dtype=torch.int32)
    return spec, inp, q, qo, nvp


def _gpu_plane(q, k, bt, sl, qo, *, cols, rank, world_size, page_size, errors=None):
    T = q.shape[0]
    B = sl.shape[0]
    plan = torch.full((icp().icp_prefill_plan_words(B, T),), -7, dtype=torch.int32,
                      device="cuda")
    icp().icp_prefill_plan(qo, sl, plan, T=T, errors=errors)
    out = sentinel_plane(T, cols)
    icp().icp_prefill_score(q, k, bt, plan, out, rank=rank, world_size=world_size,
                            page_size=page_size, errors=errors)
    return out, plan


# chunks below, at and across the 64-token records (and across their 32-token
# row halves), an empty one, a whole prompt
RAGGED = ([1000, 2500, 129, 300, 40, 9000, 5000], [1, 17, 129, 64, 0, 65, 100])


@pytest.mark.parametrize("page_size,ws", [(128, 1), (128, 2), (128, 4), (256, 1), (256, 2),
                                          (256, 4)])
def test_prefill_plane_ragged_chunks(page_size, ws):
    seq_lens, chunks = RAGGED
    spec, inp, q, qo, _ = _window(seq_lens, chunks, page_size=page_size, world_size=ws,
                                  seed=page_size + ws)
    cols = W.columns_for(spec, max(seq_lens)) + 8    # extra columns must stay untouched
    rp = page_size // ws
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    for rank in range(ws):
        shard = inp.index_k[:, rank * rp:(rank + 1) * rp].contiguous()
        gp, _ = _gpu_plane(q.cuda(), shard.cuda(), inp.block_table.cuda(), inp.seq_lens.cuda(),
                           qo.cuda(), cols=cols, rank=rank, world_size=ws, page_size=page_size,
                           errors=errors)
        torch.cuda.synchronize()
        ex, ab = oracle.score_chunks(q.numpy(), shard.numpy(), inp.block_table.numpy(),
                                     inp.seq_lens.numpy(), qo.numpy(), cols=cols, rank=rank,
                                     world_size=ws, page_size=page_size)
        assert_plane_matches(gp, ex, ab, f"prefill P{page_size} ws{ws} rank{rank}")
    assert int(errors.item()) == 0


def test_plan_records_by_hand():
    sl = torch.tensor([200, 40, 20], dtype=torch.int32, device="cuda")
    qo = torch.tensor([0, 150, 150, 153], dtype=torch.int32, device="cuda")  # chunks 150, 0, 3
    plan = torch.full((icp().icp_prefill_plan_words(3, 153),), -7, dtype=torch.int32,
                      device="cuda")
    icp().icp_prefill_plan(qo, sl, plan, T=153)
    p = plan.cpu().numpy()
    assert p[0] == 4
    recs = p[8:8 + 4 * 8].reshape(4, 8)
    # {first token, table row, last position + 1, tokens, request seq_len, 0, 0, 0}:
    # records of at most 64 tokens; request 0's chunk sits at positions 50..199
    assert recs.tolist() == [[0, 0, 114, 64, 200, 0, 0, 0], [64, 0, 178, 64, 200, 0, 0, 0],
                             [128, 0, 200, 22, 200, 0, 0, 0], [150, 2, 20, 3, 20, 0, 0, 0]]


def test_invalid_chunk_is_counted_and_its_rows_left_alone():
    seq_lens, chunks = [300, 50, 700], [5, 3, 9]
    spec, inp, q, qo, _ = _window(seq_lens, chunks, seed=4)
    sl = inp.seq_lens.clone()
    sl[1] = 2                                    # 3 tokens of a 2-token request
    cols = W.columns_for(spec, max(seq_lens))
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    gp, _ = _gpu_plane(q.cuda(), inp.index_k.cuda(), inp.block_table.cuda(), sl.cuda(),
                       qo.cuda(), cols=cols, rank=0, world_size=1, page_size=128,
                       errors=errors)
    torch.cuda.synchronize()
    assert int(errors.item()) == 1
    g = gp.cpu().numpy()
    assert np.all(g[5:8].view(np.int32) == SENTINEL_BITS)
    keep = np.r_[0:5, 8:17]
    qn = q.numpy()
    ex, ab = oracle.score_chunks(qn, inp.index_k.numpy(), inp.block_table.numpy(),
                                 inp.seq_lens.numpy(), qo.numpy(), cols=cols, rank=0,
                                 world_size=1, page_size=128)
    assert_plane_matches(g[keep], ex[keep], ab[keep], "valid requests")


def test_prefill_chain_unsharded_bit_exact():
    seq_lens, chunks = [3000, 700, 5000, 90], [64, 200, 13, 90]
    spec, inp, q, qo, nvp = _window(seq_lens, chunks, seed=9)
    cols = W.columns_for(spec, max(seq_lens))
    gp, _ = _gpu_plane(q.cuda(), inp.index_k.cuda(), inp.block_table.cuda(),
                       inp.seq_lens.cuda(), qo.cuda(), cols=cols, rank=0, world_size=1,
                       page_size=128)
    T = q.shape[0]
    car = torch.zeros((1, T, 4, 32), dtype=torch.int32, device="cuda")
    icp().icp_prefill_select(gp, nvp.cuda(), car, world_size=1, heads_per_rank=4, init_blocks=1,
                             local_blocks=3)
    out_s = torch.empty((T, 4, 16), device="cuda")
    out_i = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    icp().icp_prefill_merge(car, nvp.cuda(), out_s, out_i, world_size=1, heads_per_rank=4,
                            init_blocks=1, local_blocks=3)
    torch.cuda.synchronize()
    plane = gp.cpu().numpy()
    ref = oracle.carrier(plane, nvp.numpy(), world_size=1, heads_per_rank=4, init_blocks=1,
                         local_blocks=3)
    np.testing.assert_array_equal(car.cpu().numpy(), ref)
    ms, mi = oracle.merge_carrier(ref, nvp.numpy(), world_size=1, heads_per_rank=4,
                                  init_blocks=1, local_blocks=3)
    np.testing.assert_array_equal(out_i.cpu().numpy(), mi)
    np.testing.assert_array_equal(out_s.cpu().numpy().view(np.int32), ms.view(np.int32))


@pytest.mark.parametrize("page_size,ws", [(128, 2), (128, 4), (256, 2), (256, 4)])
def test_sharded_prefill_merge_equals_unsharded(page_size, ws):
    seq_lens, chunks = [4000, 900, 2600], [40, 100, 7]
    spec, inp, q, qo, nvp = _window(seq_lens, chunks, page_size=page_size, world_size=ws,
                                    seed=21 + ws)
    T = q.shape[0]
    hpr = 4 // ws
    rp = page_size // ws
    cols = W.columns_for(spec, max(seq_lens))
    qd, btd, sld, qod, nvpd = (q.cuda(), inp.block_table.cuda(), inp.seq_lens.cuda(),
                               qo.cuda(), nvp.cuda())
    cars = []
    for rank in range(ws):
        shard = inp.index_k[:, rank * rp:(rank + 1) * rp].contiguous().cuda()
        gp, _ = _gpu_plane(qd, shard, btd, sld, qod, cols=cols, rank=rank, world_size=ws,
                           page_size=page_size)
        scale, offset = (1, 0) if page_size == 128 else (2, rank * 2 // ws)
        car = torch.zeros((ws, T, hpr, 32), dtype=torch.int32, device="cuda")
        icp().icp_prefill_select(gp, nvpd, car, world_size=ws, heads_per_rank=hpr,
                                 init_blocks=1, local_blocks=3, index_scale=scale,
                                 index_offset=offset)
        torch.cuda.synchronize()
        ref = oracle.carrier(gp.cpu().numpy(), nvp.numpy(), world_size=ws, heads_per_rank=hpr,
                             init_blocks=1, local_blocks=3, index_scale=scale,
                             index_offset=offset)
        np.testing.assert_array_equal(car.cpu().numpy(), ref)
        cars.append(car)
    # unsharded plane (one column per B128 block) and its Top16
    ucols = W.columns_for(W.DecodeSpec("u", batch=1, page_size=page_size, world_size=1,
                                       decode_query_len=1, max_decode_query_len=1,
                                       init_blocks=0, local_blocks=0, seq_lens=(1,)),
                          max(seq_lens))
    up, _ = _gpu_plane(qd, inp.index_k.cuda(), btd, sld, qod, cols=ucols, rank=0, world_size=1,
                       page_size=page_size)
    us = torch.empty((T, 4, 16), device="cuda")
    ui = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    icp().icp_top16_select(up, nvpd, us, ui, init_blocks=1, local_blocks=3)
    for owner in range(ws):
        received = torch.stack([cars[s][owner] for s in range(ws)]).contiguous()
        ms = torch.empty((T, hpr, 16), device="cuda")
        mi = torch.empty((T, hpr, 16), dtype=torch.int32, device="cuda")
        icp().icp_prefill_merge(received, nvpd, ms, mi, world_size=ws, heads_per_rank=hpr,
                                init_blocks=1, local_blocks=3)
        torch.cuda.synchronize()
        heads = slice(owner * hpr, (owner + 1) * hpr)
        assert torch.equal(mi, ui[:, heads]), f"owner {owner}: merged ids differ"
        assert torch.equal(ms.view(torch.int32), us[:, heads].view(torch.int32))
        os_, oi = oracle.merge_carrier(received.cpu().numpy(), nvp.numpy(), world_size=ws,
                                       heads_per_rank=hpr, init_blocks=1, local_blocks=3)
        np.testing.assert_array_equal(mi.cpu().numpy(), oi)


def test_window_of_uniform_chunks_equals_the_decode_scorer():
    # a window whose requests all bring dql <= 8 tokens is a decode batch
    spec = W.DecodeSpec("d", batch=20, page_size=256, world_size=1, decode_query_len=4,
                        max_decode_query_len=8, init_blocks=2, local_blocks=4,
                        seq_range=(300, 20000))
    inp = W.make_decode_inputs(spec, seed=13)
    q, k, bt, sl = (inp.index_q.cuda(), inp.index_k.cuda(), inp.block_table.cuda(),
                    inp.seq_lens.cuda())
    cols = W.columns_for(spec, int(inp.seq_lens.max()))
    qo = torch.arange(0, 4 * 21, 4, dtype=torch.int32, device="cuda")
    gp, _ = _gpu_plane(q, k, bt, sl, qo, cols=cols, rank=0, world_size=1, page_size=256)
    dp = sentinel_plane(inp.T, cols)
    icp().icp_score(q, k, bt, sl, dp, rank=0, world_size=1, page_size=256, decode_query_len=4,
                    max_decode_query_len=8)
    torch.cuda.synchronize()
    assert torch.equal(gp.view(torch.int32), dp.view(torch.int32))


def test_benched_prefill_window_full_size():
    # the window bench.py --workload prefill times: B=4 requests, chunks of
    # 2048 tokens (T = 8192, 128 plan records), drawn on the GPU with seed 0
    from gpu_util import exact_selection_agrees
    from oracle.parallel import PlanePool
    spec = W.PREFILL
    inp = W.make_decode_inputs(spec, seed=0, device="cuda")
    q, k, bt, sl, nvp = (inp.index_q, inp.index_k, inp.block_table, inp.seq_lens,
                         inp.num_valid_pages)
    B, n = sl.shape[0], spec.decode_query_len
    T = B * n
    qo = torch.arange(0, (B + 1) * n, n, dtype=torch.int32, device="cuda")
    cols = W.columns_for(spec, int(sl.max()))
    errors = torch.zeros(1, dtype=torch.int32, device="cuda")
    gp, plan = _gpu_plane(q, k, bt, sl, qo, cols=cols, rank=0, world_size=1, page_size=128,
                          errors=errors)
    car = torch.zeros((1, T, 4, 32), dtype=torch.int32, device="cuda")
    icp().icp_prefill_select(gp, nvp, car, world_size=1, heads_per_rank=4,
                             init_blocks=spec.init_blocks, local_blocks=spec.local_blocks)
    out_s = torch.empty((T, 4, 16), device="cuda")
    out_i = torch.empty((T, 4, 16), dtype=torch.int32, device="cuda")
    icp().icp_prefill_merge(car, nvp, out_s, out_i, world_size=1, heads_per_rank=4,
                            init_blocks=spec.init_blocks, local_blocks=spec.local_blocks)
    torch.cuda.synchronize()
    assert int(errors.item()) == 0
    assert int(plan[0].item()) == T // 64                  # 128 records of 64 tokens
    g = gp.cpu().numpy()
    hn = nvp.cpu().numpy()
    # carrier rows and merged lists: every row, bit-exact on the GPU's plane
    ref = oracle.carrier(g, hn, world_size=1, heads_per_rank=4, init_blocks=spec.init_blocks,
                         local_blocks=spec.local_blocks)
    np.testing.assert_array_equal(car.cpu().numpy(), ref)
    ms, mi = oracle.merge_carrier(ref, hn, world_size=1, heads_per_rank=4,
                                  init_blocks=spec.init_blocks, local_blocks=spec.local_blocks)
    np.testing.assert_array_equal(out_i.cpu().numpy(), mi)
    np.testing.assert_array_equal(out_s.cpu().numpy().view(np.int32), ms.view(np.int32))
    # every token's plane row against the exact window, computed over the
    # host cores in slices of 128 tokens; a slice is scored as a window whose
    # request ends at its last token, so the request's columns past its
    # reach hold no visible key and are -inf (the whole-window reading)
    hq, hk, hbt, hsl, hqo = (t.cpu().numpy() for t in (q, k, bt, sl, qo))
    ex = np.full((T, 4, cols), np.nan)
    ab = np.full((T, 4, cols), np.nan)
    with PlanePool(hq, [hk], hbt, hsl) as pool:
        for b, j0, j1, p, a in pool.window_slices(hqo, cols=cols, page_size=128, piece=128):
            rows = slice(int(hqo[b]) + j0, int(hqo[b]) + j1)
            wreq = W.columns_for(spec, int(hsl[b]))
            reach = np.isnan(p) & (np.arange(cols) < wreq)[None, None, :]
            p[reach] = -np.inf
            a[reach] = 0.0
            ex[rows], ab[rows] = p, a
    assert not np.isnan(ex[:, :, 0]).any()
    assert_plane_matches(g, ex, ab, "prefill window, every token")
    checked, skipped = exact_selection_agrees(ex, ab, out_i.cpu().numpy(), hn, spec.init_blocks,
                                              spec.local_blocks)
    print(f"prefill window: exact selection checked on {checked} of {checked + skipped} rows")
    assert checked >= 0.97 * (checked + skipped)
