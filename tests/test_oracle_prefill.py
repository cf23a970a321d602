"""Pins of the oracle's prefill window functions (CPU only).

The pages name the prefill chain of prepare_msa_icp_indexer
(prefill_window_plan, prefill_local, prefill_merge) without its own pages;
the reading is the decode plane with a per-request query length, Top16 lists
in flag-free 32-word carrier rows, and the decode merge rule.  The pins here
come from outside the oracle: a brute-force plane in numpy (fp8 decoded by
torch), the decode plane of one-token requests, hand-computed carrier
addresses, and the sharded-merge-equals-unsharded identity of a max
reduction.
"""
import numpy as np
import pytest
import torch

import oracle
from sparse_attention_block_gb300 import workloads as W


def _window(seq_lens, chunks, page_size=128, world_size=1, seed=0):
    """Seeded window: request b contributes its newest chunks[b] tokens."""
    spec = W.DecodeSpec("w", batch=len(seq_lens), page_size=page_size, world_size=world_size,
                        decode_query_len=1, max_decode_query_len=1, init_blocks=1,
                        local_blocks=2, seq_lens=tuple(seq_lens))
    inp = W.make_decode_inputs(spec, seed=seed)
    qo = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(qo[-1])
    g = torch.Generator().manual_seed(seed + 100)
    q = (0.5 * torch.randn((T, 4, 128), generator=g)).to(torch.float8_e4m3fn).view(torch.uint8)
    return inp, q.numpy(), qo


def _deq(u8):
    return torch.from_numpy(np.ascontiguousarray(u8)).view(torch.float8_e4m3fn).to(
        torch.float64).numpy()


def test_brute_force_plane_tiny_window():
    seq_lens, chunks = [300, 140], [5, 3]
    inp, q, qo = _window(seq_lens, chunks)
    cols = 4
    plane, _ = oracle.score_chunks(q, inp.index_k.numpy(), inp.block_table.numpy(),
                                   inp.seq_lens.numpy(), qo, cols=cols, rank=0, world_size=1,
                                   page_size=128)
    qd, kd = _deq(q), _deq(inp.index_k.numpy())
    bt = inp.block_table.numpy()
    for b, (L, n) in enumerate(zip(seq_lens, chunks)):
        width = (-(-L // 128) + 3) // 4 * 4
        for j in range(n):
            t, p = qo[b] + j, L - n + j
            for h in range(4):
                for c in range(cols):
                    if c >= width:
                        assert np.isnan(plane[t, h, c])
                        continue
                    best = -np.inf
                    for pos in range(c * 128, min((c + 1) * 128, L)):
                        if pos > p:
                            break
                        key = kd[bt[b, pos // 128], pos % 128]
                        best = max(best, float(np.dot(qd[t, h], key)))
                    assert plane[t, h, c] == best, (b, j, h, c)


def test_each_row_is_the_decode_row_of_a_one_token_request():
    seq_lens, chunks = [700, 1000, 129], [40, 17, 129]
    inp, q, qo = _window(seq_lens, chunks, seed=3)
    cols = 8
    plane, absplane = oracle.score_chunks(q, inp.index_k.numpy(), inp.block_table.numpy(),
                                          inp.seq_lens.numpy(), qo, cols=cols, rank=0,
                                          world_size=1, page_size=128)
    for b, (L, n) in enumerate(zip(seq_lens, chunks)):
        width = oracle.columns_written(L, 128, 1)
        for j in range(0, n, 7):
            t, p = int(qo[b]) + j, L - n + j
            one, one_abs = oracle.score(q[t:t + 1], inp.index_k.numpy(),
                                        inp.block_table.numpy()[b:b + 1],
                                        np.array([p + 1], np.int32), cols=cols, rank=0,
                                        world_size=1, page_size=128, decode_query_len=1)
            w1 = oracle.columns_written(p + 1, 128, 1)
            np.testing.assert_array_equal(plane[t, :, :w1], one[0, :, :w1])
            np.testing.assert_array_equal(absplane[t, :, :w1], one_abs[0, :, :w1])
            assert np.all(plane[t, :, w1:width] == -np.inf)
            assert np.all(np.isnan(plane[t, :, width:]))


def test_uniform_chunks_equal_the_decode_plane():
    seq_lens = [500, 260, 1024]
    inp, q, qo = _window(seq_lens, [6, 6, 6], seed=5)
    args = dict(cols=8, rank=0, world_size=1, page_size=128)
    a, _ = oracle.score_chunks(q, inp.index_k.numpy(), inp.block_table.numpy(),
                               inp.seq_lens.numpy(), qo, **args)
    d, _ = oracle.score(q, inp.index_k.numpy(), inp.block_table.numpy(), inp.seq_lens.numpy(),
                        decode_query_len=6, **args)
    np.testing.assert_array_equal(a, d)


def test_empty_chunks_and_bad_indptr():
    inp, q, qo = _window([300, 140, 50], [0, 4, 0], seed=7)
    plane, _ = oracle.score_chunks(q, inp.index_k.numpy(), inp.block_table.numpy(),
                                   inp.seq_lens.numpy(), qo, cols=4, rank=0, world_size=1,
                                   page_size=128)
    assert plane.shape == (4, 4, 4)
    bad = np.array([0, 2, 1, 4], np.int32)  # decreasing
    with pytest.raises(ValueError):
        oracle.score_chunks(q, inp.index_k.numpy(), inp.block_table.numpy(),
                            inp.seq_lens.numpy(), bad, cols=4, rank=0, world_size=1,
                            page_size=128)
    long_chunk = np.array([0, 0, 0, 51], np.int32)  # 51 tokens of a 50-token request
    with pytest.raises(ValueError):
        oracle.score_chunks(np.zeros((51, 4, 128), np.uint8), inp.index_k.numpy(),
                            inp.block_table.numpy(), inp.seq_lens.numpy(), long_chunk, cols=4,
                            rank=0, world_size=1, page_size=128)


def test_carrier_row_addresses_by_hand():
    T, K = 3, 40
    rng = np.random.default_rng(0)
    plane = rng.standard_normal((T, 4, K)).astype(np.float32)
    nvp = np.array([40, 10, 33], np.int32)
    car = oracle.carrier(plane, nvp, world_size=2, heads_per_rank=2, init_blocks=1,
                         local_blocks=2)
    s, i = oracle.select(plane, nvp, init_blocks=1, local_blocks=2)
    # head 3 of token 2 goes to owner 1, local head 1
    row = car[1, 2, 1]
    np.testing.assert_array_equal(row[16:], i[2, 3])
    np.testing.assert_array_equal(row[:16].view(np.float32), s[2, 3])
    # head 0 of token 0 goes to owner 0, local head 0
    np.testing.assert_array_equal(car[0, 0, 0, 16:], i[0, 0])


@pytest.mark.parametrize("ws", [2, 4])
def test_merged_shard_carriers_equal_the_unsharded_top16(ws):
    seq_lens, chunks = [900, 2000, 300], [12, 33, 7]
    inp, q, qo = _window(seq_lens, chunks, world_size=ws, seed=11)
    cols = oracle.columns_written(max(seq_lens), 128, 1)
    T = int(qo[-1])
    pos = np.concatenate([np.arange(L - n, L) for L, n in zip(seq_lens, chunks)])
    nvp = ((pos + 1 + 127) // 128).astype(np.int32)
    full, _ = oracle.score_chunks(q, inp.index_k.numpy(), inp.block_table.numpy(),
                                  inp.seq_lens.numpy(), qo, cols=cols, rank=0, world_size=1,
                                  page_size=128, fill=-np.inf)
    ref_s, ref_i = oracle.select(full.astype(np.float32), nvp, init_blocks=1, local_blocks=3)
    hpr = 4 // ws
    rp = 128 // ws
    cars = []
    for r in range(ws):
        shard = inp.index_k.numpy()[:, r * rp:(r + 1) * rp].copy()
        pl, _ = oracle.score_chunks(q, shard, inp.block_table.numpy(), inp.seq_lens.numpy(), qo,
                                    cols=cols, rank=r, world_size=ws, page_size=128,
                                    fill=-np.inf)
        cars.append(oracle.carrier(pl.astype(np.float32), nvp, world_size=ws,
                                   heads_per_rank=hpr, init_blocks=1, local_blocks=3))
    for owner in range(ws):
        received = np.stack([cars[s][owner] for s in range(ws)])
        ms, mi = oracle.merge_carrier(received, nvp, world_size=ws, heads_per_rank=hpr,
                                      init_blocks=1, local_blocks=3)
        heads = slice(owner * hpr, (owner + 1) * hpr)
        np.testing.assert_array_equal(mi, ref_i[:, heads])
        np.testing.assert_array_equal(ms.view(np.int32), ref_s[:, heads].view(np.int32))
        assert mi.shape == (T, hpr, 16)
