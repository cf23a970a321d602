"""Pins for the oracle's tagged receive rows (msa_icp_topk_select_publish:
tagged rows are 32 int64 words of generation << 32 | word; generations are
per-(slot, head, token) publish counters, zeroed once)."""
import numpy as np

import oracle
from test_oracle_select_merge import _random_case


def _plane(T, K, seed):
    return np.random.default_rng(seed).normal(0, 1, (T, 4, K)).astype(np.float32)


def test_tagged_words_carry_the_legacy_row_and_the_generation():
    T, K, ws, hpr, cap = 3, 50, 2, 2, 4
    plane = _plane(T, K, 5)
    nvp = np.array([50, 9, 30], np.int32)
    legacy = [np.zeros((oracle.recv_rows_per_owner(ws, hpr, cap), 33), np.int32) for _ in range(ws)]
    oracle.publish(plane, nvp, legacy, slot=1, rank=1, world_size=ws, heads_per_rank=hpr,
                   capacity=cap, force_begin_blocks=1, force_end_blocks=2)
    tagged = [np.zeros((oracle.recv_rows_per_owner(ws, hpr, cap), 32), np.int64) for _ in range(ws)]
    gens = np.zeros((3, ws * hpr, cap), np.int32)
    for step in range(3):
        oracle.publish_tagged(plane, nvp, tagged, gens, slot=1, rank=1, world_size=ws,
                              heads_per_rank=hpr, capacity=cap, force_begin_blocks=1,
                              force_end_blocks=2)
        for t in range(T):
            for h in range(4):
                r = oracle.recv_row(1, 1, ws, hpr, h, cap, t)
                words = tagged[h // hpr][r].view(np.uint64)
                assert np.all((words >> np.uint64(32)) == step + 1)
                low = (words & np.uint64(0xFFFFFFFF)).astype(np.uint32).view(np.int32)
                assert np.array_equal(low, legacy[h // hpr][r, :32])
    assert np.all(gens[1, :, :T] == 3) and np.all(gens[0] == 0) and np.all(gens[1, :, T:] == 0)


def test_tagged_merge_equals_legacy_merge_and_reports_stale_rows():
    T, K, ws, hpr, cap = 2, 40, 2, 2, 2
    planes = [_plane(T, K, 20 + r) for r in range(ws)]
    nvp = np.array([40, 40], np.int32)
    legacy = [np.zeros((oracle.recv_rows_per_owner(ws, hpr, cap), 33), np.int32) for _ in range(ws)]
    tagged = [np.zeros((oracle.recv_rows_per_owner(ws, hpr, cap), 32), np.int64) for _ in range(ws)]
    gens = [np.zeros((3, 4, cap), np.int32) for _ in range(ws)]
    expected = [np.zeros((3, ws, hpr, cap), np.int32) for _ in range(ws)]
    for r in range(ws):
        oracle.publish(planes[r], nvp, legacy, slot=0, rank=r, world_size=ws, heads_per_rank=hpr,
                       capacity=cap, force_begin_blocks=1, force_end_blocks=1)
        oracle.publish_tagged(planes[r], nvp, tagged, gens[r], slot=0, rank=r, world_size=ws,
                              heads_per_rank=hpr, capacity=cap, force_begin_blocks=1,
                              force_end_blocks=1)
    for owner in range(ws):
        ls, li, lm = oracle.merge(legacy[owner], nvp, T=T, slot=0, owner=owner, world_size=ws,
                                  heads_per_rank=hpr, capacity=cap, init_blocks=1, local_blocks=1)
        ts, ti, tm = oracle.merge_tagged(tagged[owner], expected[owner], nvp, T=T, slot=0,
                                         world_size=ws, heads_per_rank=hpr, capacity=cap,
                                         init_blocks=1, local_blocks=1)
        assert lm == tm == 0
        assert np.array_equal(li, ti) and np.array_equal(ls.view(np.int32), ts.view(np.int32))
    # a second merge without a new publish finds stale generations everywhere
    _, _, missing = oracle.merge_tagged(tagged[0], expected[0], nvp, T=T, slot=0, world_size=ws,
                                        heads_per_rank=hpr, capacity=cap, init_blocks=1,
                                        local_blocks=1)
    assert missing == T * hpr * ws
    assert np.all(expected[0][0, :, :, :T] == 2)


def test_tagged_sharded_merge_equals_unsharded():
    for page_size, ws in [(128, 4), (256, 2)]:
        q, k, bt, sl, nvp = _random_case(9, page_size, B=3, lo=500, hi=6000, dql=2)
        hpr, T = 4 // ws, len(sl) * 2
        unit = 128 if page_size == 128 else 256
        cols = ((int(sl.max()) + unit - 1) // unit + 3) // 4 * 4
        full_cols = cols if page_size == 128 else 2 * cols
        full, _ = oracle.score(q, k, bt, sl, cols=full_cols, rank=0, world_size=1,
                               page_size=page_size, decode_query_len=2, fill=-np.inf)
        ref_s, ref_i = oracle.select(full.astype(np.float32), nvp, init_blocks=2, local_blocks=3)
        tagged = [np.zeros((oracle.recv_rows_per_owner(ws, hpr, T), 32), np.int64)
                  for _ in range(ws)]
        rp = page_size // ws
        for rank in range(ws):
            shard = np.ascontiguousarray(k[:, rank * rp:(rank + 1) * rp])
            plane, _ = oracle.score(q, shard, bt, sl, cols=cols, rank=rank, world_size=ws,
                                    page_size=page_size, decode_query_len=2, fill=-np.inf)
            scale, off = (1, 0) if page_size == 128 else (2, rank * 2 // ws)
            gens = np.zeros((3, 4, T), np.int32)
            oracle.publish_tagged(plane.astype(np.float32), nvp, tagged, gens, slot=2, rank=rank,
                                  world_size=ws, heads_per_rank=hpr, capacity=T,
                                  force_begin_blocks=2, force_end_blocks=3, index_scale=scale,
                                  index_offset=off)
        for owner in range(ws):
            exp = np.zeros((3, ws, hpr, T), np.int32)
            s, i, missing = oracle.merge_tagged(tagged[owner], exp, nvp, T=T, slot=2,
                                                world_size=ws, heads_per_rank=hpr, capacity=T,
                                                init_blocks=2, local_blocks=3)
            assert missing == 0
            assert np.array_equal(i, ref_i[:, owner * hpr:(owner + 1) * hpr])
            assert np.array_equal(s.view(np.int32),
                                  ref_s[:, owner * hpr:(owner + 1) * hpr].view(np.int32))
