"""Pins for the oracle's Top16 select, receive-row publish and owner merge (CPU).

The select is checked with an independent predicate (what a correct Top16
with forced blocks must satisfy) on random rows, and with hand-built rows;
the receive-row address with hand-computed values from the formula on the
msa_icp_topk_select_publish page; the merge with the invariant that merging
the shard lists equals the unsharded Top16 (exact under the max reduction).
"""
import numpy as np
import pytest
import torch

import oracle

NEG = -np.inf


def check_top16(ids_in, scores_in, nvp, init, local, out_s, out_i):
    """Independent validity predicate for one selected row."""
    ids_in = np.asarray(ids_in)
    sc = np.asarray(scores_in, np.float32).astype(np.float64)
    valid = (ids_in >= 0) & (ids_in < nvp)
    V = dict(zip(ids_in[valid].tolist(), sc[valid].tolist()))
    real = out_i[out_i != -1]
    n = len(real)
    # real ids first, ascending and unique; padding (-1, -inf) at the tail
    assert np.all(out_i[:n] != -1) and np.all(out_i[n:] == -1)
    assert np.all(np.isneginf(out_s[n:]))
    assert np.all(np.diff(real) > 0)
    assert n == min(16, len(V))
    for i, s in zip(real.tolist(), out_s[:n].tolist()):
        assert i in V and np.float32(V[i]) == np.float32(s)
    if nvp <= 16:
        assert set(real.tolist()) == set(V)
        return
    forced = {i for i in V if i < init or i >= nvp - local}
    assert forced <= set(real.tolist())
    chosen = set(real.tolist()) - forced
    rest = set(V) - forced - chosen

    def better(a, b):
        return V[a] > V[b] or (V[a] == V[b] and a < b)
    for a in chosen:
        for b in rest:
            assert better(a, b), (a, b)


@pytest.mark.parametrize("seed", range(6))
def test_random_rows_satisfy_the_top16_predicate(seed):
    rng = np.random.default_rng(seed)
    K = int(rng.integers(1, 300))
    scores = rng.normal(0, 1, K).astype(np.float32)
    # ties: copy some values around
    for _ in range(K // 5):
        scores[rng.integers(K)] = scores[rng.integers(K)]
    if seed % 2:
        scores[rng.integers(K, size=3)] = NEG
    ids = np.arange(K, dtype=np.int32)
    for nvp in [1, 5, 16, 17, K // 2 + 1, K, K + 10]:
        for init, local in [(0, 0), (1, 2), (4, 8), (16, 0), (0, 16), (3, 13)]:
            s, i = oracle.select_pairs(ids, scores, nvp, init, local)
            check_top16(ids, scores, nvp, init, local, s, i)


def test_all_equal_scores_give_the_lowest_free_ids():
    ids = np.arange(100, dtype=np.int32)
    sc = np.full(100, 2.5, np.float32)
    s, i = oracle.select_pairs(ids, sc, 100, 1, 2)
    # forced: 0 (begin) and 98, 99 (end); the 13 free slots go to ids 1..13
    assert i.tolist() == list(range(14)) + [98, 99]
    assert np.all(s == 2.5)


def test_few_valid_pages_pad_with_minus_one():
    ids = np.arange(40, dtype=np.int32)
    sc = np.linspace(-1, 1, 40).astype(np.float32)
    s, i = oracle.select_pairs(ids, sc, 5, 1, 2)
    assert i.tolist() == [0, 1, 2, 3, 4] + [-1] * 11
    assert np.all(np.isneginf(s[5:]))
    assert np.array_equal(s[:5], sc[:5])


def test_forced_blocks_kept_even_with_the_worst_scores():
    K = 64
    ids = np.arange(K, dtype=np.int32)
    sc = np.arange(K, dtype=np.float32)        # id 0 is the worst, 63 the best
    sc[60] = -1000.0                           # forced end block with a terrible score
    s, i = oracle.select_pairs(ids, sc, 61, 2, 3)   # forced: 0, 1, 58, 59, 60
    got = i.tolist()
    assert {0, 1, 58, 59, 60} <= set(got)
    free = [x for x in got if x not in (0, 1, 58, 59, 60)]
    assert free == list(range(47, 58))          # the 11 best ids below nvp - local
    assert s[got.index(60)] == -1000.0


def test_tie_at_the_cut_goes_to_the_lower_id():
    ids = np.arange(40, dtype=np.int32)
    sc = np.zeros(40, np.float32)
    sc[:14] = 5.0
    sc[[20, 25, 30]] = 1.0                     # 2 free slots left for three tied ids
    s, i = oracle.select_pairs(ids, sc, 40, 0, 0)
    assert i.tolist() == list(range(14)) + [20, 25]


def test_signed_zeros_tie_by_id():
    ids = np.array([7, 3], np.int32)
    sc = np.array([0.0, -0.0], np.float32)
    s, i = oracle.select_pairs(np.concatenate([ids, np.arange(10, 40, dtype=np.int32)]),
                               np.concatenate([sc, np.full(30, -1.0, np.float32)]), 40, 0, 0)
    assert 3 in i and 7 in i


def test_minus_inf_scores_are_selectable_but_rank_last():
    ids = np.arange(30, dtype=np.int32)
    sc = np.full(30, NEG, np.float32)
    sc[[4, 9]] = 1.0
    s, i = oracle.select_pairs(ids, sc, 30, 0, 0)
    assert i.tolist() == sorted([4, 9] + [x for x in range(30) if x not in (4, 9)][:14])


def test_plane_select_uses_scale_and_offset():
    plane = np.zeros((1, 4, 10), np.float32)
    plane[0, :, 3] = 9.0
    nvp = np.array([40], np.int32)
    s, i = oracle.select(plane, nvp, init_blocks=0, local_blocks=0, index_scale=2,
                         index_offset=1)
    # columns map to ids 1,3,...,19; all valid; 10 real entries
    assert i[0, 0].tolist() == [1, 3, 5, 7, 9, 11, 13, 15, 17, 19] + [-1] * 6
    assert s[0, 0, 3] == 9.0


# --------------------------------------------------------------------------
# receive rows
# --------------------------------------------------------------------------
def test_recv_row_formula_hand_values():
    # ((slot*ws + rank)*hpr + h%hpr)*capacity + t
    assert oracle.recv_row(1, 2, 4, 1, 3, 64, 5) == ((1 * 4 + 2) * 1 + 0) * 64 + 5 == 389
    assert oracle.recv_row(2, 1, 2, 2, 3, 10, 7) == ((2 * 2 + 1) * 2 + 1) * 10 + 7 == 117
    assert oracle.recv_row(0, 0, 1, 4, 2, 8, 0) == 16


def _tiny_plane(T, K, seed):
    rng = np.random.default_rng(seed)
    return rng.normal(0, 1, (T, 4, K)).astype(np.float32)


def test_publish_writes_every_row_with_flag_and_layout():
    T, K, ws, hpr, cap = 3, 40, 2, 2, 4
    plane = _tiny_plane(T, K, 1)
    nvp = np.array([3, 40, 25], np.int32)   # token 0 is mostly padding
    recv = [np.zeros((oracle.recv_rows_per_owner(ws, hpr, cap), 33), np.int32)
            for _ in range(ws)]
    busy = oracle.publish(plane, nvp, recv, slot=2, rank=1, world_size=ws, heads_per_rank=hpr,
                          capacity=cap, force_begin_blocks=1, force_end_blocks=2)
    assert busy == 0
    ref_s, ref_i = oracle.select(plane, nvp, init_blocks=1, local_blocks=2)
    written = 0
    for t in range(T):
        for h in range(4):
            row = recv[h // hpr][oracle.recv_row(2, 1, ws, hpr, h, cap, t)]
            assert row[32] == 1
            assert np.array_equal(row[:16].view(np.float32).view(np.int32),
                                  ref_s[t, h].view(np.int32))
            assert np.array_equal(row[16:32], ref_i[t, h])
            written += 1
    assert written == T * 4
    total_flags = sum(int(r[:, 32].sum()) for r in recv)
    assert total_flags == T * 4


def test_publish_leaves_a_busy_row_alone_and_counts_it():
    T, K, ws, hpr, cap = 2, 20, 1, 4, 2
    plane = _tiny_plane(T, K, 2)
    nvp = np.array([20, 20], np.int32)
    recv = [np.zeros((oracle.recv_rows_per_owner(ws, hpr, cap), 33), np.int32)]
    r = oracle.recv_row(0, 0, ws, hpr, 2, cap, 1)
    recv[0][r, :] = 77
    recv[0][r, 32] = 1
    busy = oracle.publish(plane, nvp, recv, slot=0, rank=0, world_size=ws, heads_per_rank=hpr,
                          capacity=cap, force_begin_blocks=0, force_end_blocks=0)
    assert busy == 1
    assert np.all(recv[0][r, :32] == 77)


def test_merge_counts_missing_sources_and_clears_flags():
    T, K, ws, hpr, cap = 2, 30, 2, 2, 2
    planes = [_tiny_plane(T, K, 10 + r) for r in range(ws)]
    nvp = np.array([30, 30], np.int32)
    recv = [np.zeros((oracle.recv_rows_per_owner(ws, hpr, cap), 33), np.int32)
            for _ in range(ws)]
    oracle.publish(planes[0], nvp, recv, slot=1, rank=0, world_size=ws, heads_per_rank=hpr,
                   capacity=cap, force_begin_blocks=1, force_end_blocks=1)
    s, i, missing = oracle.merge(recv[0], nvp, T=T, slot=1, owner=0, world_size=ws,
                                 heads_per_rank=hpr, capacity=cap, init_blocks=1,
                                 local_blocks=1)
    assert missing == T * hpr          # rank 1 never published
    assert np.all(recv[0][:, 32] == 0)  # rank 0's rows are free again
    ref_s, ref_i = oracle.select(planes[0], nvp, init_blocks=1, local_blocks=1)
    assert np.array_equal(i, ref_i[:, :hpr])


def test_merge_takes_the_max_score_per_id():
    T, ws, hpr, cap = 1, 2, 2, 1
    recv = np.zeros((oracle.recv_rows_per_owner(ws, hpr, cap), 33), np.int32)
    for src, vals in enumerate([[1.0, 5.0], [4.0, 2.0]]):
        row = recv[oracle.recv_row(0, src, ws, hpr, 0, cap, 0)]
        sc = np.full(16, NEG, np.float32)
        ids = np.full(16, -1, np.int32)
        sc[:2], ids[:2] = vals, [10, 20]
        row[:16] = sc.view(np.int32)
        row[16:32] = ids
        row[32] = 1
        row2 = recv[oracle.recv_row(0, src, ws, hpr, 1, cap, 0)]
        row2[16:32] = -1
        row2[:16] = np.full(16, NEG, np.float32).view(np.int32)
        row2[32] = 1
    s, i, missing = oracle.merge(recv, np.array([100], np.int32), T=1, slot=0, owner=0,
                                 world_size=ws, heads_per_rank=hpr, capacity=cap,
                                 init_blocks=0, local_blocks=0)
    assert missing == 0
    assert i[0, 0, :2].tolist() == [10, 20] and s[0, 0, :2].tolist() == [4.0, 5.0]
    assert np.all(i[0, 1] == -1)


# --------------------------------------------------------------------------
# the sharded-merge invariant
# --------------------------------------------------------------------------
def _random_case(seed, page_size, B, lo, hi, dql, planted_scale=1.5):
    rng = np.random.default_rng(seed)
    seq_lens = rng.integers(lo, hi + 1, B).astype(np.int32)
    npages = (seq_lens + page_size - 1) // page_size
    pool = int(npages.sum())
    perm = rng.permutation(pool).astype(np.int32)
    bt = np.full((B, npages.max()), -1, np.int32)
    o = 0
    for b in range(B):
        bt[b, :npages[b]] = perm[o:o + npages[b]]
        o += npages[b]
    u = rng.normal(0, 1, 128)
    u /= np.linalg.norm(u)
    q = 0.5 * rng.normal(0, 1, (B * dql, 4, 128)) + planted_scale * u
    k = 0.5 * rng.normal(0, 1, (pool, page_size, 128))
    k[rng.random((pool,)) < 0.1] += planted_scale * u
    to8 = lambda x: torch.from_numpy(x.astype(np.float32)).to(torch.float8_e4m3fn).view(
        torch.uint8).numpy()
    j = np.arange(dql)
    pos = (seq_lens[:, None] - dql + j[None, :]).reshape(-1)
    nvp = ((pos + 1 + 127) // 128).astype(np.int32)
    return to8(q), to8(k), bt, seq_lens, nvp


@pytest.mark.parametrize("page_size,ws", [(128, 2), (128, 4), (256, 2), (256, 4)])
@pytest.mark.parametrize("seed", [0, 1])
def test_sharded_merge_equals_unsharded(page_size, ws, seed):
    dql = 2
    q, k, bt, sl, nvp = _random_case(seed, page_size, B=3, lo=200, hi=3000, dql=dql)
    unit = 128 if page_size == 128 else 256
    cols = ((int(sl.max()) + unit - 1) // unit + 3) // 4 * 4
    for init, local in [(1, 2), (4, 8), (0, 0)]:
        oracle.sharded_merge_equals_unsharded(
            q, k, bt, sl, nvp, world_size=ws, page_size=page_size, decode_query_len=dql,
            cols=cols, init_blocks=init, local_blocks=local, slot=seed % 3)


def test_a_wrong_merge_rule_would_break_the_invariant():
    # Guard that the invariant is sensitive: summing instead of taking the max
    # per id over shards gives a different Top16 on the same case.
    q, k, bt, sl, nvp = _random_case(3, 128, B=2, lo=4000, hi=6000, dql=1)
    ws, rp = 4, 32
    cols = ((int(sl.max()) + 127) // 128 + 3) // 4 * 4
    planes = []
    for r in range(ws):
        shard = np.ascontiguousarray(k[:, r * rp:(r + 1) * rp])
        p, _ = oracle.score(q, shard, bt, sl, cols=cols, rank=r, world_size=ws, page_size=128,
                            decode_query_len=1, fill=-np.inf)
        planes.append(p)
    full, _ = oracle.score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=128,
                           decode_query_len=1, fill=-np.inf)
    assert np.array_equal(np.maximum.reduce(planes), full)
    with np.errstate(invalid="ignore"):
        summed = np.where(np.isneginf(full), -np.inf, sum(np.where(np.isneginf(p), 0, p)
                                                           for p in planes))
    s1, i1 = oracle.select(full.astype(np.float32), nvp, init_blocks=1, local_blocks=2)
    s2, i2 = oracle.select(summed.astype(np.float32), nvp, init_blocks=1, local_blocks=2)
    assert not np.array_equal(i1, i2)
