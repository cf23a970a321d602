"""Pins for the oracle's scoring step (CPU only).

Each test checks the oracle against something other than itself: torch's
float8_e4m3fn decoding, exact integer arithmetic, closed forms and
hand-built cases that follow the scorer page
(msa_icp_decode_index_score_sharded: column meaning, token position, write
coverage) and the block-score reading (max over visible keys).
"""
import math

import numpy as np
import pytest
import torch

import oracle

D = 128


def fp8(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8).numpy()


def torch_decode(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).float().double().numpy()


def test_e4m3_all_codes_match_torch():
    table = oracle.e4m3_table()
    ref = torch_decode(np.arange(256, dtype=np.uint8))
    nan_o, nan_r = np.isnan(table), np.isnan(ref)
    assert np.array_equal(nan_o, nan_r)
    assert set(np.nonzero(nan_o)[0].tolist()) == {0x7F, 0xFF}
    assert np.array_equal(table[~nan_o], ref[~nan_r])
    assert np.nanmax(table) == 448.0 and table[1] == 2.0 ** -9


def test_e4m3_format_landmarks():
    # exponent bias 7: 0x38 = 0.0111.000 = 1.0; 0x40 = 2.0; subnormal 0x04 = 4 * 2^-9
    assert oracle.e4m3_value(0x38) == 1.0
    assert oracle.e4m3_value(0x40) == 2.0
    assert oracle.e4m3_value(0xB8) == -1.0
    assert oracle.e4m3_value(0x04) == 4 * 2.0 ** -9
    assert oracle.e4m3_value(0x08) == 2.0 ** -6
    assert oracle.e4m3_value(0x80) == 0.0 and math.copysign(1, oracle.e4m3_value(0x80)) < 0


def _single_request(seq_len, page_size=128, world_size=1, dql=1, pool=None, seed=0,
                    q=None, k=None):
    rng = np.random.default_rng(seed)
    units = oracle.columns_with_keys(seq_len, page_size, world_size)
    npages = (seq_len + page_size - 1) // page_size
    pool = pool or npages
    bt = rng.permutation(pool)[:npages].astype(np.int32)[None, :]
    if q is None:
        q = fp8(rng.normal(0, 1, (dql, 4, D)).astype(np.float32))
    if k is None:
        k = fp8(rng.normal(0, 1, (pool, page_size // world_size, D)).astype(np.float32))
    return q, k, bt, units


def brute_force_plane(q, k_full, bt, seq_lens, dql, page_size, cols):
    """Exact integer brute force over unsharded B128 blocks: int dot of
    (value * 2^9) integers, masked by position, max per block."""
    qi = np.rint(torch_decode(q) * 512).astype(np.int64)          # [T,4,128]
    ki = np.rint(torch_decode(k_full) * 512).astype(np.int64)     # [pool, ps, 128]
    T = q.shape[0]
    out = np.full((T, 4, cols), np.nan)
    for b, L in enumerate(seq_lens):
        nb = (L + 127) // 128
        ncol = (nb + 3) // 4 * 4
        keys = np.stack([ki[bt[b, pos // page_size], pos % page_size] for pos in range(L)])
        for j in range(dql):
            t = b * dql + j
            p = L - dql + j
            dots = qi[t] @ keys.T  # [4, L], exact
            for c in range(ncol):
                lo, hi = c * 128, min((c + 1) * 128, p + 1)
                if hi <= lo:
                    out[t, :, c] = -np.inf
                else:
                    out[t, :, c] = dots[:, lo:hi].max(axis=1) / 2.0 ** 18
    return out


@pytest.mark.parametrize("page_size", [128, 256])
@pytest.mark.parametrize("dql", [1, 3])
def test_exact_against_integer_brute_force(page_size, dql):
    rng = np.random.default_rng(7)
    seq_lens = np.array([5, 300, 129], np.int32)
    B = len(seq_lens)
    npages = (seq_lens + page_size - 1) // page_size
    pool = int(npages.sum()) + 3
    perm = rng.permutation(pool).astype(np.int32)
    bt = np.full((B, npages.max()), -1, np.int32)
    o = 0
    for b in range(B):
        bt[b, :npages[b]] = perm[o:o + npages[b]]
        o += npages[b]
    q = fp8(rng.normal(0, 2, (B * dql, 4, D)).astype(np.float32))
    k = fp8(rng.normal(0, 2, (pool, page_size, D)).astype(np.float32))
    cols = 12
    plane, _ = oracle.score(q, k, bt, seq_lens, cols=cols, rank=0, world_size=1,
                            page_size=page_size, decode_query_len=dql)
    ref = brute_force_plane(q, k, bt, seq_lens, dql, page_size, cols)
    written = ~np.isnan(ref)
    assert np.array_equal(np.isnan(plane), np.isnan(ref))
    assert np.array_equal(plane[written], ref[written])


def test_closed_form_constant_vectors():
    # q = a everywhere, k = b everywhere -> every visible dot is 128 a b
    a, bval = 0.5, -3.0
    q = fp8(np.full((1, 4, D), a, np.float32))
    k = fp8(np.full((2, 128, D), bval, np.float32))
    bt = np.array([[1, 0]], np.int32)
    plane, absplane = oracle.score(q, k, bt, np.array([200], np.int32), cols=4, rank=0,
                                   world_size=1, page_size=128, decode_query_len=1)
    assert np.all(plane[0, :, 0] == 128 * a * bval)
    assert np.all(plane[0, :, 1] == 128 * a * bval)
    assert np.all(np.isneginf(plane[0, :, 2:4]))
    assert np.all(absplane[0, :, :2] == 128 * abs(a * bval))


def test_one_hot_query_reads_one_dimension():
    # q = e_5, so the score of a key is its 5th component; block max picks the largest
    q = np.zeros((1, 4, D), np.uint8)
    q[0, :, 5] = fp8([1.0])[0]
    k = np.zeros((1, 128, D), np.uint8)
    vals = [0.25, -2.0, 7.0, 3.5]
    for r, v in enumerate(vals):
        k[0, 10 * r, 5] = fp8([v])[0]
    bt = np.array([[0]], np.int32)
    plane, _ = oracle.score(q, k, bt, np.array([128], np.int32), cols=4, rank=0, world_size=1,
                            page_size=128, decode_query_len=1)
    assert np.all(plane[0, :, 0] == 7.0)


def test_mask_excludes_keys_after_the_token():
    # seq_len 100, dql 2: tokens sit at positions 98 and 99.  A huge key at
    # position 99 is visible to token 1 only.
    q = np.full((2, 4, D), fp8([0.5])[0], np.uint8)
    k = np.zeros((1, 128, D), np.uint8)
    k[0, 99, :] = fp8([448.0])[0]
    k[0, 98, :] = fp8([1.0])[0]
    bt = np.array([[0]], np.int32)
    plane, _ = oracle.score(q, k, bt, np.array([100], np.int32), cols=4, rank=0, world_size=1,
                            page_size=128, decode_query_len=2)
    assert np.all(plane[0, :, 0] == 128 * 0.5 * 1.0)
    assert np.all(plane[1, :, 0] == 128 * 0.5 * 448.0)


def test_keys_beyond_seq_len_never_count():
    q = np.full((1, 4, D), fp8([1.0])[0], np.uint8)
    k = np.zeros((1, 128, D), np.uint8)
    k[0, 50, :] = fp8([2.0])[0]   # position 50 >= seq_len 40
    bt = np.array([[0]], np.int32)
    plane, _ = oracle.score(q, k, bt, np.array([40], np.int32), cols=4, rank=0, world_size=1,
                            page_size=128, decode_query_len=1)
    assert np.all(plane[0, :, 0] == 0.0)


@pytest.mark.parametrize("page_size,ws,expect_cols", [
    (128, 1, [4, 4, 8, 12]), (128, 4, [4, 4, 8, 12]), (256, 2, [4, 4, 4, 8]),
    (256, 1, [4, 4, 8, 12]), (256, 4, [4, 4, 4, 8])])
def test_written_columns_round_up_to_four(page_size, ws, expect_cols):
    lens = [1, 128, 640, 1200]
    got = [oracle.columns_written(L, page_size, ws) for L in lens]
    assert got == expect_cols
    assert oracle.columns_written(0, page_size, ws) == 0


def test_other_columns_are_not_written():
    q, k, bt, units = _single_request(300)
    plane, _ = oracle.score(q, k, bt, np.array([300], np.int32), cols=16, rank=0, world_size=1,
                            page_size=128, decode_query_len=1, fill=12345.0)
    assert units == 3
    assert np.all(np.isfinite(plane[:, :, :3]))
    assert np.all(np.isneginf(plane[:, :, 3]))          # padding column inside the round-up
    assert np.all(plane[:, :, 4:] == 12345.0)           # untouched


def test_token_with_no_visible_key_gets_minus_inf():
    # dql 3 but seq_len 2: token 0 sits at position -1 and sees nothing
    q, k, bt, _ = _single_request(2, dql=3)
    plane, _ = oracle.score(q, k, bt, np.array([2], np.int32), cols=4, rank=0, world_size=1,
                            page_size=128, decode_query_len=3)
    assert np.all(np.isneginf(plane[0, :, 0]))
    assert np.all(np.isfinite(plane[1, :, 0])) and np.all(np.isfinite(plane[2, :, 0]))


def _hot_key_layout(page_size, ws, hot_pos, seq_len):
    """One hot key (all 4.0) among zeros at token position hot_pos; returns the
    per-rank planes for a single page-table request."""
    npages = (seq_len + page_size - 1) // page_size
    full = np.zeros((npages, page_size, D), np.uint8)
    full[hot_pos // page_size, hot_pos % page_size, :] = fp8([4.0])[0]
    q = np.full((1, 4, D), fp8([1.0])[0], np.uint8)
    bt = np.arange(npages, dtype=np.int32)[None, :]
    rp = page_size // ws
    out = []
    for r in range(ws):
        shard = np.ascontiguousarray(full[:, r * rp:(r + 1) * rp])
        plane, _ = oracle.score(q, shard, bt, np.array([seq_len], np.int32), cols=16, rank=r,
                                world_size=ws, page_size=page_size, decode_query_len=1,
                                fill=np.nan)
        out.append(plane[0, 0])
    return out


def test_p128_sharded_rows_belong_to_the_global_block():
    # P128 ws 4: rank r holds rows [32 r, 32 r + 32) of every page; column = global block
    hot = 3 * 128 + 70        # block 3, row 70 -> rank 2
    planes = _hot_key_layout(128, 4, hot, 1000)
    for r, p in enumerate(planes):
        assert (p[3] == 128 * 4.0) == (r == 2)


@pytest.mark.parametrize("ws", [2, 4])
def test_p256_sharded_column_is_the_local_page(ws):
    # P256: column c = local page c; rank r's rows lie in global block 2c + r*2//ws
    hot = 2 * 256 + 130       # page 2, row 130 -> global block 5
    planes = _hot_key_layout(256, ws, hot, 1500)
    rp = 256 // ws
    owner = 130 // rp
    for r, p in enumerate(planes):
        assert (p[2] == 128 * 4.0) == (r == owner)
        if r == owner:
            assert 2 * 2 + r * 2 // ws == hot // 128


def test_p256_unsharded_has_one_column_per_b128_block():
    hot = 2 * 256 + 130       # global block 5
    (p,) = _hot_key_layout(256, 1, hot, 1500)
    assert p[5] == 128 * 4.0
    assert np.all(p[[0, 1, 2, 3, 4, 6, 7, 8, 9, 10, 11]] == 0.0)


def test_block_table_entries_past_the_request_are_never_read():
    q, k, bt, _ = _single_request(200, pool=4)
    bt = np.concatenate([bt, np.full((1, 5), -7, np.int32)], axis=1)
    oracle.score(q, k, bt, np.array([200], np.int32), cols=4, rank=0, world_size=1,
                 page_size=128, decode_query_len=1)
    bad = bt.copy()
    bad[0, 1] = 99
    with pytest.raises(ValueError):
        oracle.score(q, k, bad, np.array([200], np.int32), cols=4, rank=0, world_size=1,
                     page_size=128, decode_query_len=1)


def test_nan_codes_are_rejected():
    q, k, bt, _ = _single_request(10)
    k = k.copy()
    k[bt[0, 0], 3, 0] = 0x7F
    with pytest.raises(ValueError):
        oracle.score(q, k, bt, np.array([10], np.int32), cols=4, rank=0, world_size=1,
                     page_size=128, decode_query_len=1)


def test_request_wider_than_the_plane_is_rejected():
    q, k, bt, _ = _single_request(1000)
    with pytest.raises(ValueError):
        oracle.score(q, k, bt, np.array([1000], np.int32), cols=4, rank=0, world_size=1,
                     page_size=128, decode_query_len=1)
