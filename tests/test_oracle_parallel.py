"""The oracle's chain as the CPU baseline runs it (oracle/parallel.py).

At world size 1 the owner merge receives one list per row, so the chain's
merged Top16 must equal the oracle's select on the request's plane.  The
worker pool must run the chain over every request it is given."""
import numpy as np

import oracle
from oracle.parallel import ParallelChain, decode_request
from sparse_attention_block_gb300 import workloads as W


def _tiny():
    spec = W.TINY
    inp = W.make_decode_inputs(spec, seed=0)
    cols = W.columns_for(spec, int(inp.seq_lens.max()))
    arrays = (inp.index_q.numpy(), [inp.index_k.numpy()], inp.block_table.numpy(),
              inp.seq_lens.numpy(), inp.num_valid_pages.numpy())
    params = dict(cols=cols, world_size=1, page_size=spec.page_size,
                  decode_query_len=spec.decode_query_len, init_blocks=spec.init_blocks,
                  local_blocks=spec.local_blocks)
    return spec, arrays, params


def test_chain_merge_equals_select_of_the_plane():
    spec, (q, shards, bt, sl, nvp), params = _tiny()
    dql = spec.decode_query_len
    for b in range(len(sl)):
        (ms, mi, missing), = decode_request(q, shards, bt, sl, nvp, b, **params)
        assert missing == 0
        plane, _ = oracle.score(q[b * dql:(b + 1) * dql], shards[0], bt[b:b + 1], sl[b:b + 1],
                                cols=params["cols"], rank=0, world_size=1,
                                page_size=spec.page_size, decode_query_len=dql, fill=-np.inf)
        ss, si = oracle.select(plane.astype(np.float32), nvp[b * dql:(b + 1) * dql],
                               init_blocks=spec.init_blocks, local_blocks=spec.local_blocks)
        assert np.array_equal(mi, si)
        assert np.array_equal(ms.view(np.int32), ss.view(np.int32))


def test_worker_pool_runs_the_chain_over_the_requests():
    _, arrays, params = _tiny()
    with ParallelChain(*arrays, params, workers=2) as pc:
        assert pc.workers == 2
        assert pc.time(range(len(arrays[3]))) > 0.0


def test_plane_pool_equals_the_oracle_over_the_whole_batch():
    from oracle.parallel import PlanePool
    spec = W.DecodeSpec("p", batch=5, page_size=256, world_size=1, decode_query_len=3,
                        max_decode_query_len=3, init_blocks=1, local_blocks=2,
                        seq_lens=(1, 300, 129, 700, 2500))
    inp = W.make_decode_inputs(spec, seed=3)
    q, k, bt, sl = (inp.index_q.numpy(), inp.index_k.numpy(), inp.block_table.numpy(),
                    inp.seq_lens.numpy())
    cols = W.columns_for(spec, 2500) + 4
    whole, whole_abs = oracle.score(q, k, bt, sl, cols=cols, rank=0, world_size=1,
                                    page_size=256, decode_query_len=3, fill=np.nan)
    with PlanePool(q, [k], bt, sl, workers=2) as pool:
        plane, absplane = pool.decode_plane(k=0, cols=cols, rank=0, world_size=1,
                                            page_size=256, decode_query_len=3)
    np.testing.assert_array_equal(plane, whole)
    np.testing.assert_array_equal(absplane, whole_abs)


def test_window_slices_equal_the_whole_window():
    # a slice of a chunk, scored as a window whose request ends at its last
    # token, gives the whole window's rows on the columns it writes; the
    # whole window's remaining columns of the request are -inf (no key at or
    # before those tokens' positions)
    from oracle.parallel import PlanePool
    seq_lens, chunks = [300, 1000, 2600], [40, 200, 150]
    spec = W.DecodeSpec("w", batch=3, page_size=128, world_size=1, decode_query_len=1,
                        max_decode_query_len=1, init_blocks=1, local_blocks=3,
                        seq_lens=tuple(seq_lens))
    inp = W.make_decode_inputs(spec, seed=6)
    qo = np.concatenate([[0], np.cumsum(chunks)]).astype(np.int32)
    T = int(qo[-1])
    rng = np.random.default_rng(6)
    q = rng.integers(0, 0x7F, size=(T, 4, 128), dtype=np.uint8)   # finite e4m3 codes
    k, bt, sl = inp.index_k.numpy(), inp.block_table.numpy(), inp.seq_lens.numpy()
    cols = W.columns_for(spec, max(seq_lens))
    whole, whole_abs = oracle.score_chunks(q, k, bt, sl, qo, cols=cols, rank=0, world_size=1,
                                           page_size=128)
    seen = np.zeros(T, bool)
    with PlanePool(q, [k], bt, sl, workers=2) as pool:
        for b, j0, j1, p, ab in pool.window_slices(qo, cols=cols, page_size=128, piece=64):
            rows = slice(qo[b] + j0, qo[b] + j1)
            w = ~np.isnan(p)
            np.testing.assert_array_equal(p[w], whole[rows][w])
            np.testing.assert_array_equal(ab[w], whole_abs[rows][w])
            rest = np.isnan(p) & ~np.isnan(whole[rows])
            assert np.all(np.isneginf(whole[rows][rest]))
            seen[rows] = True
    assert seen.all()
