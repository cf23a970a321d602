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
