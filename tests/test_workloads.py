"""The seeded input recipe: determinism, shapes and stated distributions (CPU)."""
import numpy as np
import torch

import oracle
from sparse_attention_block_gb300 import workloads as W


def test_tiny_workload_shapes_and_determinism():
    a = W.make_decode_inputs(W.TINY, seed=0)
    b = W.make_decode_inputs(W.TINY, seed=0)
    assert torch.equal(a.index_k, b.index_k) and torch.equal(a.index_q, b.index_q)
    assert a.index_q.shape == (2, 4, 128) and a.index_k.shape == (64, 128, 128)
    assert a.seq_lens.tolist() == [1000, 2500]
    bt = a.block_table
    used = bt[bt >= 0]
    assert used.numel() == 8 + 20 and used.unique().numel() == 28   # a permutation
    assert a.num_valid_pages.tolist() == [8, 20]
    c = W.make_decode_inputs(W.TINY, seed=1)
    assert not torch.equal(a.index_k, c.index_k)


def test_queries_and_planted_keys_share_the_direction():
    inp = W.make_decode_inputs(W.BATCHED, seed=0, batch=6)
    q = inp.index_q.view(torch.float8_e4m3fn).float()
    proj = (q @ inp.u).mean().item()
    assert 1.2 < proj < 1.8                       # every query carries +1.5 u
    k = inp.index_k.view(torch.float8_e4m3fn).float()
    frac = inp.planted[:, :].float().sum() / ((inp.seq_lens + 127) // 128).sum()
    assert 0.0 < frac < 0.2
    # a planted block's keys project on u by about 1.5
    b, c = [int(x) for x in torch.nonzero(inp.planted)[0]]
    page = int(inp.block_table[b, c])
    assert 1.2 < (k[page] @ inp.u).mean().item() < 1.8


def test_sharded_workload_hands_out_contiguous_rows():
    inp = W.make_decode_inputs(W.SHARDED, seed=0, batch=2, seq_lens=[300, 700])
    assert len(inp.shards) == 4
    for r, s in enumerate(inp.shards):
        assert s.shape == (inp.index_k.shape[0], 32, 128)
        assert torch.equal(s, inp.index_k[:, 32 * r:32 * (r + 1)])


def test_select_plane_has_duplicates_and_valid_counts():
    plane, nvp = W.make_select_plane(T=4, K=1000)
    assert plane.shape == (4, 4, 1000)
    row = plane[0, 0].numpy()
    assert len(np.unique(row)) <= 1000 - 10
    assert int(nvp.min()) >= 1 and int(nvp.max()) <= 1000


def test_columns_for_matches_the_oracle():
    for spec in W.DECODE_SPECS.values():
        for L in [1, 128, 129, 1000, 262144]:
            want = max(4, oracle.columns_written(L, spec.page_size, spec.world_size))
            assert W.columns_for(spec, L) == want


def test_tiny_workload_sharded_merge_invariant_in_the_oracle():
    inp = W.make_decode_inputs(W.SHARDED, seed=0, batch=2, seq_lens=[3000, 5000])
    oracle.sharded_merge_equals_unsharded(
        inp.index_q.numpy(), inp.index_k.numpy(), inp.block_table.numpy(),
        inp.seq_lens.numpy(), inp.num_valid_pages.numpy(), world_size=4, page_size=128,
        decode_query_len=2, cols=W.columns_for(W.SHARDED, 5000), init_blocks=1, local_blocks=3)
