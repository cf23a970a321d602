"""The N > 1 path of bench.py on CPU with gloo (world size 2): timing is the
maximum over ranks, every rank runs its own batch (no data-path collective),
and only rank 0 prints a JSON line."""
import json
import os
import socket
import subprocess
import sys

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench
    d = bench.init_dist(world, "gloo")
    got = bench.max_over_ranks(d, 10.0 + rank, torch.device("cpu"))
    bench.barrier(d)
    out[rank] = got
    dist.destroy_process_group()


def test_max_over_ranks_with_gloo():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] == 11.0 and out[1] == 11.0


def test_reference_arm_under_torchrun_prints_once():
    port = _free_port()
    env = dict(os.environ, ICP_REF_STEP_SECONDS="0.05", CUDA_VISIBLE_DEVICES="")
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--workload", "tiny", "--gpus", "2", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["n_gpus"] == 2 and d["value"] > 0
    assert d["cpu_baseline"]["kind"] == "oracle"


def test_workloads_differ_per_rank_seed():
    from sparse_attention_block_gb300 import workloads as W
    a = W.make_decode_inputs(W.TINY, seed=0)
    b = W.make_decode_inputs(W.TINY, seed=1)
    assert not torch.equal(a.index_k, b.index_k)


def _prefill_exchange_worker(rank, world, port, out):
    """One prefill window on a world_size-2 key shard: oracle plane and
    carrier on this rank, the caller's one exchange per layer as an
    equal-split all_to_all of the carrier, then this owner's merge."""
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    import numpy as np
    import oracle
    from test_oracle_prefill import _window
    dist.init_process_group("gloo", rank=rank, world_size=world)
    seq_lens, chunks = [900, 2000, 300], [12, 33, 7]
    inp, q, qo = _window(seq_lens, chunks, world_size=world, seed=31)
    pos = np.concatenate([np.arange(L - n, L) for L, n in zip(seq_lens, chunks)])
    nvp = ((pos + 1 + 127) // 128).astype(np.int32)
    cols = oracle.columns_written(max(seq_lens), 128, 1)
    rp, hpr = 128 // world, 4 // world
    shard = inp.index_k.numpy()[:, rank * rp:(rank + 1) * rp].copy()
    plane, _ = oracle.score_chunks(q, shard, inp.block_table.numpy(), inp.seq_lens.numpy(), qo,
                                   cols=cols, rank=rank, world_size=world, page_size=128,
                                   fill=-np.inf)
    car = oracle.carrier(plane.astype(np.float32), nvp, world_size=world, heads_per_rank=hpr,
                         init_blocks=1, local_blocks=3)
    send = torch.from_numpy(car).contiguous()          # block o is bound for owner o
    recv = torch.empty_like(send)                      # block s comes from rank s
    dist.all_to_all_single(recv, send)
    ms, mi = oracle.merge_carrier(recv.numpy(), nvp, world_size=world, heads_per_rank=hpr,
                                  init_blocks=1, local_blocks=3)
    full, _ = oracle.score_chunks(q, inp.index_k.numpy(), inp.block_table.numpy(),
                                  inp.seq_lens.numpy(), qo, cols=cols, rank=0, world_size=1,
                                  page_size=128, fill=-np.inf)
    rs, ri = oracle.select(full.astype(np.float32), nvp, init_blocks=1, local_blocks=3)
    heads = slice(rank * hpr, (rank + 1) * hpr)
    out[rank] = bool(np.array_equal(mi, ri[:, heads]) and
                     np.array_equal(ms.view(np.int32), rs[:, heads].view(np.int32)))
    dist.destroy_process_group()


def test_prefill_carrier_exchange_with_gloo():
    port = _free_port()
    out = mp.get_context("spawn").Manager().dict()
    mp.spawn(_prefill_exchange_worker, args=(2, port, out), nprocs=2, join=True)
    assert out[0] and out[1]
