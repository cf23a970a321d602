"""The N > 1 path of bench.py on CPU with gloo (world size 2): timing is the
maximum over ranks, every rank runs its own batch (no data-path collective),
and only rank 0 prints a JSON line."""
import json
import os
import socket
import subprocess
import sys

import pytest
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
    out = mp.Manager().dict()
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
