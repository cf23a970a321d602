"""Phase timeline of the decode scorer's launches (timeline build).

    python -m sparse_attention_block_gb300.timeline [--workload batched] [--pdl]
                                                    [--launches 3]

Builds ``_lib/libicp_timeline.so`` (the library compiled with ICP_TIMELINE:
every scorer CTA writes globaltimer stamps of its phases, see
include/icp_timeline.h), draws the workload as bench.py does, warms up, and
then, for each of a few single scorer launches (rank 0's shard), prints per
phase the median / min / max over the CTAs, in microseconds from the
earliest CTA entry of that launch.  The stamps cost a few global stores per
tile, so the absolute times are slightly above the uninstrumented kernel's;
the phases' shares are what the table shows.
"""
from __future__ import annotations

import argparse
import ctypes
import os
import sys

PHASES = [
    (0, "CTA entry"),
    (15, "request lengths read (thread 0's share)"),
    (1, "set-up done (barriers, TMEM, tile prefix sums)"),
    (18, "producer found its first tile (search in the prefix sums)"),
    (12, "producer's griddepcontrol.wait returned (early start)"),
    (16, "producer read its first request's length"),
    (17, "queries' slot free"),
    (13, "producer at its first request (queries' TMA issued)"),
    (14, "first block-table entries read"),
    (2, "first index-K TMA issued"),
    (4, "first tile's MMAs committed"),
    (6, "first tile finished (epilogue warp 0)"),
    (3, "last index-K TMA issued"),
    (5, "last tile's MMAs committed"),
    (10, "last tile finished"),
    (11, "CTA exit"),
]

# slots that hold per-CTA sums: (slot, meaning, divisor to print)
TOTALS = [
    (19, "us the producer waited for a free ring stage", 1e3),
    (20, "us the MMA thread waited for key tiles (prefill)", 1e3),
    (21, "us the MMA thread waited for an accumulator (prefill)", 1e3),
    (22, "us epilogue warp 0 waited for a finished item (prefill)", 1e3),
    (23, "request segments (plan records) of the CTA", 1.0),
]


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="batched",
                    choices=["batched", "multitoken", "sharded", "longctx", "tiny", "prefill"])
    ap.add_argument("--pdl", action="store_true", help="launch with early start")
    ap.add_argument("--launches", type=int, default=3)
    ap.add_argument("--slowest", type=int, default=0,
                    help="also list this many CTAs that exit last, with their sums")
    args = ap.parse_args(argv)

    from . import build
    lib_path = build.build(timeline=True)
    os.environ["ICP_LIBRARY"] = lib_path
    import numpy as np
    import torch

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    if root not in sys.path:
        sys.path.insert(0, root)
    import bench
    from . import icp
    assert icp.LIB_PATH == lib_path
    read = icp.lib.icp_timeline_read
    read.restype = ctypes.c_int
    read.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]

    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    b = bench.make_bench(args.workload, 0, dev)
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    spec = b.spec

    if args.workload == "prefill":
        b.step()                   # the window's plan
        launch = b.kernel_only     # the prefill scorer over the plan's records
        what = f"{b.flops / 1e9:.1f} GFLOP of causal work per launch"
    else:
        def launch():
            icp.icp_score(b.q, b.shards[0], b.bt, b.sl, b.planes[0], rank=0,
                          world_size=spec.world_size, page_size=spec.page_size,
                          decode_query_len=spec.decode_query_len,
                          max_decode_query_len=spec.max_decode_query_len,
                          enable_pdl=args.pdl, errors=b.errors)
        what = f"{b.kbytes / b.ws / 1e6:.1f} MB of index-K per launch"

    for _ in range(5):
        launch()
    torch.cuda.synchronize()
    buf = np.zeros((sms, 24), np.uint64)
    print(f"workload {args.workload}: {what}, {sms} CTAs, "
          f"early start {'on' if args.pdl else 'off'}")
    for n in range(args.launches):
        assert read(buf.ctypes.data, sms, 1) == 0
        launch()
        torch.cuda.synchronize()
        assert read(buf.ctypes.data, sms, 0) == 0
        t0 = int(buf[:, 0].min())
        print(f"launch {n}: us from the first CTA entry, median / min / max over CTAs")
        for slot, name in PHASES:
            col = buf[:, slot].astype(np.int64)
            if not (col > 0).all():
                continue
            d = (col - t0) / 1e3
            print(f"  {name:<55s} {np.median(d):7.2f} {d.min():7.2f} {d.max():7.2f}")
        if args.slowest:
            order = np.argsort(-buf[:, 11].astype(np.int64))
            sel = list(order[:args.slowest]) + list(order[-3:])
            print("  CTA: exit us, first / last TMA us, segments, waits (us): "
                  "free stage, keys, accumulator, item")
            for c in sel:
                r = buf[c].astype(np.int64)
                print(f"  {c:4d}: {(r[11] - t0) / 1e3:7.2f}  {(r[2] - t0) / 1e3:6.2f} "
                      f"{(r[3] - t0) / 1e3:7.2f}  {r[23]:2d}  "
                      + " ".join(f"{r[k] / 1e3:6.2f}" for k in (19, 20, 21, 22)))
        print("  per CTA, median / min / max:")
        for slot, name, scale in TOTALS:
            col = buf[:, slot].astype(np.int64)
            if not col.any():
                continue
            d = col / scale
            print(f"  {name:<55s} {np.median(d):7.2f} {d.min():7.2f} {d.max():7.2f}")
    assert int(b.errors.item()) == 0
    return 0


if __name__ == "__main__":
    sys.exit(main())
