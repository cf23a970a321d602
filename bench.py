"""Benchmark of the decode-time ICP block indexer on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload multitoken|batched|sharded|longctx|tiny|select|prefill]

One step is one pass of the decode chain over one batch: the score plane
(icp_score, one launch per shard), the Top16 select + publish into legacy
receive rows (icp_publish_rows, one per shard) and the owner merge
(icp_merge, one per owner).  The `select` workload times icp_top16_select
alone on the standalone [256, 4, 12284] plane; the `prefill` workload times
one prefill window (plan, scorer, carrier select, carrier merge) and reports
the scorer against the fp8 tensor peak.

Metric: index-K scoring throughput as algorithmic HBM bytes per second
(index-K rows needed + queries + plane written + block table, then the
select's plane read, the published rows and the merge's reads and writes),
plus rows/s (token x head rows).  Inputs are seeded synthetic tensors that
stay resident in HBM; the default workload's index-K cache (about 1.1 GB) is
larger than L2, so no flush is needed between steps.

Prints ONE JSON line (rank 0).  Under torchrun every rank runs its own
independent batch (weak scaling, no collective on the data path); the
timing is the maximum over ranks.
"""
from __future__ import annotations

import argparse
import ctypes
import json
import os
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "index-K scoring HBM GB/s (% of peak) and score+Top16 rows/s on 1xGB300"
UNIT = "GB/s"
FALLBACK_HBM_GBS = 6800.0

# ncu DRAM counters of icp_score per unit of work (bytes per index-K byte
# streamed), measured for the kernel code with this digest (comments are
# not part of it).  When the code changes the digest no longer matches and
# `traffic` is reported null.
NCU_TRAFFIC = {
    # dram__bytes_read.sum + dram__bytes_write.sum = 278823424 + 3031552 bytes for
    # 278330624 bytes of index-K: one ncu capture of a launch over the first 32
    # requests of the multitoken workload
    ("multitoken", "2dbc8c222f6299f4"): (278823424 + 3031552) / 278330624,
}


# ---------------------------------------------------------------- utilities
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def init_dist(ws, backend):
    if ws > 1:
        import torch.distributed as dist
        if not dist.is_initialized():
            dist.init_process_group(backend=backend)
        return dist
    return None


def max_over_ranks(dist, value: float, device) -> float:
    if dist is None:
        return value
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            with open(p) as f:
                d = json.load(f)
            return float(d["hbm_gbs"]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def measured_tensor_peak_fp8():
    """Dense fp8 tensor peak: the measured bf16 burst figure times the
    nominal fp8 / bf16 ratio (4.5 / 2.25 PFLOP/s)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return 2.0 * float(d["bf16_tflops"]), "measured bf16 burst x 2 (nominal fp8/bf16)"
    except Exception:
        return 2.0 * 1900.0, "fallback 1.9 PFLOP/s bf16 x 2 (nominal fp8/bf16)"


KERNEL_SOURCES = ["icp_score.cu", "icp_fused.cuh", "icp_device.cuh"]


def code_only(text: str) -> str:
    """C/CUDA source without its comments, blank lines and trailing blanks
    (none of these sources holds a comment marker inside a string)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())


def kernel_digest(read=None):
    """Digest of the scorer's code (comments excluded): the ncu traffic
    figures below hold only for the code they were captured on."""
    import hashlib
    if read is None:
        def read(f):
            with open(os.path.join(ROOT, "sparse_attention_block_gb300", "csrc", f)) as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in KERNEL_SOURCES:
        h.update(code_only(read(f)).encode())
    return h.hexdigest()[:16]


class ClockSampler:
    """Samples SM clock and clock-event reasons through NVML (read-only
    queries) in a background thread while the timed region runs."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}

    def __init__(self, device_index: int):
        self.samples = []
        self.max_mhz = None
        self.ok = False
        self._stop = threading.Event()
        try:
            self.nvml = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nvml.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            bus = None
            try:
                props = torch.cuda.get_device_properties(device_index)
                bus = "%08X:%02X:%02X.0" % (props.pci_domain_id, props.pci_bus_id,
                                            props.pci_device_id)
            except Exception:
                bus = None
            rc = -1
            if bus:
                rc = self.nvml.nvmlDeviceGetHandleByPciBusId_v2(bus.encode(), ctypes.byref(self.h))
            if rc != 0:
                rc = self.nvml.nvmlDeviceGetHandleByIndex_v2(0, ctypes.byref(self.h))
            if rc != 0:
                return
            mx = ctypes.c_uint()
            if self.nvml.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx)) == 0:
                self.max_mhz = int(mx.value)
            self._reasons_fn = getattr(self.nvml, "nvmlDeviceGetCurrentClocksEventReasons", None) \
                or self.nvml.nvmlDeviceGetCurrentClocksThrottleReasons
            self.ok = True
        except Exception:
            self.ok = False

    def _sample(self):
        clk = ctypes.c_uint()
        rs = ctypes.c_ulonglong()
        if self.nvml.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0 and \
                self._reasons_fn(self.h, ctypes.byref(rs)) == 0:
            self.samples.append((int(clk.value), int(rs.value)))

    def _run(self):
        while not self._stop.is_set():
            self._sample()
            time.sleep(0.002)

    def start(self):
        if self.ok:
            self._sample()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()

    def stop(self):
        if self.ok:
            self._stop.set()
            self._t.join()
            self._sample()

    # reasons that reject a timing (sw_power_cap is expected under load)
    REJECT = {"hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"}

    @classmethod
    def rejected(cls, summary) -> bool:
        """True when the clock record invalidates the timing: a thermal or
        hardware slowdown was active, or the median SM clock sat below 90 % of
        its maximum with no reason that explains it (a clock lock left over by
        another user)."""
        reasons = set(summary.get("reasons") or [])
        if reasons & cls.REJECT:
            return True
        mhz, mx = summary.get("sm_mhz"), summary.get("sm_max_mhz")
        if mhz is None or not mx or "unavailable" in reasons:
            return False
        explained = reasons - {"applications_clocks_setting", "sync_boost"}
        return not explained and mhz < 0.9 * mx

    def summary(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": self.max_mhz, "reasons": ["unavailable"]}
        clocks = sorted(c for c, _ in self.samples)
        reasons = set()
        for _, r in self.samples:
            for bit, name in self.REASONS.items():
                if r & bit and name != "gpu_idle":
                    reasons.add(name)
        return {"sm_mhz": clocks[len(clocks) // 2], "sm_max_mhz": self.max_mhz,
                "reasons": sorted(reasons), "samples": len(self.samples)}


# ---------------------------------------------------------------- workloads
def algorithmic_bytes(spec, seq_lens, cols):
    """Per step: (scorer bytes, select/publish bytes, merge bytes).

    Scorer: index-K rows needed (sum seq_len * 128, all shards together) +
    queries (ws * T * 512) + plane columns written (ws * sum_t 16 * cols_b) +
    block table entries (ws * sum_b 4 * ceil(seq_len / page_size)).
    Select/publish: plane columns read back + 132 B per published row.
    Merge: 132 B per source row read + 128 B per merged row written.
    """
    ws, ps, dql = spec.world_size, spec.page_size, spec.decode_query_len
    unit = 128 if (ps == 128 or ws == 1) else ps
    T = len(seq_lens) * dql
    kbytes = sum(int(L) * 128 for L in seq_lens)
    qbytes = ws * T * 512
    cols_b = [((int(L) + unit - 1) // unit + 3) // 4 * 4 for L in seq_lens]
    plane = ws * sum(16 * c * dql for c in cols_b)
    bt = ws * sum(4 * ((int(L) + ps - 1) // ps) for L in seq_lens)
    score = kbytes + qbytes + plane + bt
    select = plane + ws * T * 4 * 132 + ws * T * 4
    merge = ws * T * 4 * 132 + T * 4 * 128 + T * 4
    return score, select, merge, kbytes


class DecodeBench:
    def __init__(self, spec, seed, device):
        from sparse_attention_block_gb300 import icp
        from sparse_attention_block_gb300 import workloads as W
        self.icp = icp
        self.spec = spec
        self.device = device
        inp = W.make_decode_inputs(spec, seed=seed, device=device, make_shards=True)
        self.inp = inp
        self.T = inp.T
        ws = spec.world_size
        self.ws = ws
        self.hpr = 4 // ws
        self.cols = icp.icp_score_columns(int(inp.seq_lens.max().item()), spec.page_size, ws)
        self.cap = spec.capacity or self.T
        self.q, self.bt, self.sl, self.nvp = inp.index_q, inp.block_table, inp.seq_lens, \
            inp.num_valid_pages
        self.shards = inp.shards if ws > 1 else [inp.index_k]
        if ws > 1:
            inp.index_k = None   # only the shards stay resident
        self.planes = [torch.empty((self.T, 4, self.cols), dtype=torch.float32, device=device)
                       for _ in range(ws)]
        rows = icp.recv_rows(ws, self.hpr, self.cap)
        self.recv = [torch.zeros((rows, 33), dtype=torch.int32, device=device) for _ in range(ws)]
        self.bases = torch.tensor([r.data_ptr() for r in self.recv], dtype=torch.int64,
                                  device=device)
        self.errors = torch.zeros(1, dtype=torch.int32, device=device)
        self.out_s = [torch.empty((self.T, self.hpr, 16), dtype=torch.float32, device=device)
                      for _ in range(ws)]
        self.out_i = [torch.empty((self.T, self.hpr, 16), dtype=torch.int32, device=device)
                      for _ in range(ws)]
        self.slot = 0
        wsz = icp.icp_score_select_workspace_bytes(len(inp.seq_lens), spec.decode_query_len)
        self.work = torch.empty((wsz,), dtype=torch.uint8, device=device)
        self.f_s = [torch.empty((self.T, 4, 16), dtype=torch.float32, device=device)
                    for _ in range(ws)]
        self.f_i = [torch.empty((self.T, 4, 16), dtype=torch.int32, device=device)
                    for _ in range(ws)]
        self.seq_list = inp.seq_lens.cpu().tolist()
        self.score_bytes, self.select_bytes, self.merge_bytes, self.kbytes = \
            algorithmic_bytes(spec, self.seq_list, self.cols)
        self.launches_per_step = 3 * ws
        self.kernel_launches_per_step = ws
        # the scorers are ordinary launches: with early start (programmatic
        # dependent launch) every step measured slower on this GPU; the line
        # reports that step beside the default one
        self.score_pdl = False

    @property
    def fused_bytes(self):
        """icp_score_select per step: index-K rows needed + queries + block table +
        num_valid_pages + the Top16 output, per shard; no plane."""
        spec, ws = self.spec, self.ws
        bt = ws * sum(4 * ((int(L) + spec.page_size - 1) // spec.page_size)
                      for L in self.seq_list)
        return self.kbytes + ws * (self.T * 512 + self.T * 4 + self.T * 4 * 16 * 8) + bt

    @property
    def step_bytes(self):
        return self.score_bytes + self.select_bytes + self.merge_bytes

    @property
    def rows(self):
        return self.T * 4

    def step(self, ev=None):
        icp, spec, ws = self.icp, self.spec, self.ws
        slot = self.slot
        for rank in range(ws):
            if ev is not None and rank == 0:
                ev[0].record()
            icp.icp_score(self.q, self.shards[rank], self.bt, self.sl, self.planes[rank],
                          rank=rank, world_size=ws, page_size=spec.page_size,
                          decode_query_len=spec.decode_query_len,
                          max_decode_query_len=spec.max_decode_query_len,
                          enable_pdl=self.score_pdl, errors=self.errors)
            if ev is not None and rank == ws - 1:
                ev[1].record()
        for rank in range(ws):
            scale, offset = (1, 0) if (spec.page_size == 128 or ws == 1) else (2, rank * 2 // ws)
            icp.icp_publish_rows(self.planes[rank], self.nvp, self.bases, self.errors, slot=slot,
                                 rank=rank, world_size=ws, heads_per_rank=self.hpr,
                                 capacity=self.cap, force_begin_blocks=spec.init_blocks,
                                 force_end_blocks=spec.local_blocks, spin_limit=1 << 22,
                                 index_scale=scale, index_offset=offset, enable_pdl=True)
        for owner in range(ws):
            icp.icp_merge(self.recv[owner], self.nvp, self.out_s[owner], self.out_i[owner],
                          self.errors, T=self.T, slot=slot, world_size=ws,
                          heads_per_rank=self.hpr, capacity=self.cap,
                          init_blocks=spec.init_blocks, local_blocks=spec.local_blocks,
                          spin_limit=1 << 22, enable_pdl=True)
        self.slot = (slot + 1) % 3

    graph_period = 3   # receive slots rotate 0, 1, 2

    def kernel_only(self):
        """The scorer launches of one step (every shard), nothing else."""
        icp, spec, ws = self.icp, self.spec, self.ws
        for rank in range(ws):
            icp.icp_score(self.q, self.shards[rank], self.bt, self.sl, self.planes[rank],
                          rank=rank, world_size=ws, page_size=spec.page_size,
                          decode_query_len=spec.decode_query_len,
                          max_decode_query_len=spec.max_decode_query_len,
                          enable_pdl=self.score_pdl, errors=self.errors)

    def fused_step(self):
        """The fused scorer + Top16 select (no score plane), one launch per shard."""
        icp, spec, ws = self.icp, self.spec, self.ws
        for rank in range(ws):
            icp.icp_score_select(self.q, self.shards[rank], self.bt, self.sl, self.nvp,
                                 self.f_s[rank], self.f_i[rank], self.work, cols=self.cols,
                                 rank=rank, world_size=ws, page_size=spec.page_size,
                                 decode_query_len=spec.decode_query_len,
                                 max_decode_query_len=spec.max_decode_query_len,
                                 init_blocks=spec.init_blocks, local_blocks=spec.local_blocks,
                                 errors=self.errors)

    def e2e(self, steps, warmup):
        """The chain through the public API with every step's inputs copied
        from pinned host memory and its merged Top16 read back, all inside
        the timed region, in the order of a serving loop: two sets of device
        inputs and outputs, a host-to-device stream that fills set (i + 1) % 2
        once step i - 1 is done with it, and a device-to-host stream that
        reads step i's lists once step i is done, so both overlap the
        neighbouring steps' kernels."""
        pin = lambda t: t.cpu().pin_memory()
        h_in = [pin(self.q), pin(self.bt), pin(self.sl), pin(self.nvp)]
        d_in = [[self.q, self.bt, self.sl, self.nvp],
                [torch.empty_like(t) for t in (self.q, self.bt, self.sl, self.nvp)]]
        d_out = [(self.out_s, self.out_i),
                 ([torch.empty_like(o) for o in self.out_s],
                  [torch.empty_like(o) for o in self.out_i])]
        h_out = [[torch.empty(o.shape, dtype=o.dtype).pin_memory()
                  for o in self.out_s + self.out_i] for _ in range(2)]
        bi = sum(t.numel() * t.element_size() for t in h_in)
        bo = sum(t.numel() * t.element_size() for t in h_out[0])
        compute = torch.cuda.current_stream()
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        ev_in = [torch.cuda.Event() for _ in range(2)]
        ev_done = [torch.cuda.Event() for _ in range(2)]
        ev_read = [torch.cuda.Event() for _ in range(2)]
        for k in range(2):          # every event starts recorded
            for e in (ev_done[k], ev_read[k]):
                e.record(compute)

        def h2d(k):
            with torch.cuda.stream(s_in):
                s_in.wait_event(ev_done[k])      # step i - 2 no longer reads set k
                for d, h in zip(d_in[k], h_in):
                    d.copy_(h, non_blocking=True)
                ev_in[k].record(s_in)

        def run(n):
            h2d(0)
            for i in range(n):
                k = i % 2
                compute.wait_event(ev_in[k])
                compute.wait_event(ev_read[k])  # step i - 2's lists are read back
                self.q, self.bt, self.sl, self.nvp = d_in[k]
                self.out_s, self.out_i = d_out[k]
                self.step()
                ev_done[k].record(compute)
                if i + 1 < n:
                    h2d((i + 1) % 2)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(ev_done[k])
                    for d, h in zip(self.out_s + self.out_i, h_out[k]):
                        h.copy_(d, non_blocking=True)
                    ev_read[k].record(s_out)

        run(warmup)
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run(steps)
        torch.cuda.synchronize()
        dt = time.perf_counter() - t0
        self.q, self.bt, self.sl, self.nvp = d_in[0]
        self.out_s, self.out_i = d_out[0]
        return dt / steps, bi, bo


class SelectBench:
    def __init__(self, seed, device):
        from sparse_attention_block_gb300 import icp
        from sparse_attention_block_gb300 import workloads as W
        self.icp = icp
        self.plane, self.nvp = W.make_select_plane(seed=seed, device=device)
        self.T = self.plane.shape[0]
        self.K = self.plane.shape[2]
        self.out_s = torch.empty((self.T, 4, 16), dtype=torch.float32, device=device)
        self.out_i = torch.empty((self.T, 4, 16), dtype=torch.int32, device=device)
        self.init, self.local = W.SELECT_INIT, W.SELECT_LOCAL
        # valid columns only (ids < num_valid_pages; index scale 1, offset 0):
        # the columns past them need not be read
        valid = self.nvp.clamp(max=self.K).to(torch.int64)
        self.score_bytes = int(valid.sum().item()) * 4 * 4 + self.T * 4 + self.T * 4 * 16 * 8
        self.select_bytes = self.merge_bytes = 0
        self.kbytes = 0
        self.launches_per_step = 1
        self.kernel_launches_per_step = 1
        # rotate copies so consecutive steps do not hit the 50 MB plane in L2
        self.copies = [self.plane] + [self.plane.clone() for _ in range(5)]
        self.i = 0

    step_bytes = property(lambda self: self.score_bytes)
    rows = property(lambda self: self.T * 4)
    graph_period = 6   # the six rotated plane copies

    def kernel_only(self):
        self.step()

    def step(self, ev=None):
        p = self.copies[self.i % len(self.copies)]
        self.i += 1
        if ev is not None:
            ev[0].record()
        self.icp.icp_top16_select(p, self.nvp, self.out_s, self.out_i, init_blocks=self.init,
                                  local_blocks=self.local)
        if ev is not None:
            ev[1].record()


class PrefillBench:
    """One prefill window: plan, scorer over the plan's records, Top16 into
    carrier rows, and the merge of the (single-rank) carrier."""
    graph_period = 3   # windows per graph replay (the same window each time)

    def __init__(self, spec, seed, device):
        from sparse_attention_block_gb300 import icp
        from sparse_attention_block_gb300 import workloads as W
        self.icp = icp
        self.spec = spec
        inp = W.make_decode_inputs(spec, seed=seed, device=device)
        self.q, self.k, self.bt, self.sl, self.nvp = (inp.index_q, inp.index_k,
                                                      inp.block_table, inp.seq_lens,
                                                      inp.num_valid_pages)
        B, n = len(self.sl), spec.decode_query_len
        self.T = B * n
        self.qo = torch.arange(0, (B + 1) * n, n, dtype=torch.int32, device=device)
        self.cols = W.columns_for(spec, int(self.sl.max()))
        self.plan = torch.empty((icp.icp_prefill_plan_words(B, self.T),), dtype=torch.int32,
                                device=device)
        self.plane = torch.empty((self.T, 4, self.cols), dtype=torch.float32, device=device)
        self.carrier = torch.empty((1, self.T, 4, 32), dtype=torch.int32, device=device)
        self.out_s = torch.empty((self.T, 4, 16), dtype=torch.float32, device=device)
        self.out_i = torch.empty((self.T, 4, 16), dtype=torch.int32, device=device)
        self.errors = torch.zeros(1, dtype=torch.int32, device=device)
        self.shards = [self.k]
        sl = [int(x) for x in self.sl.tolist()]
        self.score_bytes, self.select_bytes, self.merge_bytes, self.kbytes = \
            prefill_bytes(sl, n, self.cols)
        # useful MMA work: every (token, head) against every key at or
        # before its position, 2 * 128 flops per key
        self.flops = sum(4 * 256 * (sum(range(L - n + 1, L + 1))) for L in sl)
        self.launches_per_step = 4
        self.kernel_launches_per_step = 1

    step_bytes = property(lambda self: self.score_bytes + self.select_bytes + self.merge_bytes)
    rows = property(lambda self: self.T * 4)

    def kernel_only(self):
        self.icp.icp_prefill_score(self.q, self.k, self.bt, self.plan, self.plane, rank=0,
                                   world_size=1, page_size=self.spec.page_size,
                                   errors=self.errors)

    def step(self, ev=None):
        if ev is not None:
            ev[0].record()
        self.icp.icp_prefill_plan(self.qo, self.sl, self.plan, T=self.T, errors=self.errors)
        self.kernel_only()
        self.icp.icp_prefill_select(self.plane, self.nvp, self.carrier, world_size=1,
                                    heads_per_rank=4, init_blocks=self.spec.init_blocks,
                                    local_blocks=self.spec.local_blocks)
        self.icp.icp_prefill_merge(self.carrier, self.nvp, self.out_s, self.out_i, world_size=1,
                                   heads_per_rank=4, init_blocks=self.spec.init_blocks,
                                   local_blocks=self.spec.local_blocks)
        if ev is not None:
            ev[1].record()


def prefill_bytes(seq_lens, n, cols):
    """Per window (unsharded): (scorer bytes, select bytes, merge bytes, index-K bytes).

    Scorer: index-K rows needed once (sum seq_len * 128) + queries (T * 512) +
    plane columns written (T * 16 * cols_b) + block table.  Select: the plane
    read back + 128 B per carrier row.  Merge: 128 B per carrier row read +
    128 B per output row written."""
    T = len(seq_lens) * n
    kbytes = sum(L * 128 for L in seq_lens)
    cols_b = [((L + 127) // 128 + 3) // 4 * 4 for L in seq_lens]
    plane = sum(16 * c * n for c in cols_b)
    bt = sum(4 * ((L + 127) // 128) for L in seq_lens)
    score = kbytes + T * 512 + plane + bt
    select = plane + T * 4 * 128 + T * 4
    merge = T * 4 * 128 + T * 4 * 128 + T * 4
    return score, select, merge, kbytes


# ------------------------------------------------------------ CPU baselines
def _np(x):
    """A host numpy array of a tensor (or an array already on the host)."""
    import numpy as np
    return x.cpu().numpy() if hasattr(x, "cpu") else np.asarray(x)


class OracleBatch:
    """One workload's batch for the oracle arm, as host arrays.

    It is drawn by the same seeded recipe as the CUDA arm's batch, on the GPU
    when there is one (so that both arms time the same batch), and the plane
    width comes from the oracle's own column count.  Nothing on this path
    loads the CUDA library."""

    def __init__(self, name, seed, device, batch=0):
        import dataclasses

        import oracle
        from sparse_attention_block_gb300 import workloads as W
        if name == "select":
            plane, nvp = W.make_select_plane(seed=seed, device=device)
            self.plane, self.nvp = _np(plane), _np(nvp)
            self.T, self.K = self.plane.shape[0], self.plane.shape[2]
            self.init, self.local = W.SELECT_INIT, W.SELECT_LOCAL
            self.rows = self.T * 4
            return
        spec = W.PREFILL if name == "prefill" else W.DECODE_SPECS[name]
        if batch and name != "prefill":
            spec = dataclasses.replace(spec, batch=batch, seq_lens=spec.seq_lens[:batch],
                                       description=spec.description +
                                       f" (first {batch} requests)")
        inp = W.make_decode_inputs(spec, seed=seed, device=device, make_shards=True)
        self.spec = spec
        self.q, self.bt, self.sl, self.nvp = (_np(inp.index_q), _np(inp.block_table),
                                              _np(inp.seq_lens), _np(inp.num_valid_pages))
        self.shards = ([_np(s) for s in inp.shards] if spec.world_size > 1
                       else [_np(inp.index_k)])
        self.k = self.shards[0]
        del inp
        self.seq_list = [int(x) for x in self.sl]
        self.T = len(self.seq_list) * spec.decode_query_len
        self.cols = oracle.columns_written(max(self.seq_list), spec.page_size, spec.world_size)
        self.kbytes = sum(L * 128 for L in self.seq_list)
        self.rows = self.T * 4


def _oracle_arrays(bench):
    """The batch as numpy arrays, and the chain's parameters."""
    spec = bench.spec
    arrays = (_np(bench.q), [_np(s) for s in bench.shards], _np(bench.bt), _np(bench.sl),
              _np(bench.nvp))
    params = dict(cols=bench.cols, world_size=spec.world_size, page_size=spec.page_size,
                  decode_query_len=spec.decode_query_len, init_blocks=spec.init_blocks,
                  local_blocks=spec.local_blocks)
    return arrays, params


def _sample_bytes(bench, reqs):
    sl = bench.seq_list
    nbytes = 0
    for b in reqs:
        s, se, m, _ = algorithmic_bytes(bench.spec, [int(sl[b])], bench.cols)
        nbytes += s + se + m
    return nbytes


def oracle_sample(bench, budget_s):
    """Runs the oracle's chain (score, select+publish, merge) on the first
    requests of the workload, one thread, until about budget_s seconds of
    CPU work.  Returns (seconds, algorithmic bytes of the sample, rows,
    requests)."""
    from oracle.parallel import decode_request
    (q, shards, bt, sl, nvp), params = _oracle_arrays(bench)
    spent, nreq = 0.0, 0
    for b in range(len(sl)):
        if spent >= budget_s and nreq > 0:
            break
        t0 = time.perf_counter()
        decode_request(q, shards, bt, sl, nvp, b, **params)
        spent += time.perf_counter() - t0
        nreq += 1
    rows = nreq * bench.spec.decode_query_len * 4
    return spent, _sample_bytes(bench, range(nreq)), rows, nreq


class OracleParallel:
    """The oracle's chain over the requests of the batch in one spawned
    worker process per host core (the batch in shared memory)."""

    def __init__(self, bench):
        from oracle.parallel import ParallelChain
        arrays, params = _oracle_arrays(bench)
        self.bench = bench
        self.pc = ParallelChain(*arrays, params)
        self.cores = self.pc.workers

    def sample(self, budget_s, per_request_s):
        """Wall seconds, bytes, rows and requests of one timed pass over the
        first n requests, n sized to about budget_s of wall time."""
        B = len(self.bench.seq_list)
        n = min(B, max(self.cores, int(budget_s * self.cores / max(per_request_s, 1e-6))))
        wall = self.pc.time(range(n))
        rows = n * self.bench.spec.decode_query_len * 4
        return wall, _sample_bytes(self.bench, range(n)), rows, n

    def close(self):
        self.pc.close()


def oracle_select_sample(bench, budget_s):
    import oracle
    plane = _np(bench.plane)
    nvp = _np(bench.nvp)
    spent, rows, t = 0.0, 0, 0
    while t < bench.T and (spent < budget_s or rows == 0):
        t0 = time.perf_counter()
        oracle.select(plane[t:t + 1], nvp[t:t + 1], init_blocks=bench.init,
                      local_blocks=bench.local)
        spent += time.perf_counter() - t0
        rows += 4
        t += 1
    nbytes = rows * bench.K * 4
    return spent, nbytes, rows, t


def oracle_prefill_sample(bench, budget_s):
    """The oracle's prefill chain (window plane, carrier, merge) on growing
    leading parts of request 0's chunk until about budget_s seconds."""
    import numpy as np
    import oracle
    spec = bench.spec
    n = spec.decode_query_len
    L = int(bench.sl[0])
    q = _np(bench.q[:n])
    k = _np(bench.k)
    bt = _np(bench.bt[:1])
    nvp = _np(bench.nvp[:n])
    spent, nbytes, rows, m = 0.0, 0, 0, 0
    step = 16
    while m < n and (spent < budget_s or rows == 0):
        # tokens m .. m + step - 1 of the chunk: a window of its own whose
        # request length ends at the last of them
        m1 = min(n, m + step)
        Lm = L - n + m1
        qo = np.array([0, m1 - m], np.int32)
        t0 = time.perf_counter()
        plane, _ = oracle.score_chunks(q[m:m1], k, bt, np.array([Lm], np.int32), qo,
                                       cols=bench.cols, rank=0, world_size=1,
                                       page_size=spec.page_size, fill=-np.inf)
        car = oracle.carrier(plane.astype(np.float32), nvp[m:m1], world_size=1,
                             heads_per_rank=4, init_blocks=spec.init_blocks,
                             local_blocks=spec.local_blocks)
        oracle.merge_carrier(car, nvp[m:m1], world_size=1, heads_per_rank=4,
                             init_blocks=spec.init_blocks, local_blocks=spec.local_blocks)
        spent += time.perf_counter() - t0
        s, se, me, _ = prefill_bytes([Lm], m1 - m, bench.cols)
        nbytes += s + se + me
        rows += (m1 - m) * 4
        m = m1
    return spent, nbytes, rows, m


def workload_config(name, bench):
    if name == "prefill":
        spec = bench.spec
        return {"workload": spec.description, "batch": spec.batch, "T": bench.T,
                "cols": bench.cols, "page_size": spec.page_size, "world_size": 1,
                "chunk_tokens": spec.decode_query_len, "index_k_bytes_per_step": bench.kbytes,
                "l2": "index-K cache smaller than L2 (re-read from L2 by every 64-token record)",
                "step": "icp_prefill_plan -> icp_prefill_score -> icp_prefill_select -> "
                        "icp_prefill_merge, replayed as a CUDA graph"}
    if name == "select":
        return {"workload": "standalone Top16 select: float32 plane [256, 4, 12284] N(0,1) "
                            "with 2% tied duplicates, num_valid_pages U[1, 12284], init 4, "
                            "local 8", "rows": bench.rows, "l2": "6 rotated plane copies"}
    spec = bench.spec
    return {"workload": spec.description, "batch": spec.batch, "T": bench.T, "cols": bench.cols,
            "page_size": spec.page_size, "world_size": spec.world_size,
            "decode_query_len": spec.decode_query_len,
            "index_k_bytes_per_step": bench.kbytes,
            "l2": "inputs larger than L2 (index-K cache streamed every step)"
            if bench.kbytes > 200e6 else "index-K cache smaller than L2 (partly L2-resident)",
            "step": "icp_score -> icp_publish_rows -> icp_merge (per shard / owner), "
                    "replayed as CUDA graphs"}


# ---------------------------------------------------------------- main arms
ORACLE_STEPS = {
    "decode": "the oracle's chain per request (plain C, fp64): exact score plane of every "
              "shard -> Top16 select + publish into receive rows -> owner merge",
    "select": "the oracle's brute-force Top16 select per row (plain C)",
    "prefill": "the oracle's prefill chain (plain C, fp64): exact window plane -> carrier rows "
               "-> carrier merge",
}


def run_reference(args, spec_name):
    """The oracle (plain C) timed per step on a bounded sample: decode chains
    over the requests on every host core, select and prefill on one thread."""
    ws, rank, local = dist_env()
    if rank != 0:
        return 0
    device = torch.device("cuda", local) if torch.cuda.is_available() else torch.device("cpu")
    bench = OracleBatch(spec_name, 0, device, args.batch)
    # each step a bounded sample: about two minutes of oracle work in all
    # (ICP_REF_STEP_SECONDS overrides the per-step budget)
    per_step = float(os.environ.get(
        "ICP_REF_STEP_SECONDS",
        str(min(2.0, max(0.05, 120.0 / max(1, args.steps + args.warmup / 4))))))
    cores, par = 1, None
    if spec_name not in ("select", "prefill"):
        # decode chains run over the requests on every host core
        s1, _, _, n1 = oracle_sample(bench, 0.0)
        par = OracleParallel(bench)
        cores = par.cores
        step = lambda budget: par.sample(budget, s1 / n1)
    else:
        step = lambda budget: oracle_step(bench, spec_name, budget)
    try:
        for _ in range(args.warmup):
            step(per_step / 4)
        tot_s, tot_b, tot_r, reqs = 0.0, 0, 0, 0
        for _ in range(args.steps):
            s, b, r, n = step(per_step)
            tot_s, tot_b, tot_r, reqs = tot_s + s, tot_b + b, tot_r + r, n
    finally:
        if par is not None:
            par.close()
    value = tot_b / tot_s / 1e9
    line = {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(tot_s / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": dict(workload_config(spec_name, bench), step=ORACLE_STEPS[
            spec_name if spec_name in ORACLE_STEPS else "decode"]),
        "rows_per_s": round(tot_r / tot_s, 2),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": cores, "kind": "oracle",
                         "sample": f"first {reqs} request(s) / row(s) of the workload per step, "
                                   f"about {per_step:.1f} s of C oracle work "
                                   + (f"on {cores} spawned processes" if cores > 1
                                      else "on one thread")},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def oracle_step(bench, name, budget):
    if name == "select":
        return oracle_select_sample(bench, budget)
    if name == "prefill":
        return oracle_prefill_sample(bench, budget)
    return oracle_sample(bench, budget)


def make_bench(name, seed, device, batch=0):
    import dataclasses

    from sparse_attention_block_gb300 import workloads as W
    if name == "select":
        return SelectBench(seed, device)
    if name == "prefill":
        return PrefillBench(W.PREFILL, seed, device)
    spec = W.DECODE_SPECS[name]
    if batch:
        spec = dataclasses.replace(spec, batch=batch, seq_lens=spec.seq_lens[:batch],
                                   description=spec.description + f" (first {batch} requests)")
    return DecodeBench(spec, seed, device)


def capture(bench):
    """CUDA graphs of the step and of the dominant kernel alone.  The library
    only enqueues, so its calls capture.  One graph holds a whole period of
    steps (the receive slots 0, 1, 2, or the rotated inputs) back to back,
    so that every launch inside it follows its predecessor as in a serving
    loop: launched with programmatic dependent launch, a scorer starts its
    set-up while the previous step's merge runs.  Shorter graphs cover the
    remainder of a step count that is not a multiple of the period."""
    period = bench.graph_period

    def graph_of(fn, n):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                fn()
        return g

    steps = [graph_of(bench.step, period)] + [graph_of(bench.step, r) for r in range(1, period)]
    kernels = [graph_of(bench.kernel_only, period)] + [graph_of(bench.kernel_only, r)
                                                        for r in range(1, period)]
    return steps, kernels


def replay(graphs, n):
    """Replays n steps' worth: whole periods, then the remainder graph."""
    period = len(graphs)
    for _ in range(n // period):
        graphs[0].replay()
    if n % period:
        graphs[n % period].replay()


def timed_graphs(bench, steps, warmup, local, dist=None):
    """Step and dominant-kernel times (ms) of graph replays, CUDA events on
    the launching stream, clocks sampled through the timed region.  A timing
    whose clock record shows a slowdown (or a leftover clock lock) is taken
    once more, every rank following the same decision."""
    for _ in range(max(warmup, 3)):
        bench.step()
    torch.cuda.synchronize()
    graphs, kgraphs = capture(bench)
    stream = torch.cuda.current_stream()
    device = torch.device("cuda", local)
    replay(graphs, max(warmup, 3))
    replay(kgraphs, max(warmup, 3))
    torch.cuda.synchronize()

    def region():
        start, end, ka, kb = (torch.cuda.Event(enable_timing=True) for _ in range(4))
        sampler = ClockSampler(local)
        barrier(dist)
        torch.cuda.synchronize()
        sampler.start()
        start.record(stream)
        replay(graphs, steps)
        end.record(stream)
        # the dominant kernel's launch duration, same stream, same inputs
        ka.record(stream)
        replay(kgraphs, steps)
        kb.record(stream)
        torch.cuda.synchronize()
        sampler.stop()
        barrier(dist)
        return start.elapsed_time(end) / steps, ka.elapsed_time(kb) / steps, sampler.summary()

    step_ms, kernel_ms, clocks = region()
    if max_over_ranks(dist, float(ClockSampler.rejected(clocks)), device) > 0:
        first = clocks["reasons"]
        step_ms, kernel_ms, clocks = region()
        clocks = dict(clocks, remeasured=True, first_run_reasons=first)
    return step_ms, kernel_ms, clocks


def timed_fused(bench, steps, warmup):
    """ms per step of the fused scorer + select, replayed like the step."""
    for _ in range(max(warmup, 3)):
        bench.fused_step()
    torch.cuda.synchronize()
    period = bench.graph_period
    graphs = []
    for n in [period] + list(range(1, period)):
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for _ in range(n):
                bench.fused_step()
        graphs.append(g)
    replay(graphs, 3)
    torch.cuda.synchronize()
    stream = torch.cuda.current_stream()
    fa, fb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    fa.record(stream)
    replay(graphs, steps)
    fb.record(stream)
    torch.cuda.synchronize()
    return fa.elapsed_time(fb) / steps


def timed_step_with_scorer_pdl(bench, steps, warmup, local):
    """The decode step with the scorers launched under programmatic dependent
    launch (early start: the CTAs' set-up runs ahead of griddepcontrol.wait),
    timed like the step itself: ms per step."""
    bench.score_pdl = True
    try:
        step_ms, _, _ = timed_graphs(bench, steps, warmup, local)
    finally:
        bench.score_pdl = False
    return step_ms


def roofline_of(name, bench, kernel_ms, peak, peak_kind, digest, traffic=None):
    kernel_name = "icp_top16_select" if name == "select" else (
        "icp_prefill_score" if name == "prefill" else "icp_score")
    kernel_bytes = bench.score_bytes
    achieved = kernel_bytes / (kernel_ms / 1e3) / 1e9
    if name == "prefill":
        # many query rows against the same keys: a dense fp8 contraction
        tpeak, tkind = measured_tensor_peak_fp8()
        t_achieved = bench.flops / (kernel_ms / 1e3) / 1e12
        return {"bound": "tensor", "kernel": kernel_name, "achieved": round(t_achieved, 1),
                "peak": tpeak, "unit": "TFLOP/s", "frac": round(t_achieved / tpeak, 4),
                "peak_source": tkind, "traffic": None,
                "algorithmic_flops_per_launch": bench.flops,
                "hbm_achieved_gbs": round(achieved, 1), "kernel_digest": digest}
    per = bench.kernel_launches_per_step
    return {"bound": "hbm", "kernel": kernel_name, "achieved": round(achieved, 1),
            "peak": peak, "unit": "GB/s", "frac": round(achieved / peak, 4),
            "peak_source": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
            if peak_kind == "measured" else "fallback 6.8 TB/s",
            "traffic": traffic, "algorithmic_bytes_per_launch": kernel_bytes // per,
            "launches_timed_together": per, "algorithmic_bytes_timed": kernel_bytes,
            "kernel_digest": digest}


# The other workloads, each reported as a short record in the default line.
RECORD_WORKLOADS = ("longctx", "batched", "sharded", "select", "prefill")


def one_shot_read_ms(nbytes, steps, copies=6):
    """A library reference for reading nbytes once: torch.sum over a float32
    buffer of that size, six fresh buffers taken in turn (so no read hits
    L2), replayed from one graph like the select: ms per sum."""
    n = nbytes // 4
    bufs = [torch.randn(n, device="cuda") for _ in range(copies)]
    out = torch.empty((), device="cuda")
    for b in bufs:
        torch.sum(b, dim=0, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for b in bufs:
            torch.sum(b, dim=0, out=out)
    g.replay()
    torch.cuda.synchronize()
    reps = max(1, steps // copies)
    stream = torch.cuda.current_stream()
    ea, eb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ea.record(stream)
    for _ in range(reps):
        g.replay()
    eb.record(stream)
    torch.cuda.synchronize()
    return ea.elapsed_time(eb) / (reps * copies)


def workload_record(name, steps, warmup, local, peak, peak_kind, digest):
    """Device-timed record of one more workload: its dominant kernel, its
    step, the roofline of the kernel, the fused step where there is one, the
    decode step with the scorer's early start, and the clocks."""
    bench = make_bench(name, 0, torch.device("cuda", local))
    try:
        step_ms, kernel_ms, clocks = timed_graphs(bench, steps, warmup, local)
        rec = {"config": workload_config(name, bench),
               "kernel_ms": round(kernel_ms, 5), "step_ms": round(step_ms, 5),
               "step_GB/s": round(bench.step_bytes / (step_ms / 1e3) / 1e9, 1),
               "rows_per_s": round(bench.rows / (step_ms / 1e3), 1),
               "roofline": roofline_of(name, bench, kernel_ms, peak, peak_kind, digest),
               "clocks": clocks}
        if isinstance(bench, DecodeBench):
            f_ms = timed_fused(bench, steps, warmup)
            rec["fused_step_ms"] = round(f_ms, 5)
            rec["fused_GB/s"] = round(bench.fused_bytes / (f_ms / 1e3) / 1e9, 1)
            rec["step_ms_scorer_with_pdl"] = round(
                timed_step_with_scorer_pdl(bench, steps, warmup, local), 5)
        if name == "select":
            # what reading the same valid bytes once costs a library kernel
            r_ms = one_shot_read_ms(bench.score_bytes, steps)
            rec["one_shot_read"] = {
                "what": "torch.sum over a float32 buffer of the select's algorithmic bytes, "
                        "6 rotated buffers, one graph", "ms": round(r_ms, 5),
                "GB/s": round(bench.score_bytes / (r_ms / 1e3) / 1e9, 1),
                "select_ms_over_read_ms": round(kernel_ms / r_ms, 3)}
        errors = int(bench.errors.item()) if hasattr(bench, "errors") else 0
        if errors:
            raise SystemExit(f"{name}: {errors} device errors during the benchmark")
        return rec
    finally:
        del bench
        torch.cuda.empty_cache()


def run_ours(args, spec_name):
    ws, rank, local = dist_env()
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (GB300)")
    device = torch.device("cuda", local)
    torch.cuda.set_device(device)
    dist = init_dist(ws, "nccl")
    bench = make_bench(spec_name, rank, device, args.batch)

    ms_per_step, kernel_ms, clocks = timed_graphs(bench, args.steps, args.warmup, local, dist)
    ms_per_step = max_over_ranks(dist, ms_per_step, device)
    errors = int(bench.errors.item()) if hasattr(bench, "errors") else 0
    if errors:
        raise SystemExit(f"{errors} device errors during the benchmark")

    n = ws
    value = n * bench.step_bytes / (ms_per_step / 1e3) / 1e9
    rows_per_s = n * bench.rows / (ms_per_step / 1e3)
    peak, peak_kind = measured_peaks()
    digest = kernel_digest()
    traffic = None
    tr = NCU_TRAFFIC.get((spec_name, digest))
    if tr is not None:
        traffic = int(tr * bench.kbytes) if bench.kbytes else int(tr)
    roofline = roofline_of(spec_name, bench, kernel_ms, peak, peak_kind, digest, traffic)
    kernel_name = roofline["kernel"]
    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": n,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "fp8e4m3/f32",
        "data": "synthetic (seeded; see sparse_attention_block_gb300/workloads.py)",
        "config": workload_config(spec_name, bench),
        "rows_per_s": round(rows_per_s, 1),
        "kernels": {kernel_name + "_ms": round(kernel_ms, 5)},
        "roofline": roofline,
        "clocks": clocks,
        "gpu_launches": bench.launches_per_step * args.steps,
        "kernel_timing_launches": bench.kernel_launches_per_step * args.steps,
    }
    if spec_name == "select":
        r_ms = one_shot_read_ms(bench.score_bytes, args.steps)
        line["one_shot_read"] = {
            "what": "torch.sum over a float32 buffer of the select's algorithmic bytes, "
                    "6 rotated buffers, one graph", "ms": round(r_ms, 5),
            "GB/s": round(bench.score_bytes / (r_ms / 1e3) / 1e9, 1),
            "select_ms_over_read_ms": round(kernel_ms / r_ms, 3)}
    if isinstance(bench, DecodeBench):
        f_ms = timed_fused(bench, args.steps, args.warmup)
        f_bytes = bench.fused_bytes
        line["fused_score_select"] = {
            "ms_per_step": round(f_ms, 5),
            "GB/s": round(f_bytes / (f_ms / 1e3) / 1e9, 1),
            "frac_of_peak": round(f_bytes / (f_ms / 1e3) / 1e9 / peak, 4),
            "rows_per_s": round(bench.rows / (f_ms / 1e3), 1),
            "launches_per_step": bench.ws,
            "note": "icp_score_select: scorer bytes without the plane write, plus Top16 "
                    "output; no score plane"}
        line["step_ms_scorer_with_pdl"] = round(
            timed_step_with_scorer_pdl(bench, args.steps, args.warmup, local), 5)
        e2e_s, bi, bo = bench.e2e(args.steps, max(args.warmup, 3))
        e2e_s = max_over_ranks(dist, e2e_s, device)
        line["e2e"] = {"value": round(n * bench.step_bytes / e2e_s / 1e9, 2), "unit": UNIT,
                       "h2d_bytes_per_step": bi, "d2h_bytes_per_step": bo,
                       "note": "per-step inputs (queries, block table, seq_lens, "
                               "num_valid_pages) from pinned host memory and the merged Top16 "
                               "read back, on two copy streams overlapping the neighbouring "
                               "steps (double-buffered); eager API calls; the index-K cache "
                               "stays resident in HBM"}
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        budget = float(os.environ.get("ICP_CPU_BASELINE_SECONDS", "10"))
        if spec_name == "select":
            s, b, r, nreq = oracle_select_sample(bench, budget)
            sample = f"first {nreq} token rows x 4 heads of the plane"
        elif spec_name == "prefill":
            s, b, r, nreq = oracle_prefill_sample(bench, budget)
            sample = f"first {nreq} tokens of request 0's chunk, full chain"
        else:
            s, b, r, nreq = oracle_sample(bench, budget)
            sample = f"first {nreq} requests of the batch, full chain"
        single = {"value": round(b / s / 1e9, 5), "unit": UNIT, "cores": 1, "kind": "oracle",
                  "sample": sample, "rows_per_s": round(r / s, 2), "seconds": round(s, 2)}
        line["cpu_baseline"] = single
        if spec_name not in ("select", "prefill"):
            # the same chain over the requests, one spawned process per core
            par = OracleParallel(bench)
            try:
                pw, pb, pr, pn = par.sample(budget, s / nreq)
            finally:
                par.close()
            line["cpu_baseline"] = {
                "value": round(pb / pw / 1e9, 5), "unit": UNIT, "cores": par.cores,
                "kind": "oracle",
                "sample": f"first {pn} requests of the batch, full chain, one spawned "
                          f"process per core over the requests",
                "rows_per_s": round(pr / pw, 2), "seconds": round(pw, 2),
                "single_thread": single}
    if ws == 1 and spec_name == "multitoken" and not args.batch and not args.no_workloads:
        # every other workload as a short device-timed record (no CPU baseline)
        del bench
        torch.cuda.empty_cache()
        line["workloads"] = {
            w: workload_record(w, args.steps, args.warmup, local, peak, peak_kind, digest)
            for w in RECORD_WORKLOADS}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()
    return 0


def main(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default="multitoken",
                    choices=["tiny", "batched", "multitoken", "sharded", "longctx", "select",
                             "prefill"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-workloads", action="store_true",
                    help="leave out the records of the other workloads")
    ap.add_argument("--batch", type=int, default=0,
                    help="use only the first B requests (smaller profiling cases)")
    args = ap.parse_args(argv)
    if args.impl == "reference":
        return run_reference(args, args.workload)
    return run_ours(args, args.workload)


if __name__ == "__main__":
    sys.exit(main())
