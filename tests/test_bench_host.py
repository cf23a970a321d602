"""Host-side logic of bench.py, checked without a GPU.

- The algorithmic byte counts of a decode step and of a prefill window,
  worked out by hand from their definitions on small cases: index-K rows
  needed, queries, plane columns written (a request's columns padded to the
  next multiple of 4), block table entries, the select's plane read and
  published rows, the merge's reads and writes.
- The clock record: its summary of NVML samples, and which records reject a
  timing (thermal or hardware slowdown, or clocks held low with no reason).
- The ncu traffic table is keyed by a source digest and holds ratios of DRAM
  bytes to index-K bytes that cannot fall below 1 (every row is read once).
"""
import json
from types import SimpleNamespace

import bench


def _spec(ws, ps, dql):
    return SimpleNamespace(world_size=ws, page_size=ps, decode_query_len=dql)


def test_decode_bytes_unsharded_p128_by_hand():
    # seq_lens 1000, 2500 -> 8 and 20 B128 blocks (both already multiples of 4)
    score, select, merge, kbytes = bench.algorithmic_bytes(_spec(1, 128, 1), [1000, 2500], 20)
    assert kbytes == 3500 * 128
    # K rows + 2 tokens x 512 B of queries + 16 B per (token, column) + 4 B per page
    assert score == 448000 + 1024 + 16 * (8 + 20) + 4 * (8 + 20)
    # plane read + 8 rows x 132 B + nvp
    assert select == 448 + 8 * 132 + 8
    # 8 rows of 132 B read, 8 rows of 128 B written, nvp
    assert merge == 8 * 132 + 8 * 128 + 8


def test_decode_bytes_sharded_p256_by_hand():
    # world size 2 at P256: a column is a local page, ceil(1000 / 256) = 4
    score, select, merge, kbytes = bench.algorithmic_bytes(_spec(2, 256, 2), [1000], 4)
    assert kbytes == 128000                       # all shards together
    q = 2 * 2 * 512                               # every shard reads both tokens' queries
    plane = 2 * 16 * 4 * 2                        # 2 shards x 2 tokens x 4 columns x 16 B
    bt = 2 * 4 * 4                                # 2 shards x 4 pages x 4 B
    assert score == 128000 + q + plane + bt
    assert select == plane + 2 * 2 * 4 * 132 + 2 * 2 * 4
    assert merge == 2 * 2 * 4 * 132 + 2 * 4 * 128 + 2 * 4


def test_prefill_bytes_by_hand():
    score, select, merge, kbytes = bench.prefill_bytes([1000, 2500], 3, 20)
    T = 6
    plane = 16 * 3 * (8 + 20)
    assert kbytes == 448000
    assert score == 448000 + T * 512 + plane + 4 * (8 + 20)
    assert select == plane + T * 4 * 128 + T * 4
    assert merge == T * 4 * 128 * 2 + T * 4


def _sampler(samples, max_mhz=2070):
    s = object.__new__(bench.ClockSampler)
    s.ok, s.samples, s.max_mhz = True, samples, max_mhz
    return s


def test_clock_summary_takes_the_median_and_names_the_reasons():
    s = _sampler([(2070, 0x1), (1900, 0x4), (2070, 0x4 | 0x10)])
    assert s.summary() == {"sm_mhz": 2070, "sm_max_mhz": 2070,
                           "reasons": ["sw_power_cap", "sync_boost"], "samples": 3}


def test_clock_summary_without_nvml():
    s = object.__new__(bench.ClockSampler)
    s.ok, s.samples, s.max_mhz = False, [], None
    assert s.summary()["reasons"] == ["unavailable"]


def test_which_clock_records_reject_a_timing():
    rej = bench.ClockSampler.rejected
    assert not rej({"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": []})
    for r in ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown"):
        assert rej({"sm_mhz": 2070, "sm_max_mhz": 2070, "reasons": [r]})
    # a power cap explains lower clocks and is kept
    assert not rej({"sm_mhz": 1500, "sm_max_mhz": 2070, "reasons": ["sw_power_cap"]})
    # low clocks with nothing to explain them: a leftover lock
    assert rej({"sm_mhz": 1500, "sm_max_mhz": 2070, "reasons": []})
    assert rej({"sm_mhz": 1500, "sm_max_mhz": 2070, "reasons": ["applications_clocks_setting"]})
    assert not rej({"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unavailable"]})


def test_traffic_table_keys_and_ratios():
    d = bench.kernel_digest()
    assert len(d) == 16 and int(d, 16) >= 0
    for (workload, digest), ratio in bench.NCU_TRAFFIC.items():
        assert len(digest) == 16
        assert 1.0 <= ratio < 1.1, (workload, ratio)


def test_code_digest_ignores_comments_but_not_code():
    base = {"icp_score.cu": "int a; // x\n/* y */ int b;\n", "icp_fused.cuh": "f();\n",
            "icp_device.cuh": ""}
    d = bench.kernel_digest(lambda f: base[f])
    reworded = dict(base)
    reworded["icp_score.cu"] = "int a; // other words\n\n int b; /* a\n longer note */\n"
    assert bench.kernel_digest(lambda f: reworded[f]) == d
    changed = dict(base)
    changed["icp_score.cu"] = "int a; // x\n/* y */ int c;\n"
    assert bench.kernel_digest(lambda f: changed[f]) != d


def test_reference_arm_runs_the_oracle_without_the_cuda_library(tmp_path):
    # the oracle arm draws and sizes its batch itself: the product's binding
    # (and with it libicp.so) must stay unloaded
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    code = ("import json, sys, bench\n"
            "bench.main(['--impl', 'reference', '--workload', 'tiny', '--steps', '1',"
            " '--warmup', '0'])\n"
            "assert 'sparse_attention_block_gb300.icp' not in sys.modules\n"
            "assert 'libicp' not in open('/proc/self/maps').read()\n")
    env = dict(os.environ, ICP_REF_STEP_SECONDS="0.05", CUDA_VISIBLE_DEVICES="")
    r = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True,
                       text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads([ln for ln in r.stdout.splitlines() if ln.startswith("{")][-1])
    assert line["impl"] == "reference" and line["cpu_baseline"]["kind"] == "oracle"
    assert line["config"]["cols"] == 20 and "oracle" in line["config"]["step"]
