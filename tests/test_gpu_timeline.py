"""The timeline build of the library (compiled with ICP_TIMELINE, for
measurement) scores exactly like the ordinary build, and the stamps it
records come in the order of the scorer's phases.

The timeline build runs in a subprocess (one process loads one build of the
library); it writes its plane and stamps to files that this test compares
with the ordinary library's plane on the same inputs.
"""
import os
import subprocess
import sys

import numpy as np
import pytest
import torch

from sparse_attention_block_gb300 import workloads as W

from gpu_util import gpu_score

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SPEC = W.DecodeSpec("timeline", batch=40, page_size=256, world_size=1, decode_query_len=3,
                    max_decode_query_len=4, init_blocks=1, local_blocks=2,
                    seq_range=(300, 40000))

CHILD = r"""
import os, sys
import numpy as np, torch
sys.path.insert(0, sys.argv[1])
from sparse_attention_block_gb300 import build
os.environ["ICP_LIBRARY"] = build.build(timeline=True)
import ctypes
from sparse_attention_block_gb300 import icp, workloads as W
sys.path.insert(0, os.path.join(sys.argv[1], "tests"))
import test_gpu_timeline as T
from gpu_util import gpu_score
inp = W.make_decode_inputs(T.SPEC, seed=7)
q, k, bt, sl = (x.cuda() for x in (inp.index_q, inp.index_k, inp.block_table, inp.seq_lens))
cols = W.columns_for(T.SPEC, int(inp.seq_lens.max()))
read = icp.lib.icp_timeline_read
read.restype = ctypes.c_int
read.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
sms = torch.cuda.get_device_properties(0).multi_processor_count
stamps = np.zeros((sms, 24), np.uint64)
assert read(stamps.ctypes.data, sms, 1) == 0
errors = torch.zeros(1, dtype=torch.int32, device="cuda")
plane = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=256, dql=3,
                  maxdql=4, errors=errors)
torch.cuda.synchronize()
assert read(stamps.ctypes.data, sms, 0) == 0
assert int(errors.item()) == 0
np.save(sys.argv[2], plane.cpu().numpy())
np.save(sys.argv[3], stamps)
"""


def test_timeline_build_scores_like_the_library_and_stamps_its_phases(tmp_path):
    plane_file, stamp_file = str(tmp_path / "plane.npy"), str(tmp_path / "stamps.npy")
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT, plane_file, stamp_file],
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-3000:]
    inp = W.make_decode_inputs(SPEC, seed=7)
    q, k, bt, sl = (x.cuda() for x in (inp.index_q, inp.index_k, inp.block_table, inp.seq_lens))
    cols = W.columns_for(SPEC, int(inp.seq_lens.max()))
    plane = gpu_score(q, k, bt, sl, cols=cols, rank=0, world_size=1, page_size=256, dql=3,
                      maxdql=4)
    torch.cuda.synchronize()
    timeline_plane = np.load(plane_file)
    assert np.array_equal(plane.cpu().numpy().view(np.int32), timeline_plane.view(np.int32))
    st = np.load(stamp_file).astype(np.int64)
    worked = st[:, 2] > 0                  # CTAs that issued an index-K load
    assert worked.sum() > 0
    s = st[worked]
    # entry <= set-up done <= first load <= last load <= first MMA commit
    # <= last MMA commit <= CTA exit, and the first tile is finished after
    # its MMAs are committed
    for a, b in [(0, 1), (1, 2), (2, 3), (2, 4), (4, 5), (5, 11), (3, 11)]:
        assert np.all(s[:, a] <= s[:, b]), (a, b)
    assert np.all(s[:, 11] - s[:, 0] < 10_000_000)  # under 10 ms from entry to exit
