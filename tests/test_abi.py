"""The C ABI library loads on a machine without a GPU, exports every entry
point include/icp.h declares, and rejects bad arguments on the host before
touching CUDA (no compute call is made here)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "icp.h")


@pytest.fixture(scope="module")
def lib():
    from sparse_attention_block_gb300 import build
    return ctypes.CDLL(build.build())


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(icp_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_entry_points():
    names = declared_functions()
    for n in ["icp_score", "icp_top16_select", "icp_publish_rows", "icp_merge",
              "icp_score_select", "icp_score_select_workspace_bytes",
              "icp_score_columns", "icp_status_string"]:
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for n in declared_functions():
        assert hasattr(lib, n), n


def test_only_the_c_abi_is_exported():
    from sparse_attention_block_gb300 import build
    out = os.popen(f"nm -D --defined-only {build.LIB_PATH}").read()
    syms = [l.split()[-1] for l in out.splitlines() if " T " in l]
    assert syms and all(s.startswith("icp_") for s in syms), syms


def test_timeline_build_exports_its_reader_and_the_library_does_not():
    # the measurement build (ICP_TIMELINE) adds icp_timeline_read, declared in
    # include/icp_timeline.h; the ordinary library has no such symbol
    from sparse_attention_block_gb300 import build
    ordinary = os.popen(f"nm -D --defined-only {build.build()}").read()
    assert "icp_timeline_read" not in ordinary
    path = build.build(timeline=True)
    assert path != build.LIB_PATH
    tl = ctypes.CDLL(path)
    f = tl.icp_timeline_read
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_int]
    buf = (ctypes.c_ulonglong * 24)()
    assert f(None, 1, 0) == 1 and f(buf, -1, 0) == 1 and f(buf, 1025, 0) == 1
    for n in declared_functions():
        assert hasattr(tl, n), n


def test_score_columns_host_helper(lib):
    f = lib.icp_score_columns
    assert f(1000, 128, 1) == 8
    assert f(1_000_000, 128, 1) == 7816
    assert f(131072, 256, 1) == 1024
    assert f(131072, 256, 2) == 512
    assert f(0, 128, 4) == 4
    assert f(2_000_000, 128, 1) == -1      # beyond 8192 columns
    assert f(100, 64, 1) == -1


def test_invalid_arguments_are_rejected_before_any_launch(lib):
    P = ctypes.c_void_p
    buf = ctypes.create_string_buffer(1 << 16)
    a = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 256), P)
    lib.icp_score.argtypes = [P, P, ctypes.c_int64, P, ctypes.c_int64, P, P] + \
        [ctypes.c_int] * 8 + [P, P]
    good = dict(q=a, k=a, n=4, bt=a, st=4, sl=a, out=a, B=1, cols=8, rank=0, ws=1, ps=128,
                dql=1, maxdql=1)

    def call(**kw):
        d = dict(good, **kw)
        return lib.icp_score(d["q"], d["k"], d["n"], d["bt"], d["st"], d["sl"], d["out"], d["B"],
                             d["cols"], d["rank"], d["ws"], d["ps"], d["dql"], d["maxdql"],
                             0, None, None)
    INVALID = 1
    assert call(cols=6) == INVALID            # cols % 4 != 0
    assert call(cols=8196) == INVALID         # cols > 8192
    assert call(ps=64) == INVALID
    assert call(ws=3) == INVALID
    assert call(rank=1) == INVALID
    assert call(dql=2, maxdql=1) == INVALID
    assert call(dql=1, maxdql=9) == INVALID   # 4 * max_decode_query_len > 32
    assert call(B=-1) == INVALID
    assert call(q=ctypes.c_void_p(a.value + 8)) == INVALID   # TMA needs 16-byte alignment
    assert call(B=0) == 0                     # empty batch: nothing to do
    lib.icp_top16_select.argtypes = [P, ctypes.c_int, ctypes.c_int, P] + [ctypes.c_int] * 4 + \
        [P, P, P]
    assert lib.icp_top16_select(a, 1, 12288, a, 1, 2, 1, 0, a, a, None) == INVALID  # K >= 12288
    assert lib.icp_top16_select(a, 1, 100, a, 9, 8, 1, 0, a, a, None) == INVALID   # init+local > 16
    assert lib.icp_top16_select(a, 1, 100, a, 1, 2, 0, 0, a, a, None) == INVALID   # scale 0
    lib.icp_publish_rows.argtypes = [P, ctypes.c_int, ctypes.c_int, P, P, P] + \
        [ctypes.c_int] * 7 + [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int, P]
    # T > capacity, slot 3, hpr * ws != 4
    assert lib.icp_publish_rows(a, 5, 10, a, a, a, 0, 0, 1, 4, 4, 1, 2, 100, 1, 0, 0,
                                None) == INVALID
    assert lib.icp_publish_rows(a, 4, 10, a, a, a, 3, 0, 1, 4, 4, 1, 2, 100, 1, 0, 0,
                                None) == INVALID
    assert lib.icp_publish_rows(a, 4, 10, a, a, a, 0, 0, 2, 1, 4, 1, 2, 100, 1, 0, 1,
                                None) == INVALID
    lib.icp_status_string.restype = ctypes.c_char_p
    assert lib.icp_status_string(1) == b"invalid argument"


def test_fused_workspace_size_and_checks(lib):
    lib.icp_score_select_workspace_bytes.restype = ctypes.c_size_t
    n = lib.icp_score_select_workspace_bytes(128, 4)
    assert n >= (160 + 128) * 4 * 16 * 288
    assert lib.icp_score_select_workspace_bytes(-1, 4) == 0
    assert lib.icp_score_select_workspace_bytes(4, 9) == 0
    P = ctypes.c_void_p
    buf = ctypes.create_string_buffer(1 << 16)
    a = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 256), P)
    lib.icp_score_select.argtypes = [P, P, ctypes.c_int64, P, ctypes.c_int64, P] + \
        [ctypes.c_int] * 7 + [P, ctypes.c_int, ctypes.c_int, P, ctypes.c_size_t, P, P, P, P]
    ok = lib.icp_score_select_workspace_bytes(1, 1)
    # workspace too small / init + local > 16 / misaligned workspace
    assert lib.icp_score_select(a, a, 4, a, 4, a, 1, 8, 0, 1, 128, 1, 1, a, 1, 2, a, ok - 1,
                                a, a, None, None) == 1
    assert lib.icp_score_select(a, a, 4, a, 4, a, 1, 8, 0, 1, 128, 1, 1, a, 9, 8, a, ok,
                                a, a, None, None) == 1
    bad = ctypes.c_void_p(a.value + 16)
    assert lib.icp_score_select(a, a, 4, a, 4, a, 1, 8, 0, 1, 128, 1, 1, a, 1, 2, bad, ok,
                                a, a, None, None) == 1


def test_prefill_sizes_and_checks(lib):
    lib.icp_prefill_plan_words.restype = ctypes.c_int64
    lib.icp_prefill_plan_words.argtypes = [ctypes.c_int, ctypes.c_int]
    # ceil(T / 64) + batch records of 8 ints, plus an 8-int header
    assert lib.icp_prefill_plan_words(4, 8192) == 8 + 8 * (128 + 4)   # 64-token records
    assert lib.icp_prefill_plan_words(3, 1) == 8 + 8 * 4
    assert lib.icp_prefill_plan_words(-1, 8) == -1
    assert lib.icp_prefill_plan_words(1, 4096 * 64) == -1   # more than 4096 records
    P = ctypes.c_void_p
    buf = ctypes.create_string_buffer(1 << 16)
    a = ctypes.cast(ctypes.addressof(buf) + (-ctypes.addressof(buf) % 256), P)
    INVALID = 1
    lib.icp_prefill_plan.argtypes = [P, P, ctypes.c_int, ctypes.c_int, P, ctypes.c_int64, P, P]
    assert lib.icp_prefill_plan(a, a, 2, 65, a, 8 + 8 * 3, None, None) == INVALID  # too small
    assert lib.icp_prefill_plan(a, a, 2, 64, None, 8 + 8 * 4, None, None) == INVALID
    odd = ctypes.c_void_p(a.value + 4)                    # the plan is read as int4
    assert lib.icp_prefill_plan(a, a, 2, 64, odd, 8 + 8 * 4, None, None) == INVALID
    lib.icp_prefill_score.argtypes = [P, P, ctypes.c_int64, P, ctypes.c_int64, P, ctypes.c_int64,
                                      P] + [ctypes.c_int] * 5 + [P, P]
    assert lib.icp_prefill_score(a, a, 4, a, 4, a, 8 + 8 * 4, a, 10, 6, 0, 1, 128, None,
                                 None) == INVALID                          # cols % 4
    assert lib.icp_prefill_score(a, a, 4, a, 4, a, 8, a, 10, 8, 0, 1, 128, None,
                                 None) == INVALID                          # no record room
    lib.icp_prefill_select.argtypes = [P, ctypes.c_int, ctypes.c_int, P] + [ctypes.c_int] * 6 + \
        [P, P]
    assert lib.icp_prefill_select(a, 4, 100, a, 2, 1, 1, 2, 1, 0, a, None) == INVALID  # ws*hpr
    assert lib.icp_prefill_select(a, 4, 12288, a, 1, 4, 1, 2, 1, 0, a, None) == INVALID
    lib.icp_prefill_merge.argtypes = [P, P] + [ctypes.c_int] * 5 + [P, P, P]
    assert lib.icp_prefill_merge(a, a, 4, 3, 1, 1, 2, a, a, None) == INVALID
    assert lib.icp_prefill_merge(a, a, 4, 4, 1, 9, 8, a, a, None) == INVALID


def test_binding_fails_loudly_without_the_library(tmp_path):
    # a copy of the binding beside no _lib/libicp.so must refuse to import
    import shutil
    import subprocess
    import sys
    pkg = tmp_path / "pkg"
    pkg.mkdir()
    (pkg / "__init__.py").write_text("")
    shutil.copy(os.path.join(ROOT, "sparse_attention_block_gb300", "icp.py"), pkg / "icp.py")
    r = subprocess.run([sys.executable, "-c", "import pkg.icp"], cwd=tmp_path,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode != 0
    assert "ImportError" in r.stderr and "libicp.so is missing" in r.stderr
