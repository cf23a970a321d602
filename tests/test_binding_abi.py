"""The ctypes binding declares every entry point exactly as include/icp.h
does: same parameter count, and for each position a pointer, a 32-bit int,
an int64_t or a size_t where the header has one, and the same return type.
A binding that drifts from the header would pass truncated or shifted
arguments to the library, so this is checked on the CPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "icp.h")


def _ctype(decl: str):
    decl = decl.strip()
    if "*" in decl:
        return ctypes.c_void_p
    base = decl.rsplit(None, 1)[0] if " " in decl else decl
    base = base.replace("const", "").strip()
    return {"int": ctypes.c_int, "int32_t": ctypes.c_int32, "int64_t": ctypes.c_int64,
            "size_t": ctypes.c_size_t}[base]


def _prototypes():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    out = {}
    for ret, name, params in re.findall(
            r"^\s*((?:const\s+)?\w+\s*\*?)\s*(icp_\w+)\s*\(([^)]*)\)\s*;", text, flags=re.M | re.S):
        out[name] = (ret.strip(), [p for p in params.split(",") if p.strip()])
    return out


@pytest.fixture(scope="module")
def binding():
    from sparse_attention_block_gb300 import build
    build.build()
    from sparse_attention_block_gb300 import icp
    return icp


def test_header_parses_into_every_entry_point():
    protos = _prototypes()
    assert len(protos) == 16, sorted(protos)
    assert "icp_score" in protos and len(protos["icp_score"][1]) == 17


def test_binding_matches_the_header(binding):
    for name, (ret, params) in _prototypes().items():
        fn = getattr(binding.lib, name)
        assert fn.argtypes is not None, f"{name}: no argtypes"
        want = [_ctype(p) for p in params]
        got = list(fn.argtypes)
        assert len(got) == len(want), f"{name}: {len(got)} arguments, header has {len(want)}"
        for i, (g, w) in enumerate(zip(got, want)):
            assert ctypes.sizeof(g) == ctypes.sizeof(w) and (g is ctypes.c_void_p) == \
                (w is ctypes.c_void_p), f"{name} argument {i}: {g} vs {w} ({params[i].strip()})"
        if ret == "const char *" or ret == "const char*":
            assert fn.restype is ctypes.c_char_p, name
        else:
            assert ctypes.sizeof(fn.restype) == ctypes.sizeof(_ctype(ret + " r")), name


class _FakeTensor:
    """Just what the binding's device and row checks look at."""

    def __init__(self, device_index, rows):
        self._index = device_index
        self.device = f"cuda:{device_index}"
        self.shape = (rows,)

    def get_device(self):
        return self._index


def test_device_and_row_checks(binding, monkeypatch):
    import torch
    monkeypatch.setattr(torch.cuda, "current_device", lambda: 1)
    binding._on_current_device(_FakeTensor(1, 4), None, _FakeTensor(1, 2))
    with pytest.raises(ValueError, match="current device is cuda:1"):
        binding._on_current_device(_FakeTensor(1, 4), _FakeTensor(0, 4))
    binding._rows_at_least(_FakeTensor(1, 5), 5, "num_valid_pages")
    with pytest.raises(ValueError, match="the call reads 6"):
        binding._rows_at_least(_FakeTensor(1, 5), 6, "num_valid_pages")


def test_error_counter_maps_to_the_timeout_status(binding):
    import torch
    binding.icp_check_errors(torch.zeros(1, dtype=torch.int32))
    with pytest.raises(binding.IcpError) as e:
        binding.icp_check_errors(torch.tensor([2], dtype=torch.int32), "icp_merge")
    assert e.value.status == binding.ERR_TIMEOUT
    assert "icp_merge" in str(e.value) and "timed out" in str(e.value)


def test_binding_constants_equal_the_header_defines(binding):
    # the binding keeps its own copies of the header's sizes and limits
    text = open(HEADER).read()
    defines = {m.group(1): m.group(2) for m in
               re.finditer(r"^#define\s+(ICP_\w+)\s+(.+?)\s*(?:/\*.*)?$", text, flags=re.M)}

    def value(name):
        return int(eval(re.sub(r"(\d+)u\b", r"\1", defines[name])))

    assert binding.NOALLOC_SCRATCH_BYTES == value("ICP_NOALLOC_SCRATCH_BYTES")
    assert (binding.HEADS, binding.DIM, binding.TOPK, binding.ROW_WORDS) == tuple(
        value(n) for n in ("ICP_HEADS", "ICP_DIM", "ICP_TOPK", "ICP_ROW_WORDS"))
    assert (binding.MAX_COLS, binding.MAX_K, binding.MAX_BATCH) == tuple(
        value(n) for n in ("ICP_MAX_COLS", "ICP_MAX_K", "ICP_MAX_BATCH"))
    assert (binding.OK, binding.ERR_INVALID_ARG, binding.ERR_CUDA, binding.ERR_UNSUPPORTED,
            binding.ERR_TIMEOUT) == tuple(value(n) for n in (
                "ICP_OK", "ICP_ERR_INVALID_ARG", "ICP_ERR_CUDA", "ICP_ERR_UNSUPPORTED",
                "ICP_ERR_TIMEOUT"))


def test_noalloc_batch_limits_in_the_header_hold(binding):
    # the header lists the largest batch the fixed scratch takes per query length
    text = open(HEADER).read()
    m = re.search(r"allows at most\s+([\d, ]+?)\s*or\s*(\d+)\s+requests", text.replace("*", " "))
    stated = [int(x) for x in m.group(1).replace(",", " ").split()] + [int(m.group(2))]
    assert len(stated) == 8
    lim = binding.NOALLOC_SCRATCH_BYTES
    for dql, B in enumerate(stated, start=1):
        assert 0 < binding.icp_score_select_workspace_bytes(B, dql) <= lim
        assert binding.icp_score_select_workspace_bytes(B + 1, dql) > lim
