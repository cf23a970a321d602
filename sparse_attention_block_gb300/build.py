"""Builds libicp.so (the CUDA library behind include/icp.h) in-tree.

Every translation unit is compiled for sm_103a only, in parallel, then linked
into ``sparse_attention_block_gb300/_lib/libicp.so`` with the CUDA runtime
linked statically (the library needs no libcuda at load time; it reaches the
driver through the runtime's entry-point query).

``timeline=True`` builds ``_lib/libicp_timeline.so`` instead: the same
library compiled with ICP_TIMELINE, whose scorer records globaltimer stamps
of its phases per CTA and which also exports icp_timeline_read
(include/icp_timeline.h).  It is a measurement build, loaded only by
``sparse_attention_block_gb300.timeline``.

    python -m sparse_attention_block_gb300.build [--force] [--timeline]
"""
from __future__ import annotations

import concurrent.futures as cf
import os
import shutil
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(HERE, "_lib")
LIB_PATH = os.path.join(OUT_DIR, "libicp.so")
TIMELINE_LIB_PATH = os.path.join(OUT_DIR, "libicp_timeline.so")
OBJ_DIR = os.path.join(ROOT, "_build", "icp")

ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC", "-Xcompiler", "-Wall",
              "-I" + INCLUDE, "-I" + CSRC]


def _nvcc() -> str:
    cand = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(cand):
        raise RuntimeError("nvcc not found; the ICP library needs the CUDA 13 toolkit")
    return cand


def sources():
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def _inputs():
    deps = sources() + [os.path.join(CSRC, f) for f in os.listdir(CSRC)
                        if f.endswith((".cuh", ".h"))]
    deps.append(os.path.join(INCLUDE, "icp.h"))
    deps.append(os.path.abspath(__file__))
    return deps


def up_to_date(lib_path: str = LIB_PATH) -> bool:
    if not os.path.exists(lib_path):
        return False
    t = os.path.getmtime(lib_path)
    return all(os.path.getmtime(d) <= t for d in _inputs())


def build(force: bool = False, verbose: bool = False, timeline: bool = False) -> str:
    lib_path = TIMELINE_LIB_PATH if timeline else LIB_PATH
    obj_dir = OBJ_DIR + ("_timeline" if timeline else "")
    extra = ["-DICP_TIMELINE"] if timeline else []
    if not force and up_to_date(lib_path):
        return lib_path
    nvcc = _nvcc()
    os.makedirs(obj_dir, exist_ok=True)
    os.makedirs(OUT_DIR, exist_ok=True)

    def compile_one(src):
        obj = os.path.join(obj_dir, os.path.basename(src)[:-3] + ".o")
        cmd = [nvcc, *ARCH, *NVCC_FLAGS, *extra, "-c", src, "-o", obj]
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed on {src}:\n{r.stdout}\n{r.stderr}")
        if verbose and (r.stdout or r.stderr):
            print(r.stdout + r.stderr, file=sys.stderr)
        return obj

    with cf.ThreadPoolExecutor(max_workers=min(8, os.cpu_count() or 1)) as ex:
        objs = list(ex.map(compile_one, sources()))
    # export the C ABI only; the static CUDA runtime stays private to the library
    vmap = os.path.join(obj_dir, "icp.map")
    with open(vmap, "w") as f:
        f.write("{ global: icp_*; local: *; };\n")
    tmp = lib_path + f".tmp{os.getpid()}"
    cmd = [nvcc, *ARCH, "-shared", "-cudart", "static", "-Xlinker", "--version-script=" + vmap,
           "-o", tmp, *objs]
    r = subprocess.run(cmd, capture_output=True, text=True)
    if r.returncode != 0:
        raise RuntimeError(f"link failed:\n{r.stdout}\n{r.stderr}")
    os.replace(tmp, lib_path)
    return lib_path


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose=True, timeline="--timeline" in sys.argv))
