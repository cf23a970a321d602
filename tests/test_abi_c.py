"""include/icp.h from plain C: abi_client.c is compiled as C99 with warnings
as errors, linked against libicp.so like any C program, and run.  It calls
only host paths (sizing helpers, empty calls, rejected arguments), so no GPU
is needed."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_client_builds_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    from sparse_attention_block_gb300 import build
    lib = build.build()
    libdir = os.path.dirname(lib)
    exe = str(tmp_path / "abi_client")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Wextra", "-Wpedantic", "-Werror",
                        "-I", os.path.join(ROOT, "include"), os.path.join(HERE, "abi_client.c"),
                        "-o", exe, "-L", libdir, "-l:libicp.so", f"-Wl,-rpath,{libdir}"],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0, r.stderr
    assert "abi_client: ok" in r.stdout
