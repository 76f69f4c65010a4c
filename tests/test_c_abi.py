"""The C ABI from a C11 program (no GPU): include/treewy.h compiles as plain
C, the program links against the built library and the declared entry points
answer host-side validation (tests/c/abi_from_c.c)."""
import os
import shutil
import subprocess

import pytest

from gdn_speculative_tree_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_c_client_compiles_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    try:
        nvcc = build.nvcc_path()
    except RuntimeError:
        pytest.skip("no CUDA toolkit")
    lib = build.build()
    cuda_inc = os.path.join(os.path.dirname(os.path.dirname(os.path.realpath(nvcc))), "include")
    exe = str(tmp_path / "abi_from_c")
    cmd = [cc, "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), "-I", cuda_inc,
           os.path.join(HERE, "c", "abi_from_c.c"), lib, "-Wl,-rpath," + os.path.dirname(lib),
           "-o", exe]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert run.returncode == 0, run.stderr
    assert "c abi ok" in run.stdout
