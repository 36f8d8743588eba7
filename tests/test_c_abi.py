"""The boundary from plain C: tests/c_abi/abi_check.c includes only
include/gmlp.h (C11, no C++ or CUDA headers), links libgmlp.so and runs the
calls that need no GPU (CPU)."""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c11_client_compiles_links_and_runs(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("no C compiler")
    from mxfp8_nvfp4_block_gb300 import build
    lib = build.build()
    exe = tmp_path / "abi_check"
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
                    os.path.join(ROOT, "tests", "c_abi", "abi_check.c"), "-o", str(exe),
                    "-L", os.path.dirname(lib), "-lgmlp", "-Wl,-rpath," + os.path.dirname(lib)],
                   check=True, capture_output=True, text=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True, timeout=60)
    assert res.returncode == 0 and res.stdout.strip() == "ok", res.stdout + res.stderr
