"""The C ABI from C (CPU only): tests/c/abi_host.c, compiled as C99 with warnings as errors
against include/moe_gb300.h and linked with the built library, runs its host-only checks."""
import os
import shutil
import subprocess

import pytest

from quantized_grouped_gemm_router_gb300 import build as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_c_client_links_and_runs(tmp_path):
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    lib = B.build()
    exe = str(tmp_path / "abi_host")
    cmd = [cc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", os.path.join(ROOT, "include"),
           os.path.join(ROOT, "tests", "c", "abi_host.c"), "-o", exe, lib, "-Wl,-rpath," + os.path.dirname(lib)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert run.returncode == 0, run.stderr
    assert "c abi ok" in run.stdout
