"""The C ABI from plain C: tests/c/abi_client.c is compiled with gcc against
include/crmsnorm.h, linked to libcrmsnorm.so and run (no GPU needed: it only
makes calls that return before any CUDA work)."""
import os
import shutil
import subprocess

import pytest

from normalization_rmsnorm_fwd_gb300 import build as nbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cuda_include():
    for cand in (os.environ.get("CUDA_HOME"), "/usr/local/cuda"):
        if cand and os.path.exists(os.path.join(cand, "include", "cuda_runtime_api.h")):
            return os.path.join(cand, "include")
    pytest.skip("CUDA headers not found")


def test_c_client(tmp_path):
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    lib = nbuild.build()
    exe = os.path.join(tmp_path, "abi_client")
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-I", _cuda_include(), os.path.join(ROOT, "tests", "c", "abi_client.c"),
                    "-o", exe, lib, f"-Wl,-rpath,{os.path.dirname(lib)}"], check=True)
    r = subprocess.run([exe], capture_output=True, text=True)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("ALL OK")
