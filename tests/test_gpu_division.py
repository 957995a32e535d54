"""The 1x128 block quantiser divides by each block's scale with five FMA-type
instructions from its reciprocal (Markstein's corrections) instead of CUDA's
IEEE division, and its codes must match the IEEE quotient's bit for bit; this
test builds tests/c/div_check.cu with nvcc and checks on about 67 million
quotients (dividends and divisors over the whole normal range) that the two
agree bit for bit within the stated domain and that tiny dividends give
quotients every FP8 format rounds to zero."""
import os
import subprocess

import pytest

from normalization_rmsnorm_fwd_gb300 import build as nbuild

pytestmark = pytest.mark.gpu
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_division_matches_ieee(tmp_path):
    exe = os.path.join(tmp_path, "div_check")
    subprocess.run([nbuild._nvcc(), *nbuild.ARCH, "-O3", "-std=c++17", "-I", nbuild.CSRC,
                    "-I", nbuild.INCLUDE, os.path.join(ROOT, "tests", "c", "div_check.cu"),
                    "-o", exe], check=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "mismatches 0 tiny_violations 0" in r.stdout, r.stdout
