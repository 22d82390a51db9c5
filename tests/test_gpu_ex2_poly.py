"""The forward kernel's polynomial 2^x (ex2_poly_x2 in cfa_ptx.cuh).

Part of a row's exponentials runs on the FMA pipe instead of the special
function unit: Cody and Waite's argument reduction and a degree-3 polynomial
fitted to 2^f on [-1/2, 1/2].  tests/native/ex2_poly_check.cu evaluates it on
the GPU over a dense sweep of [-140, 9] and special values, and checks it
against 2^x in double precision (relative error below 1e-4 on [-125, 9]) and
the underflow tail below -125 (a finite value no larger than 2^-124).
"""
import os
import shutil
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "tests", "native", "ex2_poly_check.cu")
INC = os.path.join(ROOT, "frozen_prefix_chunk_gb300", "csrc")


@pytest.mark.gpu
def test_ex2_poly_matches_exp2(tmp_path):
    from frozen_prefix_chunk_gb300 import build as B
    exe = str(tmp_path / "ex2_poly_check")
    subprocess.check_call([B.nvcc(), *B.ARCH, "-O3", "-std=c++17", "-I", INC, SRC, "-o", exe])
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    print(r.stdout)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "bad 0" in r.stdout
