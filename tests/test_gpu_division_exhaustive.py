"""Exhaustive proof on the GPU that the quantizer's fast per-element arithmetic (per-row
reciprocal + Markstein correction, then a magic add for rint and the bias) equals IEEE float32
division followed by round-half-even and the clamp, for every finite fp16 value and every positive
fp16 scale.  The checking kernel (tests/cuda/division_check.cu) includes the library's own device
function, so what is proven is the code the quantize kernel runs."""
import ctypes
import os
import subprocess

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu


def test_fast_quotient_and_fields_match_ieee_division_exhaustively(kvq, cuda_dev):
    src = os.path.join(ROOT, "tests", "cuda", "division_check.cu")
    out_dir = os.path.join(ROOT, "tests", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "division_check.so")
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "paged_kv_cache_fp16_gb300", "csrc"),
           "-I", os.path.join(ROOT, "include"), src, "-o", so]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    bad = (ctypes.c_ulonglong * 5)()
    assert lib.run_division_check(bad) == 0
    assert list(bad) == [0] * 5, f"mismatches quotient/q8/q6/q4/row-scale: {list(bad)}"
