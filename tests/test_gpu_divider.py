"""GPU check that the kernels' division by an invariant divisor (kvq_divu32.cuh: a multiply-high
and shifts, Granlund and Montgomery's unsigned method) equals integer division: every 32-bit
numerator for divisors the kernels meet and the extreme ones, and every divisor up to 65,536 on
numerators at each multiple scale.  The checking kernels (tests/cuda/divu32_check.cu) include
the library's own header, so what is checked is the code the kernels run."""
import ctypes
import os
import subprocess

import pytest

from conftest import ROOT

pytestmark = pytest.mark.gpu


def test_invariant_divider_matches_integer_division(kvq, cuda_dev):
    src = os.path.join(ROOT, "tests", "cuda", "divu32_check.cu")
    out_dir = os.path.join(ROOT, "tests", "_build")
    os.makedirs(out_dir, exist_ok=True)
    so = os.path.join(out_dir, "divu32_check.so")
    nvcc = os.environ.get("NVCC", "nvcc")
    cmd = [nvcc, "-gencode", "arch=compute_103a,code=sm_103a", "-O3", "-std=c++17", "-shared",
           "-Xcompiler", "-fPIC", "-I", os.path.join(ROOT, "paged_kv_cache_fp16_gb300", "csrc"),
           "-I", os.path.join(ROOT, "include"), src, "-o", so]
    subprocess.run(cmd, check=True, capture_output=True)
    lib = ctypes.CDLL(so)
    bad = (ctypes.c_ulonglong * 2)()
    assert lib.run_divu32_check(bad) == 0
    assert list(bad) == [0, 0], f"mismatches (all numerators, small divisors): {list(bad)}"
