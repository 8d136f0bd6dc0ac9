"""Exhaustive check of the quantizer's division by 6 (Markstein FMA correction,
nvfp4_quantized_linear_gb300/csrc/scale_math.cuh) against IEEE division on the
GPU: the E4M3 block-scale code must agree for every non-negative float, and
the quotient itself wherever the IEEE quotient is a normal number (below
that, at x < 6 * 2^-126, every scale code is 0).  The kernel is compiled from
tests/cuda/check_div6.cu with nvcc for sm_103a."""
import ctypes
import os
import subprocess
import tempfile

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_div6_gives_the_ieee_scale_code_for_every_input():
    from nvfp4_quantized_linear_gb300 import _build
    with tempfile.TemporaryDirectory() as d:
        so = os.path.join(d, "check_div6.so")
        subprocess.check_call([_build.nvcc(), *_build.ARCH, "-O3", "-Xcompiler", "-fPIC", "-shared",
                               "-I", os.path.join(ROOT, "nvfp4_quantized_linear_gb300", "csrc"),
                               os.path.join(ROOT, "tests", "cuda", "check_div6.cu"), "-o", so])
        lib = ctypes.CDLL(so)
        counts = (ctypes.c_ulonglong * 2)()
        assert lib.run_check_div6(counts) == 0
    assert counts[0] == 0, f"{counts[0]} inputs change their E4M3 scale code"
    assert counts[1] == 0, f"{counts[1]} inputs with a normal quotient change it"
