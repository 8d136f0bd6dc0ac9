"""Exhaustive probe of the GPU's E2M1 and E4M3 encoders (the cvt .rn.satfinite
forms the quantizers use) against the oracle's encoders, which are written
from the OCP format definitions: every finite float for E2M1, both signs
(4.28e9 inputs), and every finite non-negative float for E4M3 (2.14e9; block
scales are never negative).  The kernel and the host comparison are compiled
from tests/cuda/sweep_cvt.cu with nvcc for sm_103a; the comparison calls the
oracle's own shared library."""
import ctypes
import os
import subprocess
import tempfile

import pytest

import oracle

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_hardware_encoders_match_the_oracle_for_every_finite_input():
    from nvfp4_quantized_linear_gb300 import _build
    oracle_so = oracle.build()
    with tempfile.TemporaryDirectory() as d:
        so = os.path.join(d, "sweep_cvt.so")
        subprocess.check_call([_build.nvcc(), *_build.ARCH, "-O3", "-std=c++17", "-Xcompiler", "-fPIC,-pthread",
                               "-shared", "-I", os.path.join(ROOT, "nvfp4_quantized_linear_gb300", "csrc"),
                               os.path.join(ROOT, "tests", "cuda", "sweep_cvt.cu"), "-o", so, "-ldl"])
        lib = ctypes.CDLL(so)
        counts = (ctypes.c_ulonglong * 2)()
        first = (ctypes.c_uint * 2)()
        assert lib.run_sweep(oracle_so.encode(), counts, first) == 0
    assert counts[0] == 0, f"{counts[0]} E2M1 codes differ, first at bits {first[0]:#010x}"
    assert counts[1] == 0, f"{counts[1]} E4M3 codes differ, first at bits {first[1]:#010x}"
