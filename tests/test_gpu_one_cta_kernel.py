"""Parity of the one-CTA GEMM kernel at m > 128, where the library normally
uses the CTA-pair kernel (tcgen05 cta_group::2).  NVFP4_GEMM_ONE_CTA=1, set
before the library loads, keeps every GEMM on the one-CTA kernel; the GEMM and
linear tests run in a child process with that setting, so both kernels stay
checked against the oracle at every size."""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_one_cta_kernel_passes_gemm_parity():
    env = dict(os.environ, NVFP4_GEMM_ONE_CTA="1")
    cmd = [sys.executable, "-m", "pytest", "-q", "-x", "-m", "gpu", "-p", "no:cacheprovider",
           os.path.join(ROOT, "tests", "test_gpu_gemm.py"),
           os.path.join(ROOT, "tests", "test_gpu_linear.py") + "::test_llama_shapes",
           os.path.join(ROOT, "tests", "test_gpu_linear.py") + "::test_padded_shapes"]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-2000:]
