"""The bounded-wait failure path, without a GPU fault: every pipeline barrier
wait of the GEMM kernels gives up after a limit, sets the device error flag
and lets the launch end.  nvfp4_gemm_ex's timeout drill makes the kernel's
copy producers issue nothing, so the waits on data that never arrives run out
(a flag nothing sets); the call must come back within the limit,
nvfp4_device_error() must report NVFP4_ERR_TIMEOUT once and then be clear,
nothing may have been stored, and a normal call right after must pass oracle
parity."""
import time

import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_gemm_close, bf16_to_f64, dev_scalar, nv, require_library, syn

pytestmark = pytest.mark.gpu

LIMIT_NS = 20_000_000            # 20 ms per wait


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return require_library()


@pytest.mark.parametrize("kernel,m", [(1, 64), (1, 300), (2, 300)], ids=["one-cta-m64", "one-cta-m300", "pair-m300"])
def test_wait_timeout_is_reported_and_the_next_call_is_clean(kernel, m):
    k, n = 512, 512
    x = syn.bf16_normal((m, k), 1.0, 9100 + m)
    w = syn.bf16_normal((n, k), 0.02, 9101)
    b = syn.bf16_normal((n,), 0.1, 9102)
    gs_x, gs_w = syn.global_scale(x), syn.global_scale(w)
    alpha = syn.alpha_of(gs_x, gs_w)
    a_fp4, a_sf = nv.quant_act(x.cuda(), dev_scalar(gs_x))
    w_fp4, w_sf = nv.prepare_weight(w.cuda(), dev_scalar(gs_w))
    torch.cuda.synchronize()
    nv.nvfp4_device_error()                                    # start clean

    out = torch.full((m, n), -3.0, dtype=torch.bfloat16, device="cuda")
    t0 = time.perf_counter()
    nv.nvfp4_gemm_ex(a_fp4, a_sf, m, w_fp4, w_sf, n, n, k, dev_scalar(alpha), b.cuda(), out, n, kernel=kernel,
                     wait_limit_ns=LIMIT_NS, drill=1)
    torch.cuda.synchronize()
    elapsed = time.perf_counter() - t0
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_device_error()
    assert e.value.status == 6, str(e.value)                  # NVFP4_ERR_TIMEOUT
    nv.nvfp4_device_error()                                    # read and cleared: now clean
    assert elapsed < 5.0, f"the drill took {elapsed:.2f} s for {LIMIT_NS / 1e6:.0f} ms waits"
    assert bool((out == -3.0).all()), "the drill stored output"

    nv.nvfp4_gemm_ex(a_fp4, a_sf, m, w_fp4, w_sf, n, n, k, dev_scalar(alpha), b.cuda(), out, n, kernel=kernel)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    qa, sa = oracle.quantize(syn.bf16_bits(x), gs_x, k=k)
    qb, sb = oracle.quantize(syn.bf16_bits(w), gs_w, k=k)
    assert_gemm_close(bf16_to_f64(out), oracle.gemm(qa, sa, qb, sb, alpha, syn.bf16_bits(b)), "after the drill")
    assert np.isfinite(bf16_to_f64(out)).all()
