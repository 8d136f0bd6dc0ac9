"""Parity of the one-CTA GEMM kernel at m > 128, where the library itself uses
the CTA-pair kernel (tcgen05 cta_group::2): nvfp4_gemm_ex with kernel = 1 runs
it on several 128-row bands, and kernel = 2 forces the pair kernel, so both
stay checked against the oracle at every size."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import (assert_gemm_close, bf16_to_f64, dev_scalar, nv, require_library, sample_indices, syn,
                      tile_edges)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return require_library()


CASES = [syn.Problem("one-cta", f"m{m}-k{k}-n{n}", m, k, n, seed=5100 + i, bias=bias, n_out=n_out)
         for i, (m, k, n, n_out, bias) in enumerate([
             (1024, 4096, 6144, None, False),      # Llama qkv, prefill size
             (8192, 4096, 28672, None, False),     # Llama gate_up, full size
             (1024, 4104, 11008, 10944, True),     # padded K, bias, output slice
             (300, 5128, 640, None, True),         # ragged rows and K
             (129, 64, 256, 200, False),           # one K stage, a second row band of one row
         ])]


@pytest.mark.parametrize("p", CASES, ids=[p.name for p in CASES])
def test_one_cta_and_pair_kernels_match_the_oracle(p):
    L = syn.make_layer(p, device="cuda")
    m, k, n_out = p.m, p.k, p.n_keep
    a_fp4, a_sf = nv.quant_act(L.x, dev_scalar(L.gs_x))
    w_fp4, w_sf = nv.prepare_weight(L.w, dev_scalar(L.gs_w))
    alpha = dev_scalar(L.alpha)
    ldo = (n_out + 7) // 8 * 8
    outs = []
    for kernel in (1, 2):
        out = torch.full((m, ldo), float("nan"), dtype=torch.bfloat16, device="cuda")
        nv.nvfp4_gemm_ex(a_fp4, a_sf, m, w_fp4, w_sf, p.n, n_out, k, alpha, L.bias, out, ldo, kernel=kernel)
        torch.cuda.synchronize()
        nv.nvfp4_device_error()
        outs.append(out[:, :n_out])
    rows = np.arange(m) if m <= 160 else sample_indices(m, 48, p.seed, must=tile_edges(m, 128))
    cols = np.arange(n_out) if n_out <= 300 else sample_indices(n_out, 300, p.seed + 1, must=tile_edges(n_out, 128))
    ri, ci = torch.from_numpy(rows).cuda(), torch.from_numpy(cols).cuda()
    a, sa = oracle.quantize(syn.bf16_bits(L.x[ri]), L.gs_x, k=k)
    b, sb = oracle.quantize(syn.bf16_bits(L.w[ci]), L.gs_w, k=k)
    ref = oracle.gemm(a, sa, b, sb, L.alpha, syn.bf16_bits(L.bias[ci]) if L.bias is not None else None)
    for kernel, out in zip((1, 2), outs):
        assert_gemm_close(bf16_to_f64(out[ri][:, ci]), ref, f"kernel {kernel} {p.name}")


def test_gemm_ex_rejects_bad_choices():
    x = torch.zeros((64, 32), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(nv.nvfp4_scale_bytes(64, 64), dtype=torch.uint8, device="cuda")
    out = torch.empty((64, 64), dtype=torch.bfloat16, device="cuda")
    one = dev_scalar(1.0)
    for kw in (dict(kernel=4), dict(kernel=-1), dict(kernel=2), dict(wait_limit_ns=5), dict(drill=2)):
        with pytest.raises(nv.Nvfp4Error) as e:
            nv.nvfp4_gemm_ex(x, sf, 64, x, sf, 64, 64, 64, one, None, out, 64, **kw)
        assert e.value.status == 1, kw
