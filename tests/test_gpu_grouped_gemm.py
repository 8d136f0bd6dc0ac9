"""GPU parity of the grouped (mixture-of-experts) NVFP4 GEMM against the
oracle, group by group: each group's rows times its own expert's weight, its
own alpha and bias, at the GEMM tolerance (max|err| <= 2e-2 rms, relative
Frobenius error <= 5e-3).  Rows in 128-row bands past the last group offset
must be left untouched; empty groups contribute nothing."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_gemm_close, bf16_to_f64, nv, require_library, sample_indices, syn, tile_edges

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return require_library()


def _run(group_m, k, n, seed, bias=True, extra_bands=1, max_rows_checked=64):
    g_count = len(group_m)
    padded = [(m + 127) // 128 * 128 for m in group_m]
    offsets = np.concatenate([[0], np.cumsum(padded)]).astype(np.int32)
    rows = int(offsets[-1]) + 128 * extra_bands
    x = torch.zeros((rows, k), dtype=torch.bfloat16)
    for g, m in enumerate(group_m):
        if m:
            x[offsets[g]:offsets[g] + m] = syn.bf16_outlier_channels(m, k, seed + g)
    gs_x = syn.global_scale(x)
    kp = nv.padded_k(k)
    cp = nv.scale_shape(n, k)[1]
    w_fp4 = torch.empty((g_count * n, kp // 2), dtype=torch.uint8, device="cuda")
    w_sf = torch.empty(nv.nvfp4_scale_bytes(g_count * n, k), dtype=torch.uint8, device="cuda")
    ws, gs_w = [], []
    for g in range(g_count):
        w = syn.bf16_normal((n, k), 0.02, seed + 100 + g)
        ws.append(w)
        gs_w.append(syn.global_scale(w))
        nv.nvfp4_prepare_weight(w.cuda(), n, k, k, torch.tensor([gs_w[g]], device="cuda"),
                                w_fp4[g * n:(g + 1) * n], w_sf[g * n * cp:(g + 1) * n * cp])
    alphas = [syn.alpha_of(gs_x, gw) for gw in gs_w]
    b = syn.bf16_normal((g_count * n,), 0.1, seed + 300) if bias else None
    a_fp4, a_sf = nv.quant_act(x.cuda(), torch.tensor([gs_x], device="cuda"))
    out = torch.full((rows, n), -5.0, dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_grouped_gemm(a_fp4, a_sf, rows, torch.from_numpy(offsets).cuda(), g_count, w_fp4, w_sf, n, k,
                          torch.tensor(alphas, dtype=torch.float32, device="cuda"), b.cuda() if bias else None, out, n)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    outc = bf16_to_f64(out)
    for g, m in enumerate(group_m):
        if m == 0:
            continue
        r = np.arange(m) if m <= max_rows_checked else sample_indices(m, max_rows_checked, seed + g,
                                                                   must=tile_edges(m, 128))
        cols = np.arange(n) if n <= 512 else sample_indices(n, 384, seed + g, must=tile_edges(n, 128))
        qa, sa = oracle.quantize(syn.bf16_bits(x[offsets[g] + torch.from_numpy(r)]), gs_x, k=k)
        qb, sb = oracle.quantize(syn.bf16_bits(ws[g][torch.from_numpy(cols)]), gs_w[g], k=k)
        bb = syn.bf16_bits(b[g * n + torch.from_numpy(cols)]) if bias else None
        ref = oracle.gemm(qa, sa, qb, sb, alphas[g], bb)
        assert_gemm_close(outc[offsets[g] + r][:, cols], ref, f"group {g} (m = {m})")
    assert (outc[int(offsets[-1]):] == -5.0).all(), "rows past the last group were written"


def test_grouped_gemm_ragged_groups():
    """Six experts, an empty group, groups of 1, 37, 128, 300 and 513 rows,
    ragged K (4104: padded to 4128), bias, one unused band at the end."""
    _run([0, 37, 128, 300, 1, 513], 4104, 384, seed=7100)


def test_grouped_gemm_moe_sized():
    """Eight experts of 1536 output columns over K = 2048 with about 1000
    tokens each (the size of a prefill batch routed top-2 over 8 experts)."""
    _run([1000, 1200, 880, 1024, 1111, 960, 1030, 990], 2048, 1536, seed=7200, bias=False)


def test_grouped_gemm_single_group_equals_dense_gemm():
    """With one group the grouped GEMM is the dense GEMM on the one-CTA kernel:
    bit-identical to nvfp4_gemm_ex forced onto that kernel."""
    m, k, n = 300, 1024, 512
    x = syn.bf16_normal((384, k), 1.0, 7300)
    x[m:] = 0
    w = syn.bf16_normal((n, k), 0.02, 7301)
    gs_x, gs_w = syn.global_scale(x), syn.global_scale(w)
    a_fp4, a_sf = nv.quant_act(x.cuda(), torch.tensor([gs_x], device="cuda"))
    w_fp4, w_sf = nv.prepare_weight(w.cuda(), torch.tensor([gs_w], device="cuda"))
    alpha = torch.tensor([syn.alpha_of(gs_x, gs_w)], dtype=torch.float32, device="cuda")
    out_g = torch.empty((384, n), dtype=torch.bfloat16, device="cuda")
    out_d = torch.empty((384, n), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_grouped_gemm(a_fp4, a_sf, 384, torch.tensor([0, 384], dtype=torch.int32, device="cuda"), 1, w_fp4,
                          w_sf, n, k, alpha, None, out_g, n)
    nv.nvfp4_gemm_ex(a_fp4, a_sf, 384, w_fp4, w_sf, n, n, k, alpha, None, out_d, n, kernel=1)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    assert torch.equal(out_g.view(torch.int16), out_d.view(torch.int16))


def test_grouped_gemm_rejects_bad_arguments():
    a = torch.zeros((128, 32), dtype=torch.uint8, device="cuda")
    sf = torch.zeros(nv.nvfp4_scale_bytes(128, 64), dtype=torch.uint8, device="cuda")
    off = torch.tensor([0, 128], dtype=torch.int32, device="cuda")
    out = torch.empty((128, 192), dtype=torch.bfloat16, device="cuda")
    one = torch.ones(1, dtype=torch.float32, device="cuda")
    with pytest.raises(nv.Nvfp4Error) as e:                  # n not a multiple of 128
        nv.nvfp4_grouped_gemm(a, sf, 128, off, 1, a, sf, 192, 64, one, None, out, 192)
    assert e.value.status == 1
    with pytest.raises(nv.Nvfp4Error) as e:                  # no groups
        nv.nvfp4_grouped_gemm(a, sf, 128, off, 0, a, sf, 128, 64, one, None, out, 192)
    assert e.value.status == 1
