"""GPU parity of the MXFP4 GEMM and linear (nvfp4_mxfp4_gemm,
nvfp4_mxfp4_linear) against the oracle's FP64 MXFP4 GEMM (reading R-mx) on
identical quantized operands, at the GEMM tolerance (max|err| <= 2e-2 rms,
relative Frobenius error <= 5e-3).

Page "B12X quantized linear backends" (vLLM PR #52016), section 实现拆解:
the MXFP4 backend quantizes the activation (flashinfer_mxfp4_quantize) and
runs mm_mxfp4.  Here the weight is quantized by the same conversion, so the
oracle's operands are its own MXFP4 quantization of the same bf16 inputs
(which the quantizer tests show to be the library's bytes)."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_gemm_close, bf16_to_f64, nv, require_library, sample_indices, syn, tile_edges

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return require_library()


def _quant(x):
    return nv.quant_act_mx(x)


def _oracle(x, w, b, k, rows, cols):
    a, sa = oracle.quantize_mx(syn.bf16_bits(x[torch.from_numpy(rows).to(x.device)].cpu()), k=k)
    bq, sb = oracle.quantize_mx(syn.bf16_bits(w[torch.from_numpy(cols).to(w.device)].cpu()), k=k)
    bb = syn.bf16_bits(b[torch.from_numpy(cols).to(b.device)].cpu()) if b is not None else None
    return oracle.gemm_mx(a, sa, bq, sb, bb)


# (m, k, n_w, n_out, bias, x kind): one-CTA (m <= 128) and CTA-pair (m > 128)
# kernels, ragged K (K % 32 != 0 and K % 64 != 0), output slices, full-size
# Llama / Qwen layer shapes (sampled rows x columns)
CASES = [
    (16, 256, 128, 128, False, "normal"),
    (1, 4096, 6144, 6144, True, "normal"),
    (97, 4104, 1024, 1000, True, "outlier"),
    (128, 5128, 512, 384, False, "student_t"),
    (300, 96, 640, 640, True, "normal"),
    (257, 4104, 11008, 10944, True, "normal"),
    (8192, 4096, 28672, 28672, False, "normal"),
    (2048, 5120, 10240, 10240, False, "outlier"),
]


@pytest.mark.parametrize("m,k,n_w,n_out,bias,kind", CASES, ids=[f"m{c[0]}-k{c[1]}-n{c[2]}-o{c[3]}" for c in CASES])
def test_mxfp4_gemm_matches_oracle(m, k, n_w, n_out, bias, kind):
    seed = 6100 + m + k + n_w
    if kind == "normal":
        x = syn.bf16_normal((m, k), 1.0, seed, device="cuda")
    elif kind == "outlier":
        x = syn.bf16_outlier_channels(m, k, seed, device="cuda")
    else:
        x = syn.bf16_student_t(m, k, 3, seed, device="cuda")
    w = syn.bf16_normal((n_w, k), 0.02, seed + 1, device="cuda")
    b = syn.bf16_normal((n_out,), 0.1, seed + 2, device="cuda") if bias else None
    a_fp4, a_sf = _quant(x)
    w_fp4, w_sf = _quant(w)
    ldo = (n_out + 7) // 8 * 8
    out = torch.full((m, ldo), float("nan"), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_mxfp4_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, b, out, ldo)
    lin = nv.mxfp4_linear(x, w_fp4, w_sf, k, n_out, bias=b)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    rows = np.arange(m) if m <= 64 else sample_indices(m, 48, seed, must=tile_edges(m, 128))
    cols = np.arange(n_out) if n_out <= 384 else sample_indices(n_out, 384, seed + 1, must=tile_edges(n_out, 128))
    ref = _oracle(x, w, b, k, rows, cols)
    assert_gemm_close(bf16_to_f64(out[:, :n_out])[rows][:, cols], ref, f"mxfp4 gemm {m}x{k}->{n_out}")
    assert_gemm_close(bf16_to_f64(lin)[rows][:, cols], ref, f"mxfp4 linear {m}x{k}->{n_out}")
    assert torch.isnan(out[:, n_out:]).all() if ldo > n_out else True


def test_mxfp4_gemm_exact_power_of_two_case_is_bit_exact():
    """Every element a grid value times a power of two per 32-block: the MXFP4
    quantization is exact, so the GEMM computes sum_k x w exactly in fp32
    (small integers) and the bf16 output equals the rounded exact product."""
    rng = np.random.default_rng(61)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    m, n, k = 200, 384, 320
    xa = rng.choice(grid, (m, k)) * rng.choice([-1, 1], (m, k))
    xw = rng.choice(grid, (n, k)) * rng.choice([-1, 1], (n, k))
    xa[:, ::32] = 6                                  # every block's maximum is 6: scale 2^0
    xw[:, ::32] = 6
    x = torch.tensor(xa, dtype=torch.float32).to(torch.bfloat16).cuda()
    w = torch.tensor(xw, dtype=torch.float32).to(torch.bfloat16).cuda()
    a_fp4, a_sf = _quant(x)
    w_fp4, w_sf = _quant(w)
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_mxfp4_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n, n, k, None, out, n)
    torch.cuda.synchronize()
    exact = torch.from_numpy(xa @ xw.T)
    assert (exact.abs() < 2 ** 22).all()
    assert torch.equal(out.cpu().view(torch.int16), exact.float().to(torch.bfloat16).view(torch.int16))


@pytest.mark.parametrize("m,k,n", [(1, 14336, 4096), (3, 4104, 1024), (8, 4096, 6144), (16, 14336, 4096),
                                   (17, 4104, 2048), (64, 4096, 2048)])
def test_mxfp4_linear_split_k_matches_unsplit(m, k, n):
    """Small m: the MXFP4 linear splits K across the CTAs of a cluster (fp32
    partials summed in shared memory), and for m <= 16 the GEMM's epilogue
    warps quantize x themselves (m = 17 and 64 run the quantizer kernel);
    against the oracle and the unsplit MXFP4 GEMM on the same quantized
    operands."""
    x = syn.bf16_normal((m, k), 1.0, 6200 + m, device="cuda")
    w = syn.bf16_normal((n, k), 0.02, 6201, device="cuda")
    w_fp4, w_sf = _quant(w)
    ws = torch.full((nv.nvfp4_mxfp4_linear_workspace_bytes(m, k, n),), 0xA5, dtype=torch.uint8, device="cuda")
    lin = nv.mxfp4_linear(x, w_fp4, w_sf, k, n, workspace=ws)
    a_fp4, a_sf = _quant(x)
    unsplit = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_mxfp4_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n, n, k, None, unsplit, n)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    rows = np.arange(m)
    cols = sample_indices(n, 384, 6202, must=tile_edges(n, 128))
    ref = _oracle(x, w, None, k, rows, cols)
    for o, what in ((lin, "split"), (unsplit, "unsplit")):
        assert_gemm_close(bf16_to_f64(o)[rows][:, cols], ref, f"mxfp4 linear {what}")


@pytest.mark.parametrize("m,k", [(1, 256), (7, 96), (16, 256), (16, 224)])
def test_mxfp4_fused_linear_equals_quantizer_then_gemm(m, k):
    """For m <= 16 the MXFP4 linear quantizes x inside the GEMM (its epilogue
    warps, one half of a 32-element block per lane).  With K of one stage the
    split-K plan has nothing to split, so the output must equal
    nvfp4_mxfp4_quant_act followed by nvfp4_mxfp4_gemm bit for bit, and the
    workspace's activation area stays untouched."""
    n = 1024
    x = syn.bf16_normal((m, k), 1.0, 6300 + m + k, device="cuda")
    w = syn.bf16_normal((n, k), 0.02, 6301, device="cuda")
    b = syn.bf16_normal((n,), 0.1, 6302, device="cuda")
    w_fp4, w_sf = _quant(w)
    ws = torch.full((nv.nvfp4_mxfp4_linear_workspace_bytes(m, k, n),), 0xA5, dtype=torch.uint8, device="cuda")
    lin = nv.mxfp4_linear(x, w_fp4, w_sf, k, n, bias=b, workspace=ws)
    a_fp4, a_sf = _quant(x)
    ref = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_mxfp4_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n, n, k, b, ref, n)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    assert torch.equal(lin.view(torch.int16), ref.view(torch.int16))
    assert bool((ws == 0xA5).all()), "the fused path writes no quantized activation to the workspace"
