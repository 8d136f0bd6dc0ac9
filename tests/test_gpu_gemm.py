"""GPU parity of the block-scaled FP4 GEMM (nvfp4_gemm) against the oracle's
FP64 dequantize-then-matmul on identical quantized operands.

The GPU operands come from the CUDA quantizers, the oracle's from the oracle's
own quantizer (the quantizer tests show the bytes are identical); outputs must
satisfy max|err| <= 2e-2 * rms(ref) and ||err||_F/||ref||_F <= 5e-3.
"""
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


def _gpu_gemm(x, w, k, gs_x, gs_w, alpha, n_out=None, bias=None, ldo=None, fill=None):
    m, n_w = x.shape[0], w.shape[0]
    n_out = n_w if n_out is None else n_out
    a_fp4, a_sf = nv.quant_act(x.cuda(), dev_scalar(gs_x))
    w_fp4, w_sf = nv.prepare_weight(w.cuda(), dev_scalar(gs_w))
    ldo = (n_out + 7) // 8 * 8 if ldo is None else ldo       # 16-byte aligned output rows
    out = torch.empty((m, ldo), dtype=torch.bfloat16, device="cuda")
    if fill is not None:
        out.fill_(fill)
    nv.nvfp4_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, dev_scalar(alpha),
                  bias.cuda() if bias is not None else None, out, ldo)
    torch.cuda.synchronize()
    return out[:, :n_out]


def _oracle_gemm(x, w, k, gs_x, gs_w, alpha, bias=None, rows=None, cols=None):
    xb = syn.bf16_bits(x if rows is None else x[torch.as_tensor(rows)])
    wb = syn.bf16_bits(w if cols is None else w[torch.as_tensor(cols)])
    a, sa = oracle.quantize(xb[:, :k], gs_x, k=k)
    b, sb = oracle.quantize(wb[:, :k], gs_w, k=k)
    bb = None
    if bias is not None:
        bb = syn.bf16_bits(bias if cols is None else bias[torch.as_tensor(cols)])
    return oracle.gemm(a, sa, b, sb, alpha, bb)


def test_gemm_tiny_config_all_outputs():
    p = syn.tiny()[0]
    L = syn.make_layer(p)
    got = _gpu_gemm(L.x, L.w, p.k, L.gs_x, L.gs_w, L.alpha)
    ref = _oracle_gemm(L.x, L.w, p.k, L.gs_x, L.gs_w, L.alpha)
    assert_gemm_close(bf16_to_f64(got), ref, "tiny")


def test_gemm_exact_integer_case_is_bit_exact():
    """Unit block scales, gs = alpha = 1, small-integer products: every partial
    sum is exact in fp32, so the bf16 output must equal the correctly rounded
    exact result bit for bit (covers all 256 columns of a tile and a ragged K)."""
    rng = np.random.default_rng(30)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    k = 320
    xa = rng.choice(grid, (200, k)) * rng.choice([-1, 1], (200, k))
    xw = rng.choice(grid, (384, k)) * rng.choice([-1, 1], (384, k))
    xa[:, ::16] = 6
    xw[:, ::16] = 6
    x = torch.tensor(xa, dtype=torch.float32).to(torch.bfloat16)
    w = torch.tensor(xw, dtype=torch.float32).to(torch.bfloat16)
    got = _gpu_gemm(x, w, k, 1.0, 1.0, 1.0)
    exact = torch.from_numpy(xa @ xw.T)
    assert (exact.abs() < 2 ** 22).all()
    ref = exact.float().to(torch.bfloat16)
    assert torch.equal(got.cpu().view(torch.int16), ref.view(torch.int16))


@pytest.mark.parametrize("m,n_w,n_out,k,bias", [
    (1, 128, 128, 64, False), (16, 256, 256, 256, True), (130, 384, 300, 4104, True),
    (257, 640, 640, 96, False), (100, 512, 200, 1000, True), (129, 1000, 1000, 5128, True),
    (300, 256, 1, 128, True), (17, 11008, 10944, 4104, True), (64, 128, 100, 32, False),
])
def test_gemm_ragged_shapes(m, n_w, n_out, k, bias):
    seed = m * 7 + n_w * 3 + k
    x = syn.bf16_normal((m, k), 1.0, seed)
    w = syn.bf16_normal((n_w, k), 0.02, seed + 1)
    b = syn.bf16_normal((n_out,), 0.1, seed + 2) if bias else None
    gs_x, gs_w = syn.global_scale(x), syn.global_scale(w)
    alpha = syn.alpha_of(gs_x, gs_w)
    got = _gpu_gemm(x, w, k, gs_x, gs_w, alpha, n_out=n_out, bias=b)
    cols = None if n_out * m <= 300 * 1000 else sample_indices(n_out, 300, seed, must=tile_edges(n_out, 128))
    ref = _oracle_gemm(x, w[:n_out], k, gs_x, gs_w, alpha, bias=b, cols=cols)
    g = bf16_to_f64(got)
    assert_gemm_close(g if cols is None else g[:, cols], ref, f"{m}x{n_w}->{n_out}x{k}")


def test_gemm_slice_leaves_padded_columns_untouched():
    m, n_w, n_out, k = 70, 512, 448, 256
    x = syn.bf16_normal((m, k), 1.0, 31)
    w = syn.bf16_normal((n_w, k), 0.02, 32)
    gs_x, gs_w = syn.global_scale(x), syn.global_scale(w)
    alpha = syn.alpha_of(gs_x, gs_w)
    got = _gpu_gemm(x, w, k, gs_x, gs_w, alpha, n_out=n_out, ldo=n_w, fill=-7.0)
    full = got.as_strided((m, n_w), (n_w, 1))
    tail = full[:, n_out:].float().cpu()
    assert (tail == -7.0).all()
    ref = _oracle_gemm(x, w[:n_out], k, gs_x, gs_w, alpha)
    assert_gemm_close(bf16_to_f64(got[:, :n_out]), ref, "slice")


def test_gemm_zero_rows_is_a_noop():
    nv.nvfp4_gemm(None, None, 0, None, None, 128, 128, 64, None, None, None, 128)
