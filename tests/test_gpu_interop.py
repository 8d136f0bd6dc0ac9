"""Independent pin of the operand layouts: the library's packed FP4 operands
and tiled block scales, handed unchanged to torch._scaled_mm (cuBLASLt's
block-scaled FP4 GEMM), must give the oracle's result.

Page "TorchNvFp4LinearKernel" (vLLM PR #53319), section 关键源码片段: the
weights' block scales go through swizzle_blockscale and the activation through
scaled_fp4_quant with swizzled scales, and both are consumed by
torch._scaled_mm(x_fp4, weight.t(), scale_a, scale_b), then * alpha, slice and
+ bias.  The tiled layout used here (512-byte tiles of 128 rows x 4 scale
columns) is this build's reading of that "swizzled" layout; a library whose
own layout is fixed by the hardware path it feeds, not by this build, reads
the bytes here.  A layout that was only self-consistent between the
quantizer, the GEMM and the oracle would fail: the activations below give
every row and every 16-element block of a row a different power-of-two
magnitude, so any misplaced scale byte changes the result grossly.

cuBLASLt accumulates in fp32 and its fp32 output is checked twice: at the
GEMM tolerance (max|err| <= 2e-2 rms, rel. Frobenius <= 5e-3) after x alpha
and + bias in float64, and at 1e-5 relative Frobenius error, far below any
layout error and far above fp32 accumulation noise at these K.  The
library's own bf16 output is checked element by element against the correctly
rounded result (half a bf16 step), since the outputs of these activations
span more binades than the rms-relative bound allows for bf16 rounding.
"""
import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_gemm_close, bf16_to_f64, dev_scalar, nv, require_library, syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not hasattr(torch, "float4_e2m1fn_x2"):
        pytest.fail("this torch has no float4_e2m1fn_x2: the cuBLASLt cross-check cannot run")
    return require_library()


def _block_scaled_activation(m: int, k: int, seed: int) -> torch.Tensor:
    """N(0,1) rows whose 16-element blocks are scaled by 2^e, e in [-6, 6]
    drawn per (row, block), so that block scales differ everywhere."""
    x = syn.bf16_normal((m, k), 1.0, seed).float()
    g = torch.Generator().manual_seed(seed + 1)
    nblk = (k + 15) // 16
    e = torch.randint(-6, 7, (m, nblk), generator=g).float()
    scale = torch.repeat_interleave(torch.exp2(e), 16, dim=1)[:, :k]
    return (x * scale).to(torch.bfloat16)


# (m, k, n_w, n_out, bias): the tiny config, ragged K with padding to 32
# (4104, 5128), an output slice, partial row bands and several column tiles
CASES = [
    (16, 256, 128, 128, False),
    (200, 4104, 384, 320, True),
    (300, 1024, 512, 512, False),
    (128, 5128, 256, 200, True),
    (257, 96, 640, 640, True),
]


@pytest.mark.parametrize("m,k,n_w,n_out,bias", CASES, ids=[f"m{c[0]}-k{c[1]}-n{c[2]}-o{c[3]}" for c in CASES])
def test_scaled_mm_consumes_the_library_layouts(m, k, n_w, n_out, bias):
    seed = 7000 + m + k
    x = _block_scaled_activation(m, k, seed)
    w = syn.bf16_normal((n_w, k), 0.02, seed + 2)
    b = syn.bf16_normal((n_out,), 0.1, seed + 3) if bias else None
    gs_x, gs_w = syn.global_scale(x), syn.global_scale(w)
    alpha = syn.alpha_of(gs_x, gs_w)

    a_fp4, a_sf = nv.quant_act(x.cuda(), dev_scalar(gs_x))
    w_fp4, w_sf = nv.prepare_weight(w.cuda(), dev_scalar(gs_w))
    c = torch._scaled_mm(a_fp4.view(torch.float4_e2m1fn_x2), w_fp4.view(torch.float4_e2m1fn_x2).t(),
                         a_sf.view(torch.float8_e4m3fn), w_sf.view(torch.float8_e4m3fn), out_dtype=torch.float32)
    ldo = (n_out + 7) // 8 * 8
    ours = torch.empty((m, ldo), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm(a_fp4, a_sf, m, w_fp4, w_sf, n_w, n_out, k, dev_scalar(alpha), b.cuda() if bias else None,
                  ours, ldo)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()

    # the oracle's own quantization of the same inputs (bit-identical to the
    # library's, which is checked here too) and its FP64 GEMM
    qa, sa = oracle.quantize(syn.bf16_bits(x), gs_x, k=k)
    qb, sb = oracle.quantize(syn.bf16_bits(w), gs_w, k=k)
    assert np.array_equal(a_fp4.cpu().numpy(), qa) and np.array_equal(a_sf.cpu().numpy(), oracle.swizzle(sa))
    assert np.array_equal(w_fp4.cpu().numpy(), qb) and np.array_equal(w_sf.cpu().numpy(), oracle.swizzle(sb))
    ref = oracle.gemm(qa, sa, qb[:n_out], sb[:n_out], alpha, syn.bf16_bits(b) if bias else None)

    lib = c[:, :n_out].double().cpu().numpy() * np.float64(np.float32(alpha))
    if bias:
        lib = lib + b.double().numpy()[None, :]
    assert_gemm_close(lib, ref, "torch._scaled_mm on the library's operands")
    frob = np.linalg.norm(lib - ref) / np.linalg.norm(ref)
    assert frob <= 1e-5, f"cuBLASLt result off the oracle by {frob:.3e} (relative Frobenius)"
    # and the library's own GEMM against the same oracle result: the outputs
    # span many binades here, so instead of the rms-relative bound each
    # element must be the correctly rounded bf16 of the exact result, up to
    # half a bf16 step (2^-8 relative) plus fp32 accumulation noise
    got = bf16_to_f64(ours[:, :n_out])
    rms = float(np.sqrt(np.mean(ref * ref)))
    bound = 2.0 ** -8 * np.abs(ref) + 1e-5 * rms
    assert (np.abs(got - ref) <= bound).all(), \
        f"nvfp4_gemm off by {float((np.abs(got - ref) / bound).max()):.2f} x (half a bf16 step + fp32 noise)"
    assert np.linalg.norm(got - ref) <= 5e-3 * np.linalg.norm(ref)
