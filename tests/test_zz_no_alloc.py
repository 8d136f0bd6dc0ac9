"""nvfp4_linear_noalloc: the linear layer for callers that cannot allocate
device memory (a plugin whose framework owns all device allocations, or code
that must never call cudaMalloc).  It uses the library's built-in 16 MiB
scratch array instead of a caller workspace.  This file is collected last on
purpose: if it fails, a run that stops at the first failure has already run
the rest.

Every check calls the entry point through the C ABI, at least twice in a row
with different activations (the scratch keeps the previous call's bytes), and
compares each output with nvfp4_linear's:
  - bit for bit against nvfp4_linear given a 16 MiB workspace of its own,
    since both then run the same kernels with the same split plan;
  - against the oracle's FP64 result at the GEMM tolerance;
  - for small m (split-K), bit for bit against nvfp4_linear given exactly
    nvfp4_linear_workspace_bytes.
A problem whose minimum workspace is exactly the scratch size runs; one more
row is refused before anything runs."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import (assert_gemm_close, bf16_to_f64, dev_scalar, nv, require_library, sample_indices, syn,
                      tile_edges)

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 16 << 20


def _min_workspace(m: int, k: int) -> int:
    a = nv.nvfp4_packed_bytes(m, k)
    s = nv.nvfp4_scale_bytes(m, k)
    return (a + 255) // 256 * 256 + (s + 255) // 256 * 256


def _oracle_rows_cols(x, w, bias, k, gs_x, gs_w, alpha, rows, cols):
    a, sa = oracle.quantize(syn.bf16_bits(x[torch.from_numpy(rows)].cpu()), gs_x, k=k)
    b, sb = oracle.quantize(syn.bf16_bits(w[torch.from_numpy(cols)].cpu()), gs_w, k=k)
    bb = syn.bf16_bits(bias[torch.from_numpy(cols)].cpu()) if bias is not None else None
    return oracle.gemm(a, sa, b, sb, alpha, bb)


def _run_pair_of_calls(m, k, n_w, n_out, bias, seed, full_workspace_check):
    require_library()
    x0 = syn.bf16_normal((m, k), 1.0, seed, device="cuda")
    x1 = syn.bf16_normal((m, k), 1.0, seed + 1, device="cuda")
    w = syn.bf16_normal((n_w, k), 0.02, seed + 2, device="cuda")
    b = syn.bf16_normal((n_out,), 0.1, seed + 3, device="cuda") if bias else None
    gs_w = syn.global_scale(w)
    w_fp4, w_sf = nv.prepare_weight(w, dev_scalar(gs_w))
    ldo = (n_out + 7) // 8 * 8
    same = torch.empty(SCRATCH_BYTES, dtype=torch.uint8, device="cuda")
    full = torch.empty(max(nv.nvfp4_linear_workspace_bytes(m, k, n_w), 1), dtype=torch.uint8, device="cuda")
    rows = np.arange(m) if m <= 64 else sample_indices(m, 48, seed, must=tile_edges(m, 128))
    cols = np.arange(n_out) if n_out <= 256 else sample_indices(n_out, 256, seed + 1, must=tile_edges(n_out, 128))
    for x in (x0, x1):
        gs_x = syn.global_scale(x)
        alpha = syn.alpha_of(gs_x, gs_w)
        gs, al = dev_scalar(gs_x), dev_scalar(alpha)
        out = torch.full((m, ldo), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :n_out]
        ref16 = torch.full_like(out, float("nan"))
        nv.nvfp4_linear_noalloc(x, m, k, k, gs, None, 0, w_fp4, w_sf, n_w, n_out, al, b, out, ldo)
        nv.nvfp4_linear(x, m, k, k, gs, None, 0, w_fp4, w_sf, n_w, n_out, al, b, ref16, ldo, same, same.numel())
        torch.cuda.synchronize()
        nv.nvfp4_device_error()
        assert torch.equal(out.view(torch.int16), ref16.view(torch.int16)), "noalloc differs from nvfp4_linear"
        ref = _oracle_rows_cols(x, w, b, k, gs_x, gs_w, alpha, rows, cols)
        assert_gemm_close(bf16_to_f64(out)[rows][:, cols], ref, f"noalloc m={m} vs oracle")
        if full_workspace_check:
            ref_full = torch.empty_like(out)
            nv.nvfp4_linear(x, m, k, k, gs, None, 0, w_fp4, w_sf, n_w, n_out, al, b, ref_full, ldo, full,
                            full.numel())
            torch.cuda.synchronize()
            assert torch.equal(out.view(torch.int16), ref_full.view(torch.int16)), \
                f"noalloc m={m} differs from nvfp4_linear with its own workspace"


def test_noalloc_matches_linear_on_two_calls_in_a_row():
    _run_pair_of_calls(300, 4104, 1024, 1000, True, seed=901, full_workspace_check=False)


@pytest.mark.parametrize("m,n", [(1, 4096), (128, 2048)])
def test_noalloc_small_m_split_k_through_the_scratch(m, n):
    """m <= 128 at k = 14336 (a long K, which the split-K plan cuts into
    ranges): the same kernels and plan as nvfp4_linear with its own workspace,
    so the two outputs are equal bit for bit, over the stale bytes of the
    previous call in the scratch."""
    _run_pair_of_calls(m, 14336, n, n, m == 1, seed=910 + m, full_workspace_check=True)


def test_noalloc_at_the_scratch_limit():
    """m = 7280, k = 4096: the quantized activation and scales take exactly
    16 MiB; m = 7281 needs more and is refused."""
    assert _min_workspace(7280, 4096) == SCRATCH_BYTES
    assert _min_workspace(7281, 4096) > SCRATCH_BYTES
    _run_pair_of_calls(7280, 4096, 384, 384, False, seed=930, full_workspace_check=False)
    x = torch.empty((7281, 4096), dtype=torch.bfloat16, device="cuda")
    w_fp4 = torch.zeros((128, 2048), dtype=torch.uint8, device="cuda")
    w_sf = torch.zeros(nv.nvfp4_scale_bytes(128, 4096), dtype=torch.uint8, device="cuda")
    out = torch.empty((7281, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_linear_noalloc(x, 7281, 4096, 4096, dev_scalar(1.0), None, 0, w_fp4, w_sf, 128, 128,
                                dev_scalar(1.0), None, out, 128)
    assert e.value.status == 7 and "scratch" in str(e.value)


def test_noalloc_rejects_problems_beyond_the_scratch():
    require_library()
    m, k, n = 16384, 4096, 128            # needs ~34 MB of scratch, more than the 16 MiB built in
    assert nv.nvfp4_linear_workspace_bytes(m, k, n) > SCRATCH_BYTES
    x = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    w_fp4 = torch.zeros((n, k // 2), dtype=torch.uint8, device="cuda")
    w_sf = torch.zeros(nv.nvfp4_scale_bytes(n, k), dtype=torch.uint8, device="cuda")
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_linear_noalloc(x, m, k, k, dev_scalar(1.0), None, 0, w_fp4, w_sf, n, n, dev_scalar(1.0), None,
                                out, n)
    assert e.value.status == 7 and "scratch" in str(e.value)
