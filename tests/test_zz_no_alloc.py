"""nvfp4_linear_noalloc: the linear layer for callers that cannot allocate
device memory (a plugin whose framework owns all device allocations, or code
that must never call cudaMalloc).  It uses the library's built-in scratch
array instead of a caller workspace.  This file is collected last on purpose:
if it fails, a run that stops at the first failure has already run the rest.

The test calls the new entry point through the C ABI twice in a row, with
different activations, and checks each output against nvfp4_linear's (same
tolerance as the other GEMM tests); it also checks that a problem too large
for the scratch is refused before anything runs."""
import pytest
import torch

from _helpers import assert_gemm_close, bf16_to_f64, dev_scalar, nv, require_library, syn

pytestmark = pytest.mark.gpu


def test_noalloc_matches_linear_on_two_calls_in_a_row():
    require_library()
    p = syn.Problem("noalloc", "t", 300, 4104, 1024, seed=901, bias=True, n_out=1000)
    L = syn.make_layer(p, device="cuda")
    w_fp4, w_sf = nv.prepare_weight(L.w, dev_scalar(L.gs_w))
    gs, alpha = dev_scalar(L.gs_x), dev_scalar(L.alpha)
    out = torch.empty((p.m, 1000), dtype=torch.bfloat16, device="cuda")
    ref = torch.empty_like(out)
    ws = torch.empty(nv.nvfp4_linear_workspace_bytes(p.m, p.k, p.n), dtype=torch.uint8, device="cuda")
    xs = [L.x, syn.bf16_normal((p.m, p.k), 1.0, seed=902, device="cuda")]
    for x in xs:
        out.fill_(0)
        nv.nvfp4_linear_noalloc(x, p.m, p.k, x.stride(0), gs, None, 0, w_fp4, w_sf, p.n, 1000, alpha, L.bias,
                                out, out.stride(0))
        nv.nvfp4_linear(x, p.m, p.k, x.stride(0), gs, None, 0, w_fp4, w_sf, p.n, 1000, alpha, L.bias,
                        ref, ref.stride(0), ws, ws.numel())
        torch.cuda.synchronize()
        nv.nvfp4_device_error()
        assert_gemm_close(bf16_to_f64(out), bf16_to_f64(ref), "noalloc vs linear")


def test_noalloc_rejects_problems_beyond_the_scratch():
    require_library()
    m, k, n = 16384, 4096, 128            # needs ~34 MB of scratch, more than the 16 MiB built in
    assert nv.nvfp4_linear_workspace_bytes(m, k, n) > 16 << 20
    x = torch.empty((m, k), dtype=torch.bfloat16, device="cuda")
    w_fp4 = torch.zeros((n, k // 2), dtype=torch.uint8, device="cuda")
    w_sf = torch.zeros(nv.nvfp4_scale_bytes(n, k), dtype=torch.uint8, device="cuda")
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_linear_noalloc(x, m, k, k, dev_scalar(1.0), None, 0, w_fp4, w_sf, n, n, dev_scalar(1.0), None,
                                out, n)
    assert e.value.status == 7 and "scratch" in str(e.value)
