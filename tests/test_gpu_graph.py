"""The linear inside a captured CUDA graph: replays are bit-identical to
eager calls, and weights reloaded in place (nvfp4_prepare_weight into the same
buffers) or new activations copied into the captured input buffer take effect
on the next replay -- the stable-address weight reload of the B12X backends
page (关键源码片段: in-place weight reload for captured graphs).  The last
replay is also checked against the oracle (transform, dynamic scale and all)."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_gemm_close, bf16_to_f64, dev_scalar, nv, require_library, syn

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return require_library()


def _weights(n, k, seed):
    w = syn.bf16_normal((n, k), 0.02, seed, device="cuda")
    return w, syn.global_scale(w)


@pytest.mark.parametrize("m,k,n,bs,dynamic", [
    (16, 1024, 768, 0, False),       # one-CTA GEMM with split-K in a cluster
    (256, 512, 512, 0, False),       # CTA-pair GEMM
    (256, 512, 512, 16, False),      # transform quantizer in the graph
    (64, 1024, 512, 0, True),        # dynamic global scale (memset + amax + finalize) in the graph
])
def test_linear_graph_replay_and_in_place_reload(m, k, n, bs, dynamic):
    x = syn.bf16_normal((m, k), 1.0, seed=600 + m, device="cuda")
    t = syn.random_hadamard_transform(bs, seed=bs).cuda() if bs else None
    w1, g1 = _weights(n, k, 601)
    w2, g2 = _weights(n, k, 602)
    w_gs = dev_scalar(g1)
    w_fp4 = torch.empty((n, nv.padded_k(k) // 2), dtype=torch.uint8, device="cuda")
    w_sf = torch.empty(nv.nvfp4_scale_bytes(n, k), dtype=torch.uint8, device="cuda")
    nv.nvfp4_prepare_weight(w1, n, k, k, w_gs, w_fp4, w_sf)
    gs = dev_scalar(syn.global_scale(x) if not bs else 30.0)
    alpha = torch.empty(1, dtype=torch.float32, device="cuda")
    alpha.fill_(syn.alpha_of(float(gs.item()), g1))
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(nv.nvfp4_linear_workspace_bytes(m, k, n), dtype=torch.uint8, device="cuda")

    def step():
        if dynamic:
            nv.nvfp4_act_global_scale(x, m, k, k, t, bs, w_gs, gs, alpha)
        nv.nvfp4_linear(x, m, k, k, gs, t, bs, w_fp4, w_sf, n, n, alpha, None, out, n, ws, ws.numel())

    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        step()                                      # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    eager1 = out.clone()

    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    assert torch.equal(out, eager1), "replay differs from the eager call"

    # reload the weight in place (same buffers, new global scale) and replay
    w_gs.fill_(g2)
    nv.nvfp4_prepare_weight(w2, n, k, k, w_gs, w_fp4, w_sf)
    if not dynamic:
        alpha.fill_(syn.alpha_of(float(gs.item()), g2))
    torch.cuda.synchronize()
    step()
    torch.cuda.synchronize()
    eager2 = out.clone()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, eager2), "replay after the in-place weight reload differs"
    assert not torch.equal(eager1, eager2)

    # new activations copied into the captured input buffer
    x.copy_(syn.bf16_normal((m, k), 1.0, seed=603, device="cuda"))
    if not dynamic and not bs:
        gs.fill_(syn.global_scale(x))
        alpha.fill_(syn.alpha_of(float(gs.item()), g2))
    torch.cuda.synchronize()
    step()
    torch.cuda.synchronize()
    eager3 = out.clone()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    assert torch.equal(out, eager3), "replay with new activations differs"

    # the replayed result against the oracle: reloaded weight w2, new activations
    xb = syn.bf16_bits(x)
    t_bits = syn.bf16_bits(t) if bs else None
    gs_ref = oracle.act_global_scale(xb, t_bits, bs, k) if dynamic else float(gs.item())
    if dynamic:
        assert np.float32(gs.item()) == np.float32(gs_ref), "replayed dynamic global scale differs from the oracle's"
        assert np.float32(alpha.item()) == np.float32(oracle.alpha(gs_ref, g2)), "replayed alpha differs"
    if bs:
        xb = oracle.transform(xb, t_bits, bs, k)
    a, sa = oracle.quantize(xb, gs_ref, k=k)
    b, sb = oracle.quantize(syn.bf16_bits(w2), g2, k=k)
    ref = oracle.gemm(a, sa, b, sb, float(alpha.item()))
    assert_gemm_close(bf16_to_f64(out), ref, f"graph replay m={m} bs={bs} dynamic={dynamic}")
