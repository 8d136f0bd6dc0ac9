"""End-to-end parity of nvfp4_linear (quantize + GEMM + epilogue) against the
oracle, on every layer workload at its full size and in the launch path the
benchmark uses.  The GPU computes whole outputs; the oracle recomputes sampled
rows x sampled columns (tile edges included) from the same bf16 inputs, since
rows of the activation and rows of the weight quantize independently."""
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


def run_and_check(p: syn.Problem, n_rows=48, n_cols=384):
    L = syn.make_layer(p, device="cuda")
    m, k, n_out = p.m, p.k, p.n_keep
    w_fp4, w_sf = nv.prepare_weight(L.w, dev_scalar(L.gs_w))
    t = L.t.cuda() if L.t is not None else None
    out = nv.linear(L.x, w_fp4, w_sf, k, n_out, dev_scalar(L.gs_x), dev_scalar(L.alpha), L.bias, t, p.bs)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    rows = np.arange(m) if m <= n_rows else sample_indices(m, n_rows, p.seed, must=tile_edges(m, 128))
    cols = np.arange(n_out) if n_out <= n_cols else sample_indices(n_out, n_cols, p.seed + 1,
                                                                   must=tile_edges(n_out, 128))
    ri = torch.from_numpy(rows).cuda()
    ci = torch.from_numpy(cols).cuda()
    xb = syn.bf16_bits(L.x[ri])
    if t is not None:
        xb = oracle.transform(xb, syn.bf16_bits(L.t), p.bs)
    a, sa = oracle.quantize(xb, L.gs_x, k=k)
    b, sb = oracle.quantize(syn.bf16_bits(L.w[ci]), L.gs_w, k=k)
    bias = syn.bf16_bits(L.bias[ci]) if L.bias is not None else None
    ref = oracle.gemm(a, sa, b, sb, L.alpha, bias)
    got = bf16_to_f64(out[ri][:, ci])
    return assert_gemm_close(got, ref, f"{p.workload}/{p.name} m={m}")


def _ids(ps):
    return [f"{p.workload}-{p.name}-m{p.m}" + (f"-n{p.n_out}" if p.n_out else "") for p in ps]


TINY = syn.tiny()
LLAMA = syn.llama()
QWEN = syn.qwen()
XFORM = syn.transform_fused()
PADDED = syn.padded() + [p for p in syn.padded(n_out=10944) if p.m in (1, 128, 1024)]


@pytest.mark.parametrize("p", TINY, ids=_ids(TINY))
def test_tiny(p):
    run_and_check(p)


@pytest.mark.parametrize("p", LLAMA, ids=_ids(LLAMA))
def test_llama_shapes(p):
    run_and_check(p)


@pytest.mark.parametrize("p", QWEN, ids=_ids(QWEN))
def test_qwen_shapes(p):
    run_and_check(p)


@pytest.mark.parametrize("p", XFORM, ids=_ids(XFORM))
def test_transform_shapes(p):
    run_and_check(p)


@pytest.mark.parametrize("p", PADDED, ids=_ids(PADDED))
def test_padded_shapes(p):
    run_and_check(p)


def test_linear_reuses_caller_buffers_across_calls():
    """Same output/workspace buffers, two different activations: the second
    call fully overwrites the first (no stale scratch state)."""
    p = syn.Problem("t", "reuse", 200, 1024, 512, seed=77)
    L = syn.make_layer(p, device="cuda")
    w_fp4, w_sf = nv.prepare_weight(L.w, dev_scalar(L.gs_w))
    out = torch.empty((200, 512), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(nv.nvfp4_linear_workspace_bytes(200, 1024, 512), dtype=torch.uint8, device="cuda")
    x2 = syn.bf16_normal((200, 1024), 1.0, seed=78, device="cuda")
    for x in (L.x, x2):
        nv.linear(x, w_fp4, w_sf, 1024, 512, dev_scalar(L.gs_x), dev_scalar(L.alpha), out=out, workspace=ws)
        torch.cuda.synchronize()
        a, sa = oracle.quantize(syn.bf16_bits(x), L.gs_x)
        b, sb = oracle.quantize(syn.bf16_bits(L.w), L.gs_w)
        assert_gemm_close(bf16_to_f64(out), oracle.gemm(a, sa, b, sb, L.alpha), "reuse")


def test_linear_rejects_small_workspace():
    x = torch.zeros((4, 64), dtype=torch.bfloat16, device="cuda")
    w_fp4 = torch.zeros((128, 32), dtype=torch.uint8, device="cuda")
    w_sf = torch.zeros(nv.nvfp4_scale_bytes(128, 64), dtype=torch.uint8, device="cuda")
    out = torch.empty((4, 128), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(16, dtype=torch.uint8, device="cuda")
    with pytest.raises(nv.Nvfp4Error) as e:
        nv.nvfp4_linear(x, 4, 64, 64, dev_scalar(1.0), None, 0, w_fp4, w_sf, 128, 128, dev_scalar(1.0), None,
                        out, 128, ws, 16)
    assert e.value.status == 7


SPLIT_K = [syn.Problem("splitk", f"m{m}-n{n}-k{k}", m, k, n, seed=1300 + i, bias=bias, n_out=n_out)
           for i, (m, k, n, n_out, bias) in enumerate([
               (1, 4096, 256, None, False),      # one output tile: a cluster of 8 ranges of 2 stages
               (5, 4104, 1024, 1000, True),      # ragged K (65 k-steps), sliced output, bias
               (64, 14336, 4096, None, True),    # Llama down_proj width at decode size
               (128, 14336, 512, 500, False),    # full band, 2 tiles, long K: 7 stages per range
               (33, 64, 256, None, True),        # a single K stage: no split
           ])]


@pytest.mark.parametrize("p", SPLIT_K, ids=_ids(SPLIT_K))
def test_split_k_matches_oracle_and_unsplit(p):
    """Small m: nvfp4_linear splits K across the CTAs of a cluster (fp32
    partials summed in shared memory, rank order).  It must match the oracle on
    every element, agree with the unsplit one-CTA GEMM on the same quantized
    operands to fp32-summation-order accuracy, equal the split GEMM test hook
    (nvfp4_gemm_ex kernel 3) bit for bit, and be bit-identical across calls."""
    L = syn.make_layer(p, device="cuda")
    m, k, n_out = p.m, p.k, p.n_keep
    w_fp4, w_sf = nv.prepare_weight(L.w, dev_scalar(L.gs_w))
    gs, alpha = dev_scalar(L.gs_x), dev_scalar(L.alpha)
    ws_bytes = nv.nvfp4_linear_workspace_bytes(m, k, p.n)
    ldo = (n_out + 7) // 8 * 8                           # output rows 16-byte aligned

    def fresh():
        return torch.full((m, ldo), float("nan"), dtype=torch.bfloat16, device="cuda")[:, :n_out]

    outs = []
    for _ in range(2):
        ws = torch.full((ws_bytes,), 0xA5, dtype=torch.uint8, device="cuda")
        out = fresh()
        nv.nvfp4_linear(L.x, m, k, L.x.stride(0), gs, None, 0, w_fp4, w_sf, p.n, n_out, alpha, L.bias,
                        out, out.stride(0), ws, ws_bytes)
        outs.append(out)
    a_fp4, a_sf = nv.quant_act(L.x, gs)
    for kernel in (1, 3):                                # unsplit, split with the linear's plan
        out = fresh()
        nv.nvfp4_gemm_ex(a_fp4, a_sf, m, w_fp4, w_sf, p.n, n_out, k, alpha, L.bias, out, out.stride(0),
                         kernel=kernel)
        outs.append(out)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    assert torch.equal(outs[0].view(torch.int16), outs[1].view(torch.int16)), "split-K not deterministic"
    assert torch.equal(outs[0].view(torch.int16), outs[3].view(torch.int16)), "linear differs from the split GEMM"
    a, sa = oracle.quantize(syn.bf16_bits(L.x), L.gs_x, k=k)
    b, sb = oracle.quantize(syn.bf16_bits(L.w[:n_out]), L.gs_w, k=k)
    bias = syn.bf16_bits(L.bias[:n_out]) if L.bias is not None else None
    ref = oracle.gemm(a, sa, b, sb, L.alpha, bias)
    assert_gemm_close(bf16_to_f64(outs[0]), ref, f"split-K {p.name}")
    assert_gemm_close(bf16_to_f64(outs[2]), ref, f"unsplit {p.name}")
    split, unsplit = bf16_to_f64(outs[0]), bf16_to_f64(outs[2])
    # The fp32 sums differ only in order (a few fp32 ulp of the summed terms),
    # so after the bf16 rounding the two differ by at most one bf16 ulp
    # (2^-7 relative) plus that fp32 noise.
    rms = np.sqrt(np.mean(ref ** 2))
    bound = 2.0 ** -7 * np.maximum(np.abs(split), np.abs(unsplit)) + 1e-5 * rms
    assert np.all(np.abs(split - unsplit) <= bound), "split-K and unsplit GEMM differ beyond rounding"


@pytest.mark.parametrize("m", [1, 2, 3, 4, 5, 8, 9, 13, 16, 17, 77, 128])
def test_small_m_linear_equals_quantizer_then_gemm(m):
    """For m <= 16 nvfp4_linear runs the fused linear: the GEMM's epilogue
    warps quantize each stage of x into shared memory themselves (no quantizer
    launch); above that, the quantizer writes the workspace and the GEMM reads
    it.  The output must equal nvfp4_quant_act followed by nvfp4_gemm_ex with
    the same split-K plan (kernel 3) bit for bit either way (and for m > 16 so
    must the workspace's quantized activation)."""
    k, n = 4104, 768
    x = syn.bf16_normal((m, k), 1.0, 1400 + m, device="cuda")
    w = syn.bf16_normal((n, k), 0.02, 1401, device="cuda")
    b = syn.bf16_normal((n,), 0.1, 1402, device="cuda")
    gs_x, gs_w = syn.global_scale(x), syn.global_scale(w)
    gs, alpha = dev_scalar(gs_x), dev_scalar(syn.alpha_of(gs_x, gs_w))
    w_fp4, w_sf = nv.prepare_weight(w, dev_scalar(gs_w))
    a_fp4, a_sf = nv.quant_act(x, gs)
    ref = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_gemm_ex(a_fp4, a_sf, m, w_fp4, w_sf, n, n, k, alpha, b, ref, n, kernel=3)
    pk = nv.nvfp4_packed_bytes(m, k)
    small = (pk + 255) // 256 * 256 + (nv.nvfp4_scale_bytes(m, k) + 255) // 256 * 256
    ws = torch.full((small,), 0x5A, dtype=torch.uint8, device="cuda")
    out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_linear(x, m, k, k, gs, None, 0, w_fp4, w_sf, n, n, alpha, b, out, n, ws, small)
    torch.cuda.synchronize()
    nv.nvfp4_device_error()
    assert torch.equal(out.view(torch.int16), ref.view(torch.int16))
    if m > 16:
        assert torch.equal(ws[:pk], a_fp4.view(-1))
        sf0 = (pk + 255) // 256 * 256
        assert torch.equal(ws[sf0:sf0 + a_sf.numel()], a_sf)
