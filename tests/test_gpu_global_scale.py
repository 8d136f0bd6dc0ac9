"""GPU parity of the dynamic activation global scale (nvfp4_act_global_scale)
against the oracle: gs = fl32(448*6 / amax) over the tensor and alpha =
fl32(1 / (gs * gs_w)) bit for bit; with a transform, gs is the oracle's scale
of the y the kernel computes (exported by nvfp4_quant_act_export_y), and the
whole dynamic-scale linear matches the oracle within the GEMM tolerance."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import assert_gemm_close, dev_scalar, nv, require_library, sample_indices, syn

pytestmark = pytest.mark.gpu

FLT_MAX = float(np.finfo(np.float32).max)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return require_library()


def _gpu_scale(x: torch.Tensor, k: int, t=None, bs=0, w_gs=None):
    """x is a [m, ldx] CUDA tensor whose first k columns are the data."""
    m = x.shape[0]
    gs = torch.full((1,), -7.0, dtype=torch.float32, device="cuda")
    alpha = torch.full((1,), -7.0, dtype=torch.float32, device="cuda") if w_gs is not None else None
    wg = dev_scalar(w_gs) if w_gs is not None else None
    nv.nvfp4_act_global_scale(x, m, k, x.stride(0) if m else k, t, bs, wg, gs, alpha)
    torch.cuda.synchronize()
    return float(gs.item()), (float(alpha.item()) if alpha is not None else None)


@pytest.mark.parametrize("m,k,ldx,kind", [
    (1, 4096, 4096, "normal"),
    (97, 4104, 4112, "outlier"),          # padded-K width, strided rows
    (33, 250, 256, "student_t"),          # k % 16 != 0: scalar tail loads
    (4096, 4096, 4096, "student_t"),
    (8192, 14336, 14336, "normal"),
])
def test_global_scale_bit_exact(m, k, ldx, kind):
    seed = 5000 + m + k
    if kind == "normal":
        x = syn.bf16_normal((m, ldx), 1.0, seed)
    elif kind == "outlier":
        x = syn.bf16_outlier_channels(m, ldx, seed)
    else:
        x = syn.bf16_student_t(m, ldx, 3, seed)
    # the columns past k must not count: make them larger than anything inside
    x[:, k:] = 1e4
    gs, alpha = _gpu_scale(x.cuda(), k, w_gs=37.5)
    ref = oracle.act_global_scale(syn.bf16_bits(x)[:, :k])
    assert gs == ref, (gs, ref)
    assert alpha == oracle.alpha(ref, 37.5)
    assert ref == syn.global_scale(x[:, :k])          # the host calibration constant agrees


def test_global_scale_special_cases():
    z = torch.zeros((300, 512), dtype=torch.bfloat16, device="cuda")
    assert _gpu_scale(z, 512)[0] == 1.0                                  # amax 0
    e = torch.empty((0, 512), dtype=torch.bfloat16, device="cuda")
    assert _gpu_scale(e, 512)[0] == 1.0                                  # m = 0 still writes gs
    t = torch.zeros((16, 64), dtype=torch.int16, device="cuda")
    t[9, 33] = 1                                                         # one 2^-133, the rest +0
    assert _gpu_scale(t.view(torch.bfloat16), 64)[0] == FLT_MAX
    s = torch.zeros((8, 64), dtype=torch.bfloat16, device="cuda")
    s[3, 7] = -448.0                                                     # the sign does not matter
    s[5, 60] = 100.0
    gs, alpha = _gpu_scale(s, 64, w_gs=6.0)
    assert gs == 6.0 and alpha == float(np.float32(1) / np.float32(36.0))


@pytest.mark.parametrize("bs,m", [(16, 97), (128, 97), (64, 4096), (128, 4096)])
def test_global_scale_with_transform(bs, m):
    """gs is the oracle's scale of the kernel's own y (the amax pass and the
    quantizer run the same MMA pipeline), and that y's amax is the oracle's
    exactly rounded amax or one bf16 step from it."""
    p = syn.Problem("transform", f"bs{bs}", m, 4096, 4096, seed=5100 + bs + m, x_kind="student_t", bs=bs)
    x = syn.make_activation(p).cuda()
    t = syn.random_hadamard_transform(bs, seed=p.seed).cuda()
    gs, _ = _gpu_scale(x, 4096, t, bs)
    fp4 = torch.empty((m, 2048), dtype=torch.uint8, device="cuda")
    sf = torch.empty(nv.nvfp4_scale_bytes(m, 4096), dtype=torch.uint8, device="cuda")
    y = torch.empty((m, 4096), dtype=torch.int16, device="cuda")
    nv.nvfp4_quant_act_export_y(x, m, 4096, 4096, dev_scalar(gs), t, bs, fp4, sf, y)
    torch.cuda.synchronize()
    y_bits = y.cpu().numpy().view(np.uint16)
    assert gs == oracle.act_global_scale(y_bits)
    amax_gpu = int((y_bits & 0x7FFF).max())
    if m <= 128:
        amax_ref = int((oracle.transform(syn.bf16_bits(x.cpu()), syn.bf16_bits(t.cpu()), bs) & 0x7FFF).max())
    else:   # rounding is monotone: the largest rounded |y| is the rounding of the largest exact |y|
        exact = np.abs(x.cpu().double().numpy().reshape(-1, bs) @ t.cpu().double().numpy()).max()
        amax_ref = int(syn.bf16_bits(torch.tensor([exact], dtype=torch.float32).to(torch.bfloat16))[0])
    assert abs(amax_gpu - amax_ref) <= 1, (hex(amax_gpu), hex(amax_ref))


@pytest.mark.parametrize("name", ["qkv", "down"])
def test_dynamic_scale_linear(name):
    """The dynamic-scale linear: gs and alpha from nvfp4_act_global_scale feed
    nvfp4_linear on the same stream; the quantized activation is bit-exact and
    the output within the GEMM tolerance of the oracle using its own scale."""
    p = [q for q in syn.llama([128]) if q.name == name][0]
    L = syn.make_layer(p)
    x = L.x.cuda()
    w_gs = dev_scalar(L.gs_w)
    w_fp4, w_sf = nv.prepare_weight(L.w.cuda(), w_gs)
    gs, alpha = nv.act_global_scale(x, w_gs=w_gs)
    out = nv.linear(x, w_fp4, w_sf, p.k, p.n, gs, alpha)
    a_fp4, a_sf = nv.quant_act(x, gs)
    torch.cuda.synchronize()
    gs_ref = oracle.act_global_scale(syn.bf16_bits(L.x))
    assert float(gs.item()) == gs_ref and float(alpha.item()) == oracle.alpha(gs_ref, L.gs_w)
    a_ref, sa_ref = oracle.quantize(syn.bf16_bits(L.x), gs_ref)
    assert np.array_equal(a_fp4.cpu().numpy(), a_ref)
    assert np.array_equal(a_sf.cpu().numpy(), oracle.swizzle(sa_ref))
    cols = sample_indices(p.n, 256, seed=7, must=[255, 256])
    b_ref, sb_ref = oracle.quantize(syn.bf16_bits(L.w)[cols], L.gs_w)
    ref = oracle.gemm(a_ref, sa_ref, b_ref, sb_ref, oracle.alpha(gs_ref, L.gs_w))
    got = out.float().cpu().numpy()[:, cols]
    assert_gemm_close(got, ref, f"dynamic-scale linear {name}")


def test_global_scale_full_size():
    """65536 x 16384 (2 GiB of bf16), the largest sweep point, against the
    host calibration constant (a torch max over the same tensor)."""
    x = syn.bf16_normal((65536, 16384), 1.0, seed=5200, device="cuda")
    x[12345, 16383] = -17.5                                           # the last column of a row counts
    gs, _ = _gpu_scale(x, 16384)
    assert gs == syn.global_scale(x) == float(np.float32(2688.0) / np.float32(17.5))
