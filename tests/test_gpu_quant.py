"""GPU parity of the quantizers (nvfp4_quant_act, nvfp4_prepare_weight) against
the CPU oracle: packed FP4 bytes and tiled scale bytes, padding included, must
match bit for bit.  With the block-diagonal transform, the codes must match the
oracle's quantization of the kernel's own bf16 y bit for bit, and y must match
the exact x * blockdiag(T) within the fp32 accumulation bound."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import dev_scalar, gather_scales, nv, require_library, sample_indices, syn, tile_edges

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return require_library()


def _gpu_quant(x: torch.Tensor, k: int, gs: float, t=None, bs=0, weight=False):
    m = x.shape[0]
    xd = x.cuda()
    if xd.stride(0) % 8:                      # rows must start on 16-byte boundaries
        buf = torch.zeros((m, (xd.shape[1] + 7) // 8 * 8), dtype=xd.dtype, device="cuda")
        buf[:, :xd.shape[1]] = xd
        xd = buf[:, :xd.shape[1]]
    fp4 = torch.full((m, nv.padded_k(k) // 2), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full((nv.nvfp4_scale_bytes(m, k),), 0xCD, dtype=torch.uint8, device="cuda")
    g = dev_scalar(gs)
    if weight:
        nv.nvfp4_prepare_weight(xd, m, k, xd.stride(0), g, fp4, sf)
    else:
        td = t.cuda() if t is not None else None
        nv.nvfp4_quant_act(xd, m, k, xd.stride(0), g, td, bs, fp4, sf)
    torch.cuda.synchronize()
    return fp4.cpu().numpy(), sf.cpu().numpy()


def _oracle_quant(x: torch.Tensor, k: int, gs: float, t=None, bs=0):
    xb = syn.bf16_bits(x)[:, :k]
    if t is not None:
        xb = oracle.transform(xb, syn.bf16_bits(t), bs)
    packed, sf_lin = oracle.quantize(xb, gs, k=k)
    return packed, oracle.swizzle(sf_lin)


def _assert_bytes_equal(got, ref, what):
    bad = np.flatnonzero(got.ravel() != ref.ravel())
    assert bad.size == 0, f"{what}: {bad.size} bytes differ, first at {bad[:8]} got {got.ravel()[bad[:8]]} ref {ref.ravel()[bad[:8]]}"


def test_tiny_config_bit_exact():
    p = syn.tiny()[0]
    L = syn.make_layer(p)
    got = _gpu_quant(L.x, p.k, L.gs_x)
    ref = _oracle_quant(L.x, p.k, L.gs_x)
    _assert_bytes_equal(got[0], ref[0], "packed")
    _assert_bytes_equal(got[1], ref[1], "scales")


@pytest.mark.parametrize("m,k,kind", [
    (1, 4096, "normal"), (16, 256, "normal"), (130, 4104, "normal"), (300, 5128, "outlier"),
    (257, 40, "student_t"), (33, 16, "normal"), (128, 8, "normal"), (5, 33, "student_t"),
    (200, 14336, "outlier"), (64, 25600, "outlier"), (3, 1000, "student_t"),
])
def test_quant_shapes_bit_exact(m, k, kind):
    p = syn.Problem("t", "t", m, k, 1, seed=7000 + m + k, x_kind=kind)
    x = syn.make_activation(p)
    gs = syn.global_scale(x)
    got = _gpu_quant(x, k, gs)
    ref = _oracle_quant(x, k, gs)
    _assert_bytes_equal(got[0], ref[0], f"packed {m}x{k}")
    _assert_bytes_equal(got[1], ref[1], f"scales {m}x{k}")


@pytest.mark.parametrize("gs_mult", [1e-3, 0.37, 1.0, 25.0, 1e4])
def test_quant_global_scale_range(gs_mult):
    """Global scales far from the calibrated one push block scales into the E4M3
    subnormals (and zero) or into saturation at 448."""
    x = syn.bf16_student_t(64, 512, 3, seed=71)
    gs = float(np.float32(syn.global_scale(x) * gs_mult))
    got = _gpu_quant(x, 512, gs)
    ref = _oracle_quant(x, 512, gs)
    _assert_bytes_equal(got[0], ref[0], "packed")
    _assert_bytes_equal(got[1], ref[1], "scales")


def test_quant_special_values():
    """Zero blocks, negative zeros, tiny (subnormal) inputs, exact grid values,
    E2M1 rounding ties and values that saturate."""
    rng = np.random.default_rng(72)
    rows = []
    rows.append(np.zeros(256))
    rows.append(-np.zeros(256))
    rows.append(rng.normal(size=256) * 1e-38)
    grid = np.array([0, 0.5, 1, 1.5, 2, 3, 4, 6])
    r = rng.choice(grid, 256) * rng.choice([-1, 1], 256)
    r[::16] = 6
    rows.append(r)
    ties = np.tile(np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 6.0, 0.1, -0.1, 3.0, 2.0, 1.0, 0.5]), 16)
    rows.append(ties)
    rows.append(rng.normal(size=256) * 1e30)
    x = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.bfloat16)
    for gs in [1.0, 448.0 * 6 / 6.0, 0.5, 1e-30]:
        got = _gpu_quant(x, 256, gs)
        ref = _oracle_quant(x, 256, gs)
        _assert_bytes_equal(got[0], ref[0], f"packed gs={gs}")
        _assert_bytes_equal(got[1], ref[1], f"scales gs={gs}")


def test_quant_strided_input():
    """A non-contiguous row view (row stride > k) is read in place."""
    wide = syn.bf16_normal((70, 4096 + 64), 1.0, seed=73)
    view = wide[:, 32:32 + 4096]
    assert not view.is_contiguous()
    gs = syn.global_scale(view)
    got = _gpu_quant(view, 4096, gs)
    ref = _oracle_quant(view.contiguous(), 4096, gs)
    _assert_bytes_equal(got[0], ref[0], "packed")
    _assert_bytes_equal(got[1], ref[1], "scales")


def test_prepare_weight_bit_exact():
    p = syn.tiny()[0]
    L = syn.make_layer(p)
    got = _gpu_quant(L.w, p.k, L.gs_w, weight=True)
    ref = _oracle_quant(L.w, p.k, L.gs_w)
    _assert_bytes_equal(got[0], ref[0], "packed weight")
    _assert_bytes_equal(got[1], ref[1], "weight scales")
    w = syn.bf16_normal((11008, 4104), 0.02, seed=74)
    gs = syn.global_scale(w)
    got = _gpu_quant(w, 4104, gs, weight=True)
    rows = sample_indices(11008, 40, seed=74, must=[127, 128, 10943, 10944])
    packed, sf_lin = oracle.quantize(syn.bf16_bits(w)[rows], gs, k=4104)
    _assert_bytes_equal(got[0][rows], packed, "packed weight rows")
    _assert_bytes_equal(gather_scales(got[1], rows, sf_lin.shape[1], 4104), sf_lin, "weight scale rows")


def _gpu_quant_export(x: torch.Tensor, k: int, gs: float, t: torch.Tensor, bs: int):
    """The transform quantizer through nvfp4_quant_act_export_y: (packed, tiled
    scales, y bits); also checks that nvfp4_quant_act writes the same bytes."""
    m = x.shape[0]
    xd = x.cuda()
    fp4 = torch.full((m, nv.padded_k(k) // 2), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full((nv.nvfp4_scale_bytes(m, k),), 0xCD, dtype=torch.uint8, device="cuda")
    y = torch.full((m, k), -1, dtype=torch.int16, device="cuda")          # 0xFFFF: a NaN pattern
    g, td = dev_scalar(gs), t.cuda()
    nv.nvfp4_quant_act_export_y(xd, m, k, xd.stride(0), g, td, bs, fp4, sf, y)
    plain = _gpu_quant(x, k, gs, t=t, bs=bs)
    torch.cuda.synchronize()
    got = fp4.cpu().numpy(), sf.cpu().numpy(), y.cpu().numpy().view(np.uint16)
    _assert_bytes_equal(plain[0], got[0], "packed (plain vs export entry point)")
    _assert_bytes_equal(plain[1], got[1], "scales (plain vs export entry point)")
    return got


def _check_transform_y(y_bits, x: torch.Tensor, t: torch.Tensor, bs: int, rows=None):
    """The kernel's y against x * blockdiag(T): within half a bf16 step plus the
    fp32 accumulation bound bs * 2^-23 * sum|x_i T_ij| of the exact sum
    (float64 matmul of the bf16 values), and equal to the oracle's exactly
    rounded sum except at a small fraction of near ties.  Returns the number
    of elements that differ from the oracle's y."""
    xs = x if rows is None else x[rows]
    ref = oracle.transform(syn.bf16_bits(xs), syn.bf16_bits(t), bs)
    xd = xs.double().numpy().reshape(-1, bs)
    td = t.double().numpy()
    exact = (xd @ td).reshape(ref.shape)
    mag = (np.abs(xd) @ np.abs(td)).reshape(ref.shape)
    yg = (y_bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    assert np.isfinite(yg).all(), "y has unwritten elements"
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact), 2.0 ** -126))) - 8)
    err = np.abs(yg - exact)
    tol = half_ulp * 1.0001 + bs * 2.0 ** -23 * mag
    assert (err <= tol).all(), f"y off by {float((err / tol).max()):.2f} x tolerance"
    n_diff = int((y_bits != ref).sum())
    assert n_diff <= max(2, 1e-3 * ref.size), f"{n_diff} of {ref.size} y values differ from the exact rounding"
    return n_diff


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
@pytest.mark.parametrize("m", [16, 97])
def test_transform_quant_parity(bs, m):
    """Transform + quantizer (reading A12, tiered): y within the fp32
    accumulation bound of the exact x * blockdiag(T); codes and scales are the
    oracle's quantization of that y, bit for bit; end to end, against the
    oracle's exactly rounded y, at most a 1e-4 fraction of bytes differ."""
    p = syn.Problem("transform", f"bs{bs}", m, 4096, 4096, seed=3100 + bs + m, x_kind="student_t", bs=bs)
    x = syn.make_activation(p)
    t = syn.random_hadamard_transform(bs, seed=p.seed)
    gs = float(np.float32(syn.E4M3_MAX * syn.FP4_MAX) / np.float32(syn.transformed_amax(x, t)))
    got_pk, got_sf, y = _gpu_quant_export(x, 4096, gs, t, bs)
    packed, sf_lin = oracle.quantize(y, gs, k=4096)
    _assert_bytes_equal(got_pk, packed, f"packed vs oracle(y) bs={bs}")
    _assert_bytes_equal(got_sf, oracle.swizzle(sf_lin), f"scales vs oracle(y) bs={bs}")
    _check_transform_y(y, x, t, bs)
    ref = _oracle_quant(x, 4096, gs, t=t, bs=bs)
    n_bad = int((got_pk != ref[0]).sum() + (got_sf != ref[1]).sum())
    assert n_bad <= max(2, 1e-4 * (got_pk.size + got_sf.size)), f"{n_bad} bytes differ end to end"


def _exact_sum_activation(m: int, k: int, bs: int, seed: int) -> torch.Tensor:
    """Small integers times a per-row power of two: in every bs-block the first
    element is odd and the others even, so each y = t * (sum of +-x_i) is an
    odd multiple of t (never zero, so no sign-of-zero choice arises), and every
    partial sum of the exact bf16 x bf16 products is exact in fp32 (T's
    entries all have the magnitude t, and |sum| <= 7 * bs)."""
    g = torch.Generator().manual_seed(seed)
    v = torch.randint(-3, 4, (m, k), generator=g) * 2                      # even in [-6, 6]
    odd = torch.randint(0, 4, (m, k // bs), generator=g) * 2 + 1            # 1, 3, 5, 7
    sign = torch.randint(0, 2, (m, k // bs), generator=g) * 2 - 1
    v[:, ::bs] = odd * sign
    e = torch.randint(-3, 4, (m, 1), generator=g).float()
    return (v.float() * torch.exp2(e)).to(torch.bfloat16)


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
@pytest.mark.parametrize("m", [300, 4096])
def test_transform_quant_exact_sums_zero_mismatch(bs, m):
    """Transform inputs whose sums are exact in fp32 (reading A12: the exact
    case of the tiered parity): whatever order the tensor core sums in, y is
    the exact sum rounded once, so y, the packed codes and the scales must
    equal the oracle's end to end with no byte different."""
    k = 1024
    x = _exact_sum_activation(m, k, bs, seed=8100 + bs + m)
    t = syn.random_hadamard_transform(bs, seed=8200 + bs)
    gs = float(np.float32(syn.E4M3_MAX * syn.FP4_MAX) / np.float32(syn.transformed_amax(x, t)))
    got_pk, got_sf, y = _gpu_quant_export(x, k, gs, t, bs)
    rows = np.arange(m) if m <= 300 else sample_indices(m, 64, seed=bs, must=tile_edges(m, 128))
    y_ref = oracle.transform(syn.bf16_bits(x[torch.from_numpy(rows)]), syn.bf16_bits(t), bs)
    assert int((y[rows] != y_ref).sum()) == 0, "y differs from the exactly rounded sum"
    packed, sf_lin = oracle.quantize(y_ref, gs, k=k)
    assert int((got_pk[rows] != packed).sum()) == 0, "packed codes differ end to end"
    assert int((gather_scales(got_sf, rows, sf_lin.shape[1], k) != sf_lin).sum()) == 0, "scales differ end to end"


@pytest.mark.parametrize("bs", [16, 32, 64, 128])
def test_transform_quant_full_size_sampled(bs):
    """The transform workload's M = 4096, K = 4096 at full size (32 x 32 tiles
    of 128 x 128 over the persistent CTAs); sampled rows, tile edges included,
    checked as in test_transform_quant_parity."""
    p = [q for q in syn.transform_fused() if q.m == 4096 and q.bs == bs][0]
    L = syn.make_layer(p)
    got_pk, got_sf, y = _gpu_quant_export(L.x, p.k, L.gs_x, L.t, bs)
    rows = sample_indices(p.m, 48, seed=bs, must=tile_edges(p.m, 128))
    packed, sf_lin = oracle.quantize(y[rows], L.gs_x, k=p.k)
    _assert_bytes_equal(got_pk[rows], packed, f"packed rows vs oracle(y) bs={bs}")
    _assert_bytes_equal(gather_scales(got_sf, rows, sf_lin.shape[1], p.k), sf_lin, f"scale rows bs={bs}")
    # the tiled buffer holds exactly these scales plus zero padding (rows are all < m here)
    full = oracle.unswizzle(got_sf, p.m, sf_lin.shape[1])
    assert np.array_equal(oracle.swizzle(full), got_sf)
    _check_transform_y(y[rows], L.x, L.t, bs, rows=rows)


def test_transform_quant_odd_k():
    """k = 4112 (multiple of 16, not of 32): the last scale block is K padding."""
    x = syn.bf16_student_t(40, 4112, 3, seed=75)
    t = syn.random_hadamard_transform(16, seed=75)
    got_pk, got_sf, y = _gpu_quant_export(x, 4112, 3.0, t, 16)
    packed, sf_lin = oracle.quantize(y, 3.0, k=4112)
    _assert_bytes_equal(got_pk, packed, "packed")
    _assert_bytes_equal(got_sf, oracle.swizzle(sf_lin), "scales")
    _check_transform_y(y, x, t, 16)


@pytest.mark.parametrize("m,k", [(65536, 16384), (8192, 4096)])
def test_quant_sweep_full_size_sampled(m, k):
    """Largest sweep points, run at full size on the GPU; the oracle checks a
    sample of rows (rows are independent)."""
    x = syn.bf16_normal((m, k), 1.0, seed=4500 + m % 1000 + k % 1000, device="cuda")
    gs = syn.global_scale(x)
    got = _gpu_quant(x, k, gs)
    rows = sample_indices(m, 24, seed=m + k, must=[127, 128, m - 2])
    xs = x[torch.from_numpy(rows).cuda()].cpu()
    packed, sf_lin = oracle.quantize(syn.bf16_bits(xs), gs, k=k)
    _assert_bytes_equal(got[0][rows], packed, "packed rows")
    _assert_bytes_equal(gather_scales(got[1], rows, sf_lin.shape[1], k), sf_lin, "scale rows")
    # padded scale rows beyond m are zero
    mp, cp = nv.scale_shape(m, k)
    if mp > m:
        pad = oracle.unswizzle(got[1], mp, cp)[m:]
        assert (pad == 0).all()


def test_quant_zero_rows_is_a_noop():
    x = torch.zeros((0, 64), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_quant_act(x, 0, 64, 64, dev_scalar(1.0), None, 0, None, None)
