"""GPU parity of the MXFP4 activation quantizer (nvfp4_mxfp4_quant_act)
against the oracle (reading R-mx): packed E2M1 bytes and tiled E8M0 scale
bytes, padding included, bit for bit."""
import numpy as np
import pytest
import torch

import oracle
from _helpers import gather_scales, nv, require_library, sample_indices, syn, tile_edges

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    return require_library()


def _gpu_mx(x: torch.Tensor, k: int):
    """x: [m, ldx] CUDA tensor, the first k columns are the data."""
    m = x.shape[0]
    fp4 = torch.full((m, nv.padded_k(k) // 2), 0xAB, dtype=torch.uint8, device="cuda")
    sf = torch.full((max(nv.nvfp4_mxfp4_scale_bytes(m, k), 1),), 0xCD, dtype=torch.uint8, device="cuda")
    nv.nvfp4_mxfp4_quant_act(x, m, k, x.stride(0), fp4, sf)
    torch.cuda.synchronize()
    return fp4.cpu().numpy(), sf.cpu().numpy()


def _check(x_cpu: torch.Tensor, k: int):
    got_pk, got_sf = _gpu_mx(x_cpu.cuda(), k)
    packed, sf_lin = oracle.quantize_mx(syn.bf16_bits(x_cpu), k=k)
    assert np.array_equal(got_pk, packed), f"{int((got_pk != packed).sum())} packed bytes differ"
    ref_sf = oracle.swizzle(sf_lin)
    assert np.array_equal(got_sf, ref_sf), f"{int((got_sf != ref_sf).sum())} scale bytes differ"


@pytest.mark.parametrize("m,k,ldx,kind", [
    (1, 4096, 4096, "normal"),
    (16, 256, 256, "normal"),
    (97, 4104, 4112, "outlier"),          # K % 32 = 8: a partial last block, strided rows
    (33, 250, 256, "student_t"),          # K % 16 != 0
    (130, 5128, 5128, "student_t"),       # rows past one 128-row band; scale columns 161 -> 164
    (4096, 4096, 4096, "normal"),
])
def test_mxfp4_shapes_bit_exact(m, k, ldx, kind):
    seed = 5300 + m + k
    if kind == "normal":
        x = syn.bf16_normal((m, ldx), 1.0, seed)
    elif kind == "outlier":
        x = syn.bf16_outlier_channels(m, ldx, seed)
    else:
        x = syn.bf16_student_t(m, ldx, 3, seed)
    _check(x, k)


def test_mxfp4_special_values():
    """Zero blocks, values between 6 and 8 times the scale (saturation), E2M1
    ties, signed zeros, bf16 subnormals and values near the bf16 maximum."""
    rows = []
    rows.append(np.zeros(128))
    ties = np.tile([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, -0.25, -5.0, 7.5, -7.0, 6.0, -0.0, 0.1, 3.0, 1.0], 8)
    rows.append(ties)
    rows.append(np.concatenate([np.full(32, 2.0 ** -130), np.full(32, -(2.0 ** -133)), np.full(32, 3e38),
                                np.linspace(-1e-38, 1e-38, 32)]))
    rng = np.random.default_rng(54)
    rows.append(rng.standard_normal(128) * 2.0 ** rng.integers(-60, 60, 128))
    x = torch.tensor(np.stack(rows), dtype=torch.float32).to(torch.bfloat16)
    _check(x, 128)


def test_mxfp4_full_size_sampled():
    """65536 x 16384 at full size; sampled rows against the oracle."""
    m, k = 65536, 16384
    x = syn.bf16_normal((m, k), 1.0, seed=5400, device="cuda")
    got_pk, got_sf = _gpu_mx(x, k)
    rows = sample_indices(m, 24, seed=5400, must=tile_edges(m, 128)[:6] + [m - 1])
    packed, sf_lin = oracle.quantize_mx(syn.bf16_bits(x[torch.as_tensor(rows, device="cuda")].cpu()), k=k)
    assert np.array_equal(got_pk[rows], packed)
    assert np.array_equal(gather_scales(got_sf, rows, sf_lin.shape[1], k), sf_lin)


def test_mxfp4_zero_rows_is_a_noop():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    nv.nvfp4_mxfp4_quant_act(x, 0, 256, 256, None, None)
