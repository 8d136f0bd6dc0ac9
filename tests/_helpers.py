"""Helpers shared by the GPU parity tests (no method arithmetic lives here)."""
from __future__ import annotations

import numpy as np
import torch

import nvfp4_quantized_linear_gb300 as nv
from nvfp4_quantized_linear_gb300 import synthetic as syn

# GEMM tolerance (outputs vs the oracle's FP64 result on identical quantized
# operands): max |err| <= 2e-2 * rms(ref) and ||err||_F / ||ref||_F <= 5e-3.
MAX_ERR_RMS = 2e-2
FROB_REL = 5e-3


def require_library():
    """Build (if needed) and load the CUDA library; a GPU test that cannot run
    it fails instead of falling back to anything."""
    nv.build()
    lib = nv.load_library()
    ok, why = nv.nvfp4_is_supported(torch.cuda.current_device())
    assert ok, f"device not supported: {why}"
    return lib


def dev_scalar(v: float) -> torch.Tensor:
    return torch.tensor([v], dtype=torch.float32, device="cuda")


def sample_indices(n: int, count: int, seed: int, must=()) -> np.ndarray:
    """Sorted unique indices: the edges, tile boundaries in `must`, random rest."""
    rng = np.random.default_rng(seed)
    base = {0, n - 1, *[i for i in must if 0 <= i < n]}
    extra = rng.choice(n, size=min(n, count), replace=False)
    return np.array(sorted(base | set(int(i) for i in extra)), dtype=np.int64)


def tile_edges(n: int, tile: int) -> list[int]:
    out = []
    for t in range(tile, n, tile):
        out += [t - 1, t]
    return out


def gather_scales(sf_flat: np.ndarray, rows: np.ndarray, cols: int, k: int) -> np.ndarray:
    """Linear [len(rows), cols] scales read out of a tiled scale buffer."""
    import oracle
    full = oracle.unswizzle(sf_flat, int(rows.max()) + 1, cols)
    return full[rows]


def assert_gemm_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    err = got - ref
    rms = float(np.sqrt(np.mean(ref * ref)))
    max_err = float(np.abs(err).max()) if err.size else 0.0
    frob = float(np.linalg.norm(err) / max(np.linalg.norm(ref), 1e-300))
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    assert max_err <= MAX_ERR_RMS * rms, f"{what}: max|err| {max_err:.3e} > {MAX_ERR_RMS} * rms {rms:.3e}"
    assert frob <= FROB_REL, f"{what}: rel Frobenius error {frob:.3e} > {FROB_REL}"
    return max_err / max(rms, 1e-300), frob


def bf16_to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


__all__ = ["nv", "syn", "require_library", "dev_scalar", "sample_indices", "tile_edges", "gather_scales",
           "assert_gemm_close", "bf16_to_f64", "MAX_ERR_RMS", "FROB_REL"]
