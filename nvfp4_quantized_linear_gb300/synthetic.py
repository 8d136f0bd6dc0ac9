"""Seeded synthetic workloads for the NVFP4 linear (inputs only).

This module draws the tensors that both the CUDA path and the CPU oracle are
fed; it holds none of the quantization, GEMM or transform arithmetic.  It
depends on torch (for its seeded generator) and numpy only, and nothing else in
this package, so the tests may hand the very same bytes to both sides.

Shapes and distributions are the layer workloads of the benchmark suite:
Llama-3.1-8B and Qwen3-32B decoder linears, a transform-fused 4096x4096 layer, a
padded-K layer with bias and an activation-quantization bandwidth sweep (the
pages name these models and the transform but print no data; random tensors of
those shapes stand in for the checkpoints and prompts).  The seed of a problem
is (zero-based workload index) * 1000 + (problem index within the workload).

Calibration constants that a deployment computes once on the host are part of
the synthetic layer too: the static global scale 448*6/amax (the maximum block
scale times the maximum FP4 value, over the tensor's absolute maximum) and
alpha = 1/(gs_x*gs_w), both binary32.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np
import torch

FP4_MAX = 6.0
E4M3_MAX = 448.0


# ------------------------------------------------------------ primitives ----

def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def bf16_normal(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """N(0, std^2) rounded to bf16."""
    g = _gen(seed, device)
    return (torch.randn(*shape, generator=g, device=device, dtype=torch.float32) * std).to(torch.bfloat16)


def bf16_outlier_channels(m: int, k: int, seed: int, frac: float = 0.001, factor: float = 50.0,
                          device="cpu") -> torch.Tensor:
    """N(0,1) activations with round(frac*k) seeded channels scaled by `factor`."""
    g = _gen(seed, device)
    x = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
    n_out = max(1, int(round(frac * k)))
    gc = _gen(seed + 500_000)
    ch = torch.randperm(k, generator=gc)[:n_out].to(device)
    x[:, ch] *= factor
    return x.to(torch.bfloat16)


def bf16_student_t(m: int, k: int, nu: int, seed: int, device="cpu") -> torch.Tensor:
    """Student-t(nu) samples z / sqrt(chi2_nu / nu), integer nu, rounded to bf16."""
    g = _gen(seed, device)
    z = torch.randn(m, k, generator=g, device=device, dtype=torch.float32)
    chi2 = torch.zeros(m, k, device=device, dtype=torch.float32)
    for _ in range(nu):
        chi2 += torch.randn(m, k, generator=g, device=device, dtype=torch.float32) ** 2
    return (z / torch.sqrt(chi2 / nu)).to(torch.bfloat16)


def sylvester_hadamard(n: int) -> np.ndarray:
    """Sylvester construction of the n x n +-1 Hadamard matrix (n a power of 2)."""
    assert n > 0 and (n & (n - 1)) == 0
    h = np.ones((1, 1), np.int64)
    while h.shape[0] < n:
        h = np.block([[h, h], [h, -h]])
    return h


def random_hadamard_transform(bs: int, seed: int) -> torch.Tensor:
    """T = H_bs * diag(+-1) / sqrt(bs), rounded to bf16 (the transform page's
    HadamardTransform after its 1/sqrt(n) fold; random signs make it a random
    orthogonal block)."""
    g = _gen(seed)
    signs = (torch.randint(0, 2, (bs,), generator=g) * 2 - 1).numpy().astype(np.float64)
    t = sylvester_hadamard(bs).astype(np.float64) * signs[None, :] / math.sqrt(bs)
    return torch.from_numpy(t).to(torch.bfloat16)


def global_scale(x: torch.Tensor) -> float:
    """Static per-tensor scale gs = fl32(448*6 / amax|x|) (binary32)."""
    amax = np.float32(x.detach().abs().max().float().cpu().item())
    return float(np.float32(E4M3_MAX * FP4_MAX) / amax)


def alpha_of(gs_x: float, gs_w: float) -> float:
    """alpha = fl32(1 / fl32(gs_x * gs_w))."""
    return float(np.float32(1.0) / (np.float32(gs_x) * np.float32(gs_w)))


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a bf16 tensor as a uint16 numpy array (host copy)."""
    assert t.dtype == torch.bfloat16, t.dtype
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------- workloads ----

@dataclasses.dataclass(frozen=True)
class Problem:
    workload: str
    name: str
    m: int
    k: int
    n: int
    seed: int
    x_kind: str = "normal"          # normal | outlier | student_t
    bias: bool = False
    bs: int = 0                     # block-diagonal transform size, 0 = none
    n_out: int | None = None        # output slice (None = n)

    @property
    def n_keep(self) -> int:
        return self.n if self.n_out is None else self.n_out

    @property
    def flops(self) -> int:
        return 2 * self.m * self.n_keep * self.k


LLAMA_SHAPES = [("qkv", 4096, 6144), ("o", 4096, 4096), ("gate_up", 4096, 28672), ("down", 14336, 4096)]
LLAMA_M = [1, 16, 128, 1024, 8192]
QWEN_SHAPES = [("qkv", 5120, 10240), ("o", 8192, 5120), ("gate_up", 5120, 51200), ("down", 25600, 5120)]
QWEN_M = [64, 2048, 16384]
XFORM_BS = [16, 32, 64, 128]
XFORM_M = [16, 4096]
PAD_K = [4104, 5128]
PAD_M = [1, 16, 128, 1024, 8192]
SWEEP_M = [1, 16, 128, 1024, 8192, 65536]
SWEEP_K = [4096, 16384]


def tiny() -> list[Problem]:
    return [Problem("tiny", "tiny", 16, 256, 128, seed=0)]


def llama(m_values=LLAMA_M) -> list[Problem]:
    out = []
    for mi, m in enumerate(m_values):
        for si, (name, k, n) in enumerate(LLAMA_SHAPES):
            out.append(Problem("llama3.1-8b", name, m, k, n, seed=1000 + mi * len(LLAMA_SHAPES) + si))
    return out


def qwen(m_values=QWEN_M) -> list[Problem]:
    out = []
    for mi, m in enumerate(m_values):
        for si, (name, k, n) in enumerate(QWEN_SHAPES):
            out.append(Problem("qwen3-32b", name, m, k, n, seed=2000 + mi * len(QWEN_SHAPES) + si,
                               x_kind="outlier"))
    return out


def transform_fused() -> list[Problem]:
    out = []
    i = 0
    for m in XFORM_M:
        for bs in XFORM_BS:
            out.append(Problem("transform", f"bs{bs}", m, 4096, 4096, seed=3000 + i, x_kind="student_t", bs=bs))
            i += 1
    return out


def padded(n_out: int | None = None) -> list[Problem]:
    out = []
    i = 0
    for m in PAD_M:
        for k in PAD_K:
            out.append(Problem("padded", f"k{k}", m, k, 11008, seed=4000 + i, bias=True, n_out=n_out))
            i += 1
    return out


def quant_sweep() -> list[tuple[int, int, int]]:
    """(m, k, seed) points of the activation-quantization bandwidth sweep."""
    out = []
    i = 0
    for m in SWEEP_M:
        for k in SWEEP_K:
            out.append((m, k, 4500 + i))
            i += 1
    return out


@dataclasses.dataclass
class LayerTensors:
    x: torch.Tensor          # [m, k] bf16
    w: torch.Tensor          # [n, k] bf16
    bias: torch.Tensor | None
    t: torch.Tensor | None   # [bs, bs] bf16
    gs_x: float
    gs_w: float
    alpha: float


def make_activation(p: Problem, device="cpu", m: int | None = None) -> torch.Tensor:
    m = p.m if m is None else m
    if p.x_kind == "normal":
        return bf16_normal((m, p.k), 1.0, p.seed, device)
    if p.x_kind == "outlier":
        return bf16_outlier_channels(m, p.k, p.seed, device=device)
    if p.x_kind == "student_t":
        return bf16_student_t(m, p.k, 3, p.seed, device)
    raise ValueError(p.x_kind)


def transformed_amax(x: torch.Tensor, t: torch.Tensor) -> float:
    """max |x * blockdiag(T)| in float64: the calibration statistic of a layer
    whose activation is transformed before quantization (an estimate; it only
    sets the static global scale)."""
    bs = t.shape[0]
    xv = x.detach().double().cpu().reshape(-1, bs)
    return float((xv @ t.detach().double().cpu()).abs().max().item())


def make_layer(p: Problem, device="cpu") -> LayerTensors:
    """All tensors of one problem.  The activation global scale is calibrated
    on the activation the quantizer will see: x itself, or x * blockdiag(T)
    for the transform workload."""
    x = make_activation(p, device)
    w = bf16_normal((p.n, p.k), 0.02, p.seed + 100_000, device)
    bias = bf16_normal((p.n_keep,), 0.1, p.seed + 200_000, device) if p.bias else None
    t = random_hadamard_transform(p.bs, p.seed + 300_000).to(device) if p.bs else None
    gs_w = global_scale(w)
    if t is None:
        gs_x = global_scale(x)
    else:
        gs_x = float(np.float32(E4M3_MAX * FP4_MAX) / np.float32(transformed_amax(x, t)))
    return LayerTensors(x, w, bias, t, gs_x, gs_w, alpha_of(gs_x, gs_w))
