"""NVFP4 W4A4 linear -- plain CPU oracle (ctypes wrapper over ``nvfp4_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The test suite, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` are the only callers.  The product path (the
CUDA library and its Python binding) never imports this package, and this
package imports nothing from the product.

Every function takes and returns numpy arrays; bf16 tensors travel as their raw
``uint16`` bit patterns so that nothing here depends on a bf16 numpy dtype.
Each function names, in its docstring, the page passage or reading it follows;
the C file's header lists the readings in full.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "nvfp4_oracle.c")
_LIB = os.path.join(_HERE, "libnvfp4_oracle.so")
_lock = threading.Lock()
_lib = None

# -O2, no fast-math, no contraction of a*b+c into fma: every step stays the
# IEEE operation it is written as.
CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off", "-fno-fast-math"]


def build(force: bool = False) -> str:
    """Compile the oracle with the host C compiler (gcc) and return the .so path."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_dec_e2m1.restype = ctypes.c_double
    lib.oracle_dec_e2m1.argtypes = [ctypes.c_uint8]
    lib.oracle_enc_e2m1.restype = ctypes.c_uint8
    lib.oracle_enc_e2m1.argtypes = [ctypes.c_float]
    lib.oracle_dec_e4m3.restype = ctypes.c_double
    lib.oracle_dec_e4m3.argtypes = [ctypes.c_uint8]
    lib.oracle_enc_e4m3.restype = ctypes.c_uint8
    lib.oracle_enc_e4m3.argtypes = [ctypes.c_float]
    lib.oracle_bf16_to_f32.restype = ctypes.c_float
    lib.oracle_bf16_to_f32.argtypes = [ctypes.c_uint16]
    lib.oracle_f32_to_bf16.restype = ctypes.c_uint16
    lib.oracle_f32_to_bf16.argtypes = [ctypes.c_float]
    lib.oracle_quantize_rows.restype = None
    lib.oracle_quantize_rows.argtypes = [P, I64, I64, I64, ctypes.c_float, P, P]
    lib.oracle_swizzle_offset.restype = I64
    lib.oracle_swizzle_offset.argtypes = [I64, I64, I64]
    lib.oracle_swizzle.restype = None
    lib.oracle_swizzle.argtypes = [P, I64, I64, P]
    lib.oracle_unswizzle.restype = None
    lib.oracle_unswizzle.argtypes = [P, I64, I64, P]
    lib.oracle_transform_rows.restype = None
    lib.oracle_transform_rows.argtypes = [P, I64, I64, I64, P, ctypes.c_int, P]
    lib.oracle_mx_scale_code.restype = ctypes.c_uint8
    lib.oracle_mx_scale_code.argtypes = [ctypes.c_float]
    lib.oracle_dec_e8m0.restype = ctypes.c_double
    lib.oracle_dec_e8m0.argtypes = [ctypes.c_uint8]
    lib.oracle_quantize_rows_mx.restype = None
    lib.oracle_quantize_rows_mx.argtypes = [P, I64, I64, I64, P, P]
    lib.oracle_gemm_mx.restype = None
    lib.oracle_gemm_mx.argtypes = [P, P, P, P, I64, P, I64, P, I64, P, P]
    lib.oracle_act_global_scale.restype = ctypes.c_float
    lib.oracle_act_global_scale.argtypes = [P, I64, I64, I64]
    lib.oracle_alpha.restype = ctypes.c_float
    lib.oracle_alpha.argtypes = [ctypes.c_float, ctypes.c_float]
    lib.oracle_gemm.restype = None
    lib.oracle_gemm.argtypes = [P, P, P, P, I64, P, I64, P, I64, ctypes.c_float, P, P]
    _lib = lib
    return lib


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


# ------------------------------------------------------------------ sizes --

def padded_k(k: int) -> int:
    """Kp = roundup(K, 32): the K padding of packed operands (reading R-pad)."""
    return (k + 31) // 32 * 32


def swizzled_shape(rows: int, cols: int) -> tuple[int, int]:
    """(roundup(rows,128), roundup(cols,4)): the padded tiled scale matrix."""
    return (rows + 127) // 128 * 128, (cols + 3) // 4 * 4


# ----------------------------------------------------------------- scalars --

def dec_e2m1(code: int) -> float:
    """FP4 E2M1 code -> value (OCP MX v1.0 element format)."""
    return _load().oracle_dec_e2m1(code)


def enc_e2m1(x: float) -> int:
    """Nearest E2M1 code, ties to even, satfinite, sign kept (readings R-sign)."""
    return _load().oracle_enc_e2m1(x)


def dec_e4m3(code: int) -> float:
    """FP8 E4M3 ("fn", max 448) code -> value (OCP OFP8)."""
    return _load().oracle_dec_e4m3(code)


def enc_e4m3(x: float) -> int:
    """Nearest E4M3 code, ties to even, saturating at 448."""
    return _load().oracle_enc_e4m3(x)


def f32_to_bf16(x: float) -> int:
    return _load().oracle_f32_to_bf16(x)


def bf16_to_f32(h: int) -> float:
    return _load().oracle_bf16_to_f32(h)


def bf16_bits_to_f64(a: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bits (uint16) to float64 (exact)."""
    return (np.asarray(a, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ------------------------------------------------------------------ arrays --

def quantize(x_bits: np.ndarray, gs: float, k: int | None = None):
    """Quantize bf16 rows to NVFP4 (page "TorchNvFp4LinearKernel", apply_weights:
    scaled_fp4_quant with the global scale and K padded to the weight's padding).

    x_bits: [rows, ld] uint16 (bf16 bits); the first ``k`` columns are the data.
    Returns (packed [rows, Kp/2] uint8, sf_lin [rows, Kp/16] uint8 E4M3 codes).
    """
    lib = _load()
    x_bits = _c(x_bits, np.uint16)
    rows, ld = x_bits.shape
    k = ld if k is None else k
    kp = padded_k(k)
    packed = np.zeros((rows, kp // 2), np.uint8)
    sf = np.zeros((rows, kp // 16), np.uint8)
    if rows:
        lib.oracle_quantize_rows(_ptr(x_bits), rows, k, ld, ctypes.c_float(gs), _ptr(packed), _ptr(sf))
    return packed, sf


def mx_scale_code(amax: float) -> int:
    """E8M0 code of an MXFP4 block with absolute maximum amax (reading R-mx)."""
    return int(_load().oracle_mx_scale_code(amax))


def dec_e8m0(code: int) -> float:
    return _load().oracle_dec_e8m0(code)


def quantize_mx(x_bits: np.ndarray, k: int | None = None):
    """Quantize bf16 rows to MXFP4 (page "B12X", the MXFP4 linear backend's
    dynamic activation quantization; OCP MX v1.0 format, reading R-mx).
    Returns (packed [rows, Kp/2] uint8, sf_lin [rows, Kp/32] uint8 E8M0 codes)."""
    lib = _load()
    x_bits = _c(x_bits, np.uint16)
    rows, ld = x_bits.shape
    k = ld if k is None else k
    kp = padded_k(k)
    packed = np.zeros((rows, kp // 2), np.uint8)
    sf = np.zeros((rows, kp // 32), np.uint8)
    if rows:
        lib.oracle_quantize_rows_mx(_ptr(x_bits), rows, k, ld, _ptr(packed), _ptr(sf))
    return packed, sf


def swizzle(sf_lin: np.ndarray) -> np.ndarray:
    """Linear [R, C] scales -> flat tiled layout (reading R-swz), zero padded."""
    lib = _load()
    sf_lin = _c(sf_lin, np.uint8)
    r, c = sf_lin.shape
    rp, cp = swizzled_shape(r, c)
    out = np.zeros(rp * cp, np.uint8)
    lib.oracle_swizzle(_ptr(sf_lin), r, c, _ptr(out))
    return out


def unswizzle(sf_swz: np.ndarray, rows: int, cols: int) -> np.ndarray:
    lib = _load()
    sf_swz = _c(sf_swz, np.uint8).reshape(-1)
    out = np.zeros((rows, cols), np.uint8)
    lib.oracle_unswizzle(_ptr(sf_swz), rows, cols, _ptr(out))
    return out


def swizzle_offset(r: int, c: int, cp: int) -> int:
    return _load().oracle_swizzle_offset(r, c, cp)


def transform(x_bits: np.ndarray, t_bits: np.ndarray, bs: int, k: int | None = None) -> np.ndarray:
    """y = bf16(x * blockdiag(T)) (page "QUTLASS fusedQuantizeNv", HadamardTransform
    snippet; reading R-xform).  Returns [rows, k] uint16 bf16 bits."""
    lib = _load()
    x_bits = _c(x_bits, np.uint16)
    t_bits = _c(t_bits, np.uint16)
    assert t_bits.shape == (bs, bs)
    rows, ld = x_bits.shape
    k = ld if k is None else k
    y = np.zeros((rows, k), np.uint16)
    if rows:
        lib.oracle_transform_rows(_ptr(x_bits), rows, k, ld, _ptr(t_bits), bs, _ptr(y))
    return y


def act_global_scale(x_bits: np.ndarray, t_bits: np.ndarray | None = None, bs: int = 0,
                     k: int | None = None) -> float:
    """Dynamic activation global scale fl32(448*6 / amax) over the tensor, of
    y = bf16(x * blockdiag(T)) when a transform is given (reading R-dyn)."""
    lib = _load()
    x_bits = _c(x_bits, np.uint16)
    rows, ld = x_bits.shape
    k = ld if k is None else k
    if t_bits is not None:
        x_bits = transform(x_bits, t_bits, bs, k)
        ld = k
    return float(lib.oracle_act_global_scale(_ptr(x_bits), rows, k, ld))


def alpha(gs_x: float, gs_w: float) -> float:
    """fl32(1 / fl32(gs_x * gs_w))."""
    return float(_load().oracle_alpha(gs_x, gs_w))


def gemm(a_packed, a_sf_lin, b_packed, b_sf_lin, alpha: float, bias_bits=None,
         rows=None, cols=None) -> np.ndarray:
    """FP64 reference of the NVFP4 linear (page "TorchNvFp4LinearKernel",
    apply_weights: _scaled_mm, then * alpha, slice, + bias; reading R-gemm).

    a_packed [M, Kp/2], a_sf_lin [M, Kp/16], b_packed [N, Kp/2], b_sf_lin [N, Kp/16].
    ``rows``/``cols`` select output rows/columns (default: all).  Returns float64
    [len(rows), len(cols)].
    """
    lib = _load()
    a_packed = _c(a_packed, np.uint8)
    b_packed = _c(b_packed, np.uint8)
    a_sf_lin = _c(a_sf_lin, np.uint8)
    b_sf_lin = _c(b_sf_lin, np.uint8)
    kp = a_packed.shape[1] * 2
    assert b_packed.shape[1] * 2 == kp and a_sf_lin.shape[1] == kp // 16 == b_sf_lin.shape[1]
    rows = np.arange(a_packed.shape[0]) if rows is None else np.asarray(rows)
    cols = np.arange(b_packed.shape[0]) if cols is None else np.asarray(cols)
    rows = _c(rows, np.int64)
    cols = _c(cols, np.int64)
    out = np.zeros((rows.size, cols.size), np.float64)
    bias_p = None
    if bias_bits is not None:
        bias_bits = _c(bias_bits, np.uint16)
        bias_p = _ptr(bias_bits)
    if rows.size and cols.size:
        lib.oracle_gemm(_ptr(a_packed), _ptr(a_sf_lin), _ptr(b_packed), _ptr(b_sf_lin), kp,
                        _ptr(rows), rows.size, _ptr(cols), cols.size, ctypes.c_float(alpha),
                        bias_p, _ptr(out))
    return out


def gemm_mx(a_packed, a_sf_lin, b_packed, b_sf_lin, bias_bits=None, rows=None, cols=None) -> np.ndarray:
    """FP64 reference of an MXFP4 linear (page "B12X", the MXFP4 backend's
    mm_mxfp4; reading R-mx): sum_k deq(A) deq(B) + bias, E8M0 scales per 32
    elements, no global scale.  Arguments as for gemm, with [*, Kp/32] scales."""
    lib = _load()
    a_packed = _c(a_packed, np.uint8)
    b_packed = _c(b_packed, np.uint8)
    a_sf_lin = _c(a_sf_lin, np.uint8)
    b_sf_lin = _c(b_sf_lin, np.uint8)
    kp = a_packed.shape[1] * 2
    assert b_packed.shape[1] * 2 == kp and a_sf_lin.shape[1] == kp // 32 == b_sf_lin.shape[1]
    rows = _c(np.arange(a_packed.shape[0]) if rows is None else np.asarray(rows), np.int64)
    cols = _c(np.arange(b_packed.shape[0]) if cols is None else np.asarray(cols), np.int64)
    out = np.zeros((rows.size, cols.size), np.float64)
    bias_p = None
    if bias_bits is not None:
        bias_keep = _c(bias_bits, np.uint16)          # held until the call returns
        bias_p = _ptr(bias_keep)
    if rows.size and cols.size:
        lib.oracle_gemm_mx(_ptr(a_packed), _ptr(a_sf_lin), _ptr(b_packed), _ptr(b_sf_lin), kp,
                           _ptr(rows), rows.size, _ptr(cols), cols.size, bias_p, _ptr(out))
    return out


def dequantize(packed: np.ndarray, sf_lin: np.ndarray, gs: float) -> np.ndarray:
    """value = e2m1(q) * e4m3(sf) / gs in FP64 (the inverse of ``quantize`` up to
    rounding).  Returns [rows, Kp] float64."""
    packed = _c(packed, np.uint8)
    lo = packed & 0xF
    hi = packed >> 4
    codes = np.stack([lo, hi], axis=-1).reshape(packed.shape[0], -1)
    grid = np.array([dec_e2m1(c) for c in range(16)], np.float64)
    e4 = np.array([dec_e4m3(c) for c in range(256)], np.float64)
    d = np.repeat(e4[sf_lin], 16, axis=1)
    return grid[codes] * d / np.float64(gs)
