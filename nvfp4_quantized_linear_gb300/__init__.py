"""NVFP4 W4A4 linear layer for GB300 (sm_103a): Python binding of ``include/nvfp4.h``.

The functions below carry the C entry points' names and arguments and do
argument marshalling only (tensor -> device pointer, current CUDA stream);
every step of the computation runs in the CUDA library
``libnvfp4_gb300.so``.  There is no fallback: if the library is missing or the
device is not compute capability 10.3, calls raise.

Tensors: bf16 activations/weights/bias/outputs are ``torch.bfloat16`` CUDA
tensors (or any dtype viewed as raw 16-bit storage), packed FP4 and scales are
``torch.uint8``, global scales and alpha are 1-element ``torch.float32``
device tensors.  Row strides are taken from the tensors (``stride(0)``) and the
innermost stride must be 1.
"""
from __future__ import annotations

import ctypes
import os
import threading

__all__ = [
    "NVFP4_OK", "Nvfp4Error", "library_path", "load_library", "build",
    "nvfp4_abi_version", "nvfp4_is_supported", "nvfp4_last_error_string", "nvfp4_device_error",
    "nvfp4_packed_bytes", "nvfp4_scale_bytes", "nvfp4_linear_workspace_bytes",
    "nvfp4_prepare_weight", "nvfp4_quant_act", "nvfp4_quant_act_export_y", "nvfp4_act_global_scale", "nvfp4_mxfp4_scale_bytes", "nvfp4_mxfp4_quant_act",
    "nvfp4_mxfp4_gemm", "nvfp4_mxfp4_linear_workspace_bytes", "nvfp4_mxfp4_linear", "mxfp4_linear",
    "nvfp4_gemm", "nvfp4_gemm_ex", "nvfp4_grouped_gemm", "nvfp4_linear", "nvfp4_linear_noalloc",
    "padded_k", "scale_shape", "quant_act", "quant_act_mx", "prepare_weight", "linear", "act_global_scale",
]

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libnvfp4_gb300.so")
_lock = threading.Lock()
_lib = None

NVFP4_OK = 0
STATUS_NAMES = {0: "NVFP4_OK", 1: "NVFP4_ERR_INVALID_ARG", 2: "NVFP4_ERR_UNSUPPORTED_DEVICE",
                3: "NVFP4_ERR_ALIGNMENT", 4: "NVFP4_ERR_ALIAS", 5: "NVFP4_ERR_CUDA", 6: "NVFP4_ERR_TIMEOUT",
                7: "NVFP4_ERR_WORKSPACE"}

# (name, restype, argtypes) of every exported symbol of include/nvfp4.h
_P, _I64, _I32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int, ctypes.c_size_t
EXPORTS = [
    ("nvfp4_abi_version", _I32, []),
    ("nvfp4_is_supported", _I32, [_I32, ctypes.c_char_p, _SZ]),
    ("nvfp4_last_error_string", ctypes.c_char_p, []),
    ("nvfp4_device_error", _I32, [_I32]),
    ("nvfp4_packed_bytes", _SZ, [_I64, _I64]),
    ("nvfp4_scale_bytes", _SZ, [_I64, _I64]),
    ("nvfp4_linear_workspace_bytes", _SZ, [_I64, _I64, _I64]),
    ("nvfp4_prepare_weight", _I32, [_P, _I64, _I64, _I64, _P, _P, _P, _P]),
    ("nvfp4_quant_act", _I32, [_P, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _P]),
    ("nvfp4_quant_act_export_y", _I32, [_P, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _P, _P]),
    ("nvfp4_act_global_scale", _I32, [_P, _I64, _I64, _I64, _P, _I32, _P, _P, _P, _P]),
    ("nvfp4_mxfp4_scale_bytes", _SZ, [_I64, _I64]),
    ("nvfp4_mxfp4_quant_act", _I32, [_P, _I64, _I64, _I64, _P, _P, _P]),
    ("nvfp4_mxfp4_gemm", _I32, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _P, _I64, _P]),
    ("nvfp4_mxfp4_linear_workspace_bytes", _SZ, [_I64, _I64, _I64]),
    ("nvfp4_mxfp4_linear", _I32, [_P, _I64, _I64, _I64, _P, _P, _I64, _I64, _P, _P, _I64, _P, _SZ, _P]),
    ("nvfp4_gemm", _I32, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _P, _P, _I64, _P]),
    ("nvfp4_grouped_gemm", _I32, [_P, _P, _I64, _P, _I32, _P, _P, _I64, _I64, _P, _P, _P, _I64, _P]),
    ("nvfp4_gemm_ex", _I32, [_P, _P, _I64, _P, _P, _I64, _I64, _I64, _P, _P, _P, _I64, _I32, ctypes.c_uint64, _I32,
                             _P]),
    ("nvfp4_linear", _I32, [_P, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _I64, _I64, _P, _P, _P, _I64,
                            _P, _SZ, _P]),
    ("nvfp4_linear_noalloc", _I32, [_P, _I64, _I64, _I64, _P, _P, _I32, _P, _P, _I64, _I64, _P, _P, _P, _I64,
                                    _P]),
]


class Nvfp4Error(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def library_path() -> str:
    return _LIB_PATH


def build(force: bool = False) -> str:
    """Compile the CUDA library in-tree (nvcc, sm_103a)."""
    from . import _build
    return _build.build(force=force)


def load_library():
    """Load ``libnvfp4_gb300.so`` (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"NVFP4 CUDA library not built ({_LIB_PATH} missing); "
                               "run nvfp4_quantized_linear_gb300.build()")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, res, args in EXPORTS:
            fn = getattr(lib, name)
            fn.restype = res
            fn.argtypes = args
        _lib = lib
        return lib


def _check(status: int):
    if status != NVFP4_OK:
        raise Nvfp4Error(status, load_library().nvfp4_last_error_string().decode())


def _ptr(t):
    """Device pointer of a tensor (None -> NULL)."""
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream):
    if stream is None:
        import torch
        return torch.cuda.current_stream().cuda_stream
    if isinstance(stream, int):
        return stream
    return stream.cuda_stream


def _ld(t, name):
    if t.dim() != 2 or t.stride(1) != 1:
        raise ValueError(f"{name} must be a 2-D tensor with unit inner stride")
    return t.stride(0)


# ------------------------------------------------------------- queries ----

def padded_k(k: int) -> int:
    return (k + 31) // 32 * 32


def scale_shape(rows: int, k: int) -> tuple[int, int]:
    """(padded rows, padded scale columns) of a tiled scale tensor."""
    return (rows + 127) // 128 * 128, (padded_k(k) // 16 + 3) // 4 * 4


def nvfp4_abi_version() -> int:
    return load_library().nvfp4_abi_version()


def nvfp4_is_supported(device: int = 0) -> tuple[bool, str | None]:
    buf = ctypes.create_string_buffer(256)
    st = load_library().nvfp4_is_supported(device, buf, 256)
    return (st == NVFP4_OK, None if st == NVFP4_OK else buf.value.decode())


def nvfp4_last_error_string() -> str:
    return load_library().nvfp4_last_error_string().decode()


def nvfp4_device_error(clear: bool = True) -> None:
    _check(load_library().nvfp4_device_error(1 if clear else 0))


def nvfp4_packed_bytes(rows: int, k: int) -> int:
    return load_library().nvfp4_packed_bytes(rows, k)


def nvfp4_scale_bytes(rows: int, k: int) -> int:
    return load_library().nvfp4_scale_bytes(rows, k)


def nvfp4_linear_workspace_bytes(m: int, k: int, n_w: int) -> int:
    return load_library().nvfp4_linear_workspace_bytes(m, k, n_w)


# ---------------------------------------------------------- operations ----

def nvfp4_prepare_weight(w, n: int, k: int, ldw: int, w_gs, w_fp4, w_sf, stream=None) -> None:
    _check(load_library().nvfp4_prepare_weight(_ptr(w), n, k, ldw, _ptr(w_gs), _ptr(w_fp4), _ptr(w_sf),
                                               _stream(stream)))


def nvfp4_quant_act(x, m: int, k: int, ldx: int, gs, transform, bs: int, x_fp4, x_sf, stream=None) -> None:
    _check(load_library().nvfp4_quant_act(_ptr(x), m, k, ldx, _ptr(gs), _ptr(transform), bs, _ptr(x_fp4),
                                          _ptr(x_sf), _stream(stream)))


def nvfp4_quant_act_export_y(x, m: int, k: int, ldx: int, gs, transform, bs: int, x_fp4, x_sf, y,
                             stream=None) -> None:
    _check(load_library().nvfp4_quant_act_export_y(_ptr(x), m, k, ldx, _ptr(gs), _ptr(transform), bs, _ptr(x_fp4),
                                                   _ptr(x_sf), _ptr(y), _stream(stream)))


def nvfp4_act_global_scale(x, m: int, k: int, ldx: int, transform, bs: int, w_gs, gs_out, alpha_out,
                           stream=None) -> None:
    _check(load_library().nvfp4_act_global_scale(_ptr(x), m, k, ldx, _ptr(transform), bs, _ptr(w_gs),
                                                 _ptr(gs_out), _ptr(alpha_out), _stream(stream)))


def nvfp4_mxfp4_scale_bytes(rows: int, k: int) -> int:
    return load_library().nvfp4_mxfp4_scale_bytes(rows, k)


def nvfp4_mxfp4_quant_act(x, m: int, k: int, ldx: int, x_fp4, x_sf, stream=None) -> None:
    _check(load_library().nvfp4_mxfp4_quant_act(_ptr(x), m, k, ldx, _ptr(x_fp4), _ptr(x_sf), _stream(stream)))


def nvfp4_mxfp4_gemm(a_fp4, a_sf, m: int, w_fp4, w_sf, n_w: int, n_out: int, k: int, bias, out, ldo: int,
                     stream=None) -> None:
    _check(load_library().nvfp4_mxfp4_gemm(_ptr(a_fp4), _ptr(a_sf), m, _ptr(w_fp4), _ptr(w_sf), n_w, n_out, k,
                                           _ptr(bias), _ptr(out), ldo, _stream(stream)))


def nvfp4_mxfp4_linear_workspace_bytes(m: int, k: int, n_w: int) -> int:
    return load_library().nvfp4_mxfp4_linear_workspace_bytes(m, k, n_w)


def nvfp4_mxfp4_linear(x, m: int, k: int, ldx: int, w_fp4, w_sf, n_w: int, n_out: int, bias, out, ldo: int,
                       workspace, workspace_bytes: int, stream=None) -> None:
    _check(load_library().nvfp4_mxfp4_linear(_ptr(x), m, k, ldx, _ptr(w_fp4), _ptr(w_sf), n_w, n_out, _ptr(bias),
                                             _ptr(out), ldo, _ptr(workspace), workspace_bytes, _stream(stream)))


def nvfp4_gemm(a_fp4, a_sf, m: int, w_fp4, w_sf, n_w: int, n_out: int, k: int, alpha, bias, out, ldo: int,
               stream=None) -> None:
    _check(load_library().nvfp4_gemm(_ptr(a_fp4), _ptr(a_sf), m, _ptr(w_fp4), _ptr(w_sf), n_w, n_out, k,
                                     _ptr(alpha), _ptr(bias), _ptr(out), ldo, _stream(stream)))


def nvfp4_grouped_gemm(a_fp4, a_sf, rows: int, group_offsets, num_groups: int, w_fp4, w_sf, n: int, k: int, alpha,
                       bias, out, ldo: int, stream=None) -> None:
    _check(load_library().nvfp4_grouped_gemm(_ptr(a_fp4), _ptr(a_sf), rows, _ptr(group_offsets), num_groups,
                                             _ptr(w_fp4), _ptr(w_sf), n, k, _ptr(alpha), _ptr(bias), _ptr(out), ldo,
                                             _stream(stream)))


def nvfp4_gemm_ex(a_fp4, a_sf, m: int, w_fp4, w_sf, n_w: int, n_out: int, k: int, alpha, bias, out, ldo: int,
                  kernel: int = 0, wait_limit_ns: int = 0, drill: int = 0, stream=None) -> None:
    _check(load_library().nvfp4_gemm_ex(_ptr(a_fp4), _ptr(a_sf), m, _ptr(w_fp4), _ptr(w_sf), n_w, n_out, k,
                                        _ptr(alpha), _ptr(bias), _ptr(out), ldo, kernel, wait_limit_ns, drill,
                                        _stream(stream)))


def nvfp4_linear(x, m: int, k: int, ldx: int, gs, transform, bs: int, w_fp4, w_sf, n_w: int, n_out: int,
                 alpha, bias, out, ldo: int, workspace, workspace_bytes: int, stream=None) -> None:
    _check(load_library().nvfp4_linear(_ptr(x), m, k, ldx, _ptr(gs), _ptr(transform), bs, _ptr(w_fp4),
                                       _ptr(w_sf), n_w, n_out, _ptr(alpha), _ptr(bias), _ptr(out), ldo,
                                       _ptr(workspace), workspace_bytes, _stream(stream)))


def nvfp4_linear_noalloc(x, m: int, k: int, ldx: int, gs, transform, bs: int, w_fp4, w_sf, n_w: int, n_out: int,
                         alpha, bias, out, ldo: int, stream=None) -> None:
    """nvfp4_linear with the library's built-in 16 MiB scratch instead of a
    workspace, for callers that cannot allocate device memory (see the C
    header for the limit and the sharing rules)."""
    _check(load_library().nvfp4_linear_noalloc(_ptr(x), m, k, ldx, _ptr(gs), _ptr(transform), bs, _ptr(w_fp4),
                                               _ptr(w_sf), n_w, n_out, _ptr(alpha), _ptr(bias), _ptr(out), ldo,
                                               _stream(stream)))


# --------------------------------------------- tensor-level conveniences ----
# Thin helpers that allocate the caller-owned outputs with torch and call the
# entry points above; they add no computation.

def quant_act(x, gs, transform=None, bs: int = 0, stream=None):
    """Quantize a [m, k] bf16 CUDA tensor; returns (x_fp4 [m, Kp/2], x_sf flat)."""
    import torch
    m, k = x.shape
    x_fp4 = torch.empty((m, padded_k(k) // 2), dtype=torch.uint8, device=x.device)
    x_sf = torch.empty(max(nvfp4_scale_bytes(m, k), 1), dtype=torch.uint8, device=x.device)
    nvfp4_quant_act(x, m, k, _ld(x, "x"), gs, transform, bs if transform is not None else 0, x_fp4, x_sf, stream)
    return x_fp4, x_sf


def act_global_scale(x, transform=None, bs: int = 0, w_gs=None, stream=None):
    """Dynamic scale of a [m, k] bf16 CUDA tensor; returns (gs, alpha) as
    1-element fp32 device tensors (alpha is None without w_gs)."""
    import torch
    m, k = x.shape
    gs = torch.empty(1, dtype=torch.float32, device=x.device)
    alpha = torch.empty(1, dtype=torch.float32, device=x.device) if w_gs is not None else None
    nvfp4_act_global_scale(x, m, k, _ld(x, "x"), transform, bs if transform is not None else 0, w_gs, gs, alpha,
                           stream)
    return gs, alpha


def quant_act_mx(x, stream=None):
    """MXFP4-quantize a [m, k] bf16 CUDA tensor; returns (x_fp4 [m, Kp/2], x_sf flat E8M0 codes)."""
    import torch
    m, k = x.shape
    x_fp4 = torch.empty((m, padded_k(k) // 2), dtype=torch.uint8, device=x.device)
    x_sf = torch.empty(max(nvfp4_mxfp4_scale_bytes(m, k), 1), dtype=torch.uint8, device=x.device)
    nvfp4_mxfp4_quant_act(x, m, k, _ld(x, "x"), x_fp4, x_sf, stream)
    return x_fp4, x_sf


def mxfp4_linear(x, w_fp4, w_sf, k: int, n_out: int, bias=None, out=None, workspace=None, stream=None):
    """out[m, n_out] = MXFP4 linear of a [m, k] bf16 CUDA tensor against a weight
    quantized by quant_act_mx (allocates out/workspace if not given)."""
    import torch
    m = x.shape[0]
    n_w = w_fp4.shape[0]
    if out is None:
        out = torch.empty((m, n_out), dtype=torch.bfloat16, device=x.device)
    if workspace is None:
        workspace = torch.empty(max(nvfp4_mxfp4_linear_workspace_bytes(m, k, n_w), 1), dtype=torch.uint8,
                                device=x.device)
    nvfp4_mxfp4_linear(x, m, k, _ld(x, "x"), w_fp4, w_sf, n_w, n_out, bias, out, _ld(out, "out"), workspace,
                       workspace.numel(), stream)
    return out


def prepare_weight(w, w_gs, stream=None):
    """Prepare a [n, k] bf16 CUDA weight; returns (w_fp4 [n, Kp/2], w_sf flat)."""
    import torch
    n, k = w.shape
    w_fp4 = torch.empty((n, padded_k(k) // 2), dtype=torch.uint8, device=w.device)
    w_sf = torch.empty(max(nvfp4_scale_bytes(n, k), 1), dtype=torch.uint8, device=w.device)
    nvfp4_prepare_weight(w, n, k, _ld(w, "w"), w_gs, w_fp4, w_sf, stream)
    return w_fp4, w_sf


def linear(x, w_fp4, w_sf, k: int, n_out: int, gs, alpha, bias=None, transform=None, bs: int = 0,
           out=None, workspace=None, stream=None):
    """out[m, n_out] = NVFP4 linear of a [m, k] bf16 CUDA tensor (allocates out/workspace if not given)."""
    import torch
    m = x.shape[0]
    n_w = w_fp4.shape[0]
    if out is None:
        out = torch.empty((m, n_out), dtype=torch.bfloat16, device=x.device)
    need = nvfp4_linear_workspace_bytes(m, k, n_w)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=x.device)
    nvfp4_linear(x, m, k, _ld(x, "x"), gs, transform, bs if transform is not None else 0, w_fp4, w_sf, n_w, n_out,
                 alpha, bias, out, _ld(out, "out"), workspace, workspace.numel(), stream)
    return out
