"""Host-side checks of the C ABI (no GPU needed): the library builds and loads,
exports every entry point include/nvfp4.h declares, answers size queries, and
rejects invalid calls with the documented status before touching a device.

Fake device addresses below are only ever used in calls that must fail
validation, so no kernel can be launched on them.
"""
import os
import re

import pytest

import nvfp4_quantized_linear_gb300 as nv

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "nvfp4.h")

OK, INVALID, UNSUPPORTED, ALIGN, ALIAS, CUDA, TIMEOUT, WORKSPACE = range(8)
A = 1 << 20          # aligned fake addresses, far apart
B = 1 << 30
C = 1 << 34
D = 1 << 36


@pytest.fixture(scope="module")
def lib():
    nv.build()
    return nv.load_library()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(", text)))


def test_header_declarations_are_all_exported(lib):
    names = declared_functions()
    assert len(names) >= 11
    for name in names:
        assert hasattr(lib, name), name
    assert sorted(n for n, _, _ in nv.EXPORTS) == names


def _prototypes():
    """name -> parameter count of every function declared in the header."""
    text = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for name, params in re.findall(r"\b(nvfp4_[a-z0-9_]+)\s*\(([^)]*)\)\s*;", text):
        params = params.strip()
        out[name] = 0 if params in ("", "void") else params.count(",") + 1
    return out


def test_binding_arity_matches_the_header():
    protos = _prototypes()
    assert set(protos) == {n for n, _, _ in nv.EXPORTS}
    for name, _, args in nv.EXPORTS:
        assert len(args) == protos[name], (name, len(args), protos[name])


def test_header_is_plain_c():
    """include/nvfp4.h compiles as C11 (and as C++17) on its own: a C ABI."""
    import shutil
    import subprocess
    import tempfile
    if shutil.which("gcc") is None:
        pytest.skip("no gcc")
    with tempfile.TemporaryDirectory() as d:
        src = os.path.join(d, "use.c")
        with open(src, "w") as f:
            f.write('#include "nvfp4.h"\nint f(void) { return nvfp4_abi_version() + (int)NVFP4_ERR_ALIAS; }\n')
        inc = os.path.dirname(HEADER)
        subprocess.check_call(["gcc", "-std=c11", "-Wall", "-Werror", "-fsyntax-only", "-I", inc, src])
        subprocess.check_call(["g++", "-std=c++17", "-Wall", "-Werror", "-fsyntax-only", "-x", "c++", "-I", inc, src])


def test_abi_version(lib):
    assert nv.nvfp4_abi_version() == 1


def test_size_queries(lib):
    assert nv.nvfp4_packed_bytes(16, 256) == 16 * 128
    assert nv.nvfp4_packed_bytes(3, 40) == 3 * 32            # K padded to 64
    assert nv.nvfp4_scale_bytes(16, 256) == 128 * 16
    assert nv.nvfp4_scale_bytes(1, 4104) == 128 * 260        # 258 scale columns padded to 260
    assert nv.nvfp4_scale_bytes(129, 32) == 256 * 4
    assert nv.nvfp4_packed_bytes(0, 64) == 0 and nv.nvfp4_scale_bytes(0, 64) == 0
    ws = nv.nvfp4_linear_workspace_bytes(100, 1000, 512)
    assert ws >= nv.nvfp4_packed_bytes(100, 1000) + nv.nvfp4_scale_bytes(100, 1000)
    assert nv.nvfp4_linear_workspace_bytes(0, 1000, 512) == 0
    # the quantized activation and its scales, each 256-byte aligned (split-K
    # partial sums stay in the CTAs' shared memory, at every m)
    base = lambda m, k: (nv.nvfp4_packed_bytes(m, k) + 255) // 256 * 256 + (nv.nvfp4_scale_bytes(m, k) + 255) // 256 * 256
    assert ws == base(100, 1000)
    assert nv.nvfp4_linear_workspace_bytes(129, 1000, 512) == base(129, 1000)
    assert nv.nvfp4_linear_workspace_bytes(1, 14336, 4096) == base(1, 14336)


def quant(lib, x=A, m=16, k=256, ldx=256, gs=B, t=None, bs=0, out=C, sf=D):
    return lib.nvfp4_quant_act(x, m, k, ldx, gs, t, bs, out, sf, None)


def test_quant_validation(lib):
    assert quant(lib, m=0) == OK                             # empty call: no device needed
    assert quant(lib, x=None) == INVALID
    assert quant(lib, gs=None) == INVALID
    assert quant(lib, k=0) == INVALID
    assert quant(lib, ldx=100) == INVALID                    # ldx < k
    assert quant(lib, m=-1) == INVALID
    assert quant(lib, x=A + 8) == ALIGN
    assert quant(lib, k=250, ldx=250) == ALIGN               # rows not 16-byte aligned
    assert quant(lib, out=C + 4) == ALIGN
    assert quant(lib, t=A + B, bs=24) == INVALID             # bad block size
    assert quant(lib, t=None, bs=16) == INVALID              # bs without matrix
    assert quant(lib, t=A + B, bs=128, k=192, ldx=192) == INVALID    # bs does not divide k
    assert quant(lib, out=A + 64) == ALIAS                   # packed output inside x
    assert quant(lib, sf=A) == ALIAS
    assert quant(lib, sf=C + 1024) == ALIAS                  # scale output overlaps packed output
    assert "overlaps" in nv.nvfp4_last_error_string()


def test_quant_export_y_validation(lib):
    T = A + (1 << 30)
    Y = A + (1 << 31)
    f = lambda m=16, t=T, bs=16, y=Y: lib.nvfp4_quant_act_export_y(A, m, 256, 256, B, t, bs, C, D, y, None)
    assert f(m=0) == OK
    assert f(t=None, bs=0) == INVALID                        # only with a transform
    assert f(y=None) == INVALID
    assert f(y=Y + 8) == ALIGN
    assert f(y=A + 512) == ALIAS                             # y inside x
    assert f(y=C) == ALIAS                                   # y over the packed output
    assert f(bs=24) == INVALID


def test_act_global_scale_validation(lib):
    G, AL, WG = C, C + 64, D
    f = lambda x=A, m=16, k=256, ldx=256, t=None, bs=0, wg=None, gs=G, al=None: \
        lib.nvfp4_act_global_scale(x, m, k, ldx, t, bs, wg, gs, al, None)
    assert f(gs=None) == INVALID
    assert f(wg=WG) == INVALID                               # w_gs without alpha_out
    assert f(al=AL) == INVALID                               # alpha_out without w_gs
    assert f(gs=G + 2) == ALIGN
    assert f(x=None) == INVALID
    assert f(ldx=100) == INVALID
    assert f(x=A + 8) == ALIGN
    assert f(t=A + B, bs=24) == INVALID
    assert f(gs=A + 64) == ALIAS                             # scale output inside x
    assert f(wg=WG, al=WG) == ALIAS                          # alpha over w_gs
    assert f(wg=WG, al=G) == ALIAS                           # alpha over gs


def test_mxfp4_validation_and_sizes(lib):
    assert nv.nvfp4_mxfp4_scale_bytes(1, 4096) == 128 * 128          # 128 blocks -> 128 columns
    assert nv.nvfp4_mxfp4_scale_bytes(129, 4104) == 256 * 132        # Kp 4128 -> 129 blocks -> 132
    assert nv.nvfp4_mxfp4_scale_bytes(0, 4096) == 0
    f = lambda x=A, m=16, k=256, ldx=256, out=C, sf=D: lib.nvfp4_mxfp4_quant_act(x, m, k, ldx, out, sf, None)
    assert f(m=0) == OK
    assert f(x=None) == INVALID
    assert f(sf=None) == INVALID
    assert f(ldx=100) == INVALID
    assert f(x=A + 8) == ALIGN
    assert f(out=A + 64) == ALIAS
    assert f(sf=C + 1024) == ALIAS                         # scales over the packed output (2 KB)


def test_prepare_weight_validation(lib):
    assert lib.nvfp4_prepare_weight(A, 0, 64, 64, B, C, D, None) == OK
    assert lib.nvfp4_prepare_weight(None, 128, 64, 64, B, C, D, None) == INVALID
    assert lib.nvfp4_prepare_weight(A, 128, 64, 64, B, A + 256, D, None) == ALIAS


def gemm(lib, a=A, a_sf=B, m=16, w=C, w_sf=D, n_w=128, n_out=128, k=256, alpha=B + 4096, bias=None,
         out=(1 << 38), ldo=128):
    return lib.nvfp4_gemm(a, a_sf, m, w, w_sf, n_w, n_out, k, alpha, bias, out, ldo, None)


def test_gemm_validation(lib):
    assert gemm(lib, m=0) == OK
    assert gemm(lib, n_out=129) == INVALID                   # n_out > n_w
    assert gemm(lib, n_out=0) == INVALID
    assert gemm(lib, ldo=100) == INVALID                     # ldo < n_out
    assert gemm(lib, alpha=None) == INVALID
    assert gemm(lib, a=None) == INVALID
    assert gemm(lib, out=(1 << 38) + 2) == ALIGN
    assert gemm(lib, n_out=100, ldo=100) == ALIGN            # rows of out not 16-byte aligned
    assert gemm(lib, bias=(1 << 38) - 8) == ALIGN
    assert gemm(lib, out=C) == ALIAS                         # output over the weight
    assert gemm(lib, out=B + 4096 - 16) == ALIAS             # output over alpha


def test_linear_validation(lib):
    args = dict(x=A, m=16, k=256, ldx=256, gs=B, t=None, bs=0, w=C, w_sf=D, n_w=128, n_out=128,
                alpha=B + 64, bias=None, out=1 << 38, ldo=128, ws=1 << 39, ws_bytes=1 << 20)

    def call(**kw):
        a = dict(args, **kw)
        return lib.nvfp4_linear(a["x"], a["m"], a["k"], a["ldx"], a["gs"], a["t"], a["bs"], a["w"], a["w_sf"],
                                a["n_w"], a["n_out"], a["alpha"], a["bias"], a["out"], a["ldo"], a["ws"],
                                a["ws_bytes"], None)

    assert call(m=0) == OK
    assert call(ws=None) == WORKSPACE
    assert call(ws_bytes=100) == WORKSPACE
    assert call(ws=(1 << 39) + 8) == ALIGN
    assert call(ws=A) == ALIAS                               # workspace over x
    assert call(out=(1 << 39) + 512) == ALIAS                # output over workspace
    assert call(n_out=256) == INVALID


def test_is_supported_reports_a_reason_without_raising(lib):
    ok, why = nv.nvfp4_is_supported(0)
    if not ok:
        assert why
    ok, why = nv.nvfp4_is_supported(10 ** 6)
    assert not ok and why


def test_product_path_fails_loudly_without_library(tmp_path, monkeypatch):
    monkeypatch.setattr(nv, "_LIB_PATH", str(tmp_path / "missing.so"))
    monkeypatch.setattr(nv, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        nv.load_library()
