"""The C-ABI library builds, loads and exports every entry point that
include/fp8fg.h declares; host-side argument validation rejects bad calls
with the documented status before touching the GPU (runs without a GPU)."""
import ctypes
import os
import re

import pytest

import fp8_fine_grained_x128_gb300 as fg
from fp8_fine_grained_x128_gb300 import build as fgbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    fgbuild.build()
    return fg.lib()


def declared_symbols():
    names = []
    inc = os.path.join(ROOT, "include")
    for f in sorted(os.listdir(inc)):
        if not f.endswith(".h"):
            continue
        text = open(os.path.join(inc, f)).read()
        names += re.findall(r"FP8FG_API\s+[\w\s\*]+?\b(\w+)\s*\(", text)
    return names


def test_every_declared_symbol_is_exported(lib):
    names = declared_symbols()
    assert len(names) >= 15
    for n in names:
        assert hasattr(lib, n), f"{n} declared in include/ but not exported"


def test_debug_build_exports_the_same_abi_and_says_so(lib):
    """The index-checked variant (FP8FG_DEBUG) builds from the same sources,
    exports every declared entry point and reports itself as the debug build;
    the release library reports 0."""
    path = fgbuild.build(debug=True)
    dbg = ctypes.CDLL(path)
    for n in declared_symbols():
        assert hasattr(dbg, n), f"{n} missing from the debug build"
    assert dbg.fp8_debug_build() == 1
    assert lib.fp8_debug_build() == 0
    assert fg.status_string(fg.ERR_BOUNDS) == "FP8_ERR_BOUNDS"


def test_selftest_bounds_validates_extents_on_the_host(lib):
    S = ctypes.c_void_p(0)
    f = lib.fp8_selftest_bounds
    assert f(None, -1, 4, S) == fg.ERR_INVALID_ARG
    assert f(None, 5, 4, S) == fg.ERR_INVALID_ARG
    assert f(None, 0, 0, S) == fg.OK              # nothing to write
    assert f(None, 0, 4, S) == fg.ERR_INVALID_ARG


def test_binding_covers_the_abi():
    assert set(declared_symbols()) <= set(fg._SIGS), set(declared_symbols()) - set(fg._SIGS)


def test_version_and_strings(lib):
    assert lib.fp8_abi_version() == 1
    assert fg.status_string(fg.ERR_SHAPE) == "FP8_ERR_SHAPE"
    assert fg.status_string(fg.ERR_TIMEOUT) == "FP8_ERR_TIMEOUT"
    assert fg.status_string(99) == "FP8_ERR_UNKNOWN"
    assert fg.workspace_bytes() >= 8192


def test_pertensor_workspace_fits_the_noalloc_scratch(lib):
    """The delayed-scaling step's workspace (ticket, amax, 65536-key presence
    bitmap, 256-key bitmap) is 8240 bytes; the no-allocation entry point keeps
    it in a fixed 16 KiB device block, so it must fit there."""
    src = open(os.path.join(ROOT, "fp8_fine_grained_x128_gb300", "csrc", "noalloc.cu")).read()
    block = int(re.search(r"kNoAllocScratchBytes\s*=\s*(\d+)", src).group(1))
    assert block == 16384
    assert fg.workspace_bytes() == 4 + 4 + 8 + 2048 * 4 + 8 * 4 == 8240
    assert fg.workspace_bytes() <= block


def test_host_validation_without_launch(lib):
    P = ctypes.c_void_p
    good = P(4096)            # a 16-byte aligned (never dereferenced) address
    odd = P(4097)
    S = None
    # quantizer: cols not a multiple of 128, bad format, misaligned, negative rows
    assert lib.fp8_quant_1x128(good, 4, 100, 100, 0, good, good, None, None, S) == fg.ERR_SHAPE
    assert lib.fp8_quant_1x128(good, 4, 128, 128, 7, good, good, None, None, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_quant_1x128(odd, 4, 128, 128, 0, good, good, None, None, S) == fg.ERR_ALIGNMENT
    assert lib.fp8_quant_1x128(good, -1, 128, 128, 0, good, good, None, None, S) == fg.ERR_SHAPE
    assert lib.fp8_quant_1x128(good, 100, 128, 128, 0, good, good, good, good, S) == fg.ERR_SHAPE  # T needs rows%128
    assert lib.fp8_quant_1x128(good, 128, 128, 128, 0, good, good, good, None, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_quant_1x128(good, 0, 128, 128, 0, None, None, None, None, S) == fg.OK          # empty
    assert lib.fp8_quant_128x128(good, 100, 128, 128, 0, good, good, None, None, S) == fg.ERR_SHAPE
    assert lib.fp8_transpose_128x128(good, good, 128, 64, good, good, S) == fg.ERR_SHAPE
    # GEMM: shapes, mixed TENSOR granularity, bad output dtype, misaligned ldD
    g = lambda M, N, K, ga=0, gb=1, out=0, ld=None, A=good: lib.fp8_blockscaled_gemm(
        M, N, K, A, 0, good, ga, good, 0, good, gb, good, out, N if ld is None else ld, S)
    assert g(100, 128, 128) == fg.ERR_SHAPE
    assert g(128, 128, 100) == fg.ERR_SHAPE
    assert g(128, 128, 128, ga=2, gb=1) == fg.ERR_UNSUPPORTED
    assert g(128, 128, 128, out=3) == fg.ERR_INVALID_ARG
    assert g(128, 128, 128, ld=100) == fg.ERR_SHAPE
    assert g(128, 128, 128, ld=132) == fg.ERR_ALIGNMENT
    assert g(128, 128, 128, A=odd) == fg.ERR_ALIGNMENT
    assert g(0, 128, 128) == fg.OK
    # grouped GEMM and MoE glue
    assert lib.fp8_grouped_gemm(0, good, 128, 128, 128, good, good, good, good, good, 0, 128, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_grouped_gemm(2, good, 100, 128, 128, good, good, good, good, good, 0, 128, S) == fg.ERR_SHAPE
    w = lambda G=2, cap=256, N=128, K=128, fa=1, out=1, ld=128, D=good: lib.fp8_grouped_gemm_wgrad(
        G, good, cap, N, K, good, fa, good, good, 0, good, D, out, ld, S)
    assert w(G=0) == fg.ERR_INVALID_ARG
    assert w(fa=5) == fg.ERR_INVALID_ARG
    assert w(cap=200) == fg.ERR_SHAPE
    assert w(K=100) == fg.ERR_SHAPE
    assert w(ld=64) == fg.ERR_SHAPE
    assert w(out=0, ld=132) == fg.ERR_ALIGNMENT
    assert w(D=odd) == fg.ERR_ALIGNMENT
    assert w(N=0) == fg.OK
    assert lib.fp8_transpose_128x128_batched(good, good, 2, 128, 64, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_transpose_128x128_batched(good, good, -1, 128, 128, good, good, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_transpose_128x128_batched(good, good, 0, 128, 128, good, good, S) == fg.OK
    assert lib.fp8_quant_pertensor_current(good, 4, 12, 12, 0, good, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_quant_pertensor_current(good, 4, 16, 16, 9, good, good, good, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_quant_pertensor_current(good, 4, 16, 16, 0, good, good, None, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_quant_pertensor_current(odd, 4, 16, 16, 0, good, good, good, S) == fg.ERR_ALIGNMENT
    assert lib.fp8_wgrad_recompute_error(-1, 128, 128, good, good, good, 128, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_wgrad_recompute_error(128, 128, 128, good, good, good, 100, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_wgrad_recompute_error(128, 128, 128, good, good, good, 128, good, None, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_wgrad_recompute_error(128, 128, 128, odd, good, good, 128, good, good, S) == fg.ERR_ALIGNMENT
    hp = fg.adamw_hparams(1e-3, 0.9, 0.95, 1e-8, 0.1, 1)
    assert lib.fp8_adamw_step_fp8_states(good, good, good, good, good, good, 100, ctypes.byref(hp), S) == fg.ERR_SHAPE
    assert lib.fp8_adamw_step_fp8_states(good, good, good, good, good, good, 128, None, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_adamw_step_fp8_states(odd, good, good, good, good, good, 128, ctypes.byref(hp), S) == fg.ERR_ALIGNMENT
    assert lib.fp8_adamw_step_fp8_states(None, None, None, None, None, None, 0, ctypes.byref(hp), S) == fg.OK
    assert lib.fp8_moe_route_pad(good, 16, 300, 8, 128, 1024, good, good, good, good, good, good, None, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_moe_route_pad(good, 16, 8, 9, 128, 1024, good, good, good, good, good, good, None, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_swiglu_fwd(good, 4, 12, good, S) == fg.ERR_SHAPE
    assert lib.fp8_swiglu_quant_fwd(good, 128, 96, 0, good, good, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_swiglu_quant_fwd(good, 100, 128, 0, good, good, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_swiglu_quant_fwd(good, 128, 128, 7, good, good, good, good, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_swiglu_quant_fwd(good, 128, 128, 0, good, good, None, good, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_swiglu_quant_fwd(odd, 128, 128, 0, good, good, good, good, S) == fg.ERR_ALIGNMENT
    assert lib.fp8_swiglu_quant_fwd(None, 0, 128, 0, None, None, None, None, S) == fg.OK
    assert lib.fp8_swiglu_bwd_quant(good, None, 128, 128, 0, good, good, good, good, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_swiglu_bwd_quant(good, odd, 128, 128, 1, good, good, good, good, S) == fg.ERR_ALIGNMENT
    assert lib.fp8_swiglu_bwd_quant(good, good, 1 << 24, 1 << 16, 1, good, good, good, good, S) == fg.ERR_SHAPE
    # delayed scaling: recipe checks
    rec = fg.DelayedRecipe(0, 0, 0, 0)
    assert lib.fp8_quant_pertensor_delayed(good, 128, 128, 128, ctypes.byref(rec), good, good, good, good,
                                           None, None, good, S) == fg.ERR_INVALID_ARG
    rec = fg.DelayedRecipe(0, 16, 200, 0)
    assert lib.fp8_quant_pertensor_delayed(good, 128, 128, 128, ctypes.byref(rec), good, good, good, good,
                                           None, None, good, S) == fg.ERR_INVALID_ARG
    rec = fg.DelayedRecipe(1, 16, 0, 1)
    assert lib.fp8_quant_pertensor_delayed(good, 128, 100, 128, ctypes.byref(rec), good, good, good, good,
                                           None, None, good, S) == fg.ERR_SHAPE
    # MXFP8 quantizer
    assert lib.fp8_quant_mx(good, 4, 48, 48, 0, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_quant_mx(good, 4, 64, 32, 0, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_quant_mx(good, 4, 64, 64, 5, good, good, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_quant_mx(good, 4, 64, 64, 0, good, None, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_quant_mx(odd, 4, 64, 64, 0, good, good, S) == fg.ERR_ALIGNMENT
    assert lib.fp8_quant_mx(good, 4, 64, 68, 0, good, good, S) == fg.ERR_ALIGNMENT
    assert lib.fp8_quant_mx(good, 4, 64, 64, 0, P(4100), good, S) == fg.ERR_ALIGNMENT
    assert lib.fp8_quant_mx(None, 0, 64, 64, 1, None, None, S) == fg.OK
    # MXFP8 quantizer, tiled scale codes: whole 128 x 128 tiles only
    assert lib.fp8_quant_mx_tiled(good, 100, 128, 128, 0, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_quant_mx_tiled(good, 128, 64, 64, 0, good, good, S) == fg.ERR_SHAPE
    assert lib.fp8_quant_mx_tiled(good, 128, 128, 128, 5, good, good, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_quant_mx_tiled(good, 128, 128, 128, 0, good, None, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_quant_mx_tiled(odd, 128, 128, 128, 0, good, good, S) == fg.ERR_ALIGNMENT
    assert lib.fp8_quant_mx_tiled(None, 0, 128, 128, 1, None, None, S) == fg.OK
    # MXFP8 GEMMs: the row-major scale codes need 4-byte alignment, the tiles 16
    assert lib.fp8_mx_gemm(100, 128, 128, good, 0, good, good, 0, good, good, 0, 128, S) == fg.ERR_SHAPE
    assert lib.fp8_mx_gemm(128, 128, 128, good, 0, P(4098), good, 0, good, good, 0, 128, S) == fg.ERR_ALIGNMENT
    assert lib.fp8_mx_gemm_tiled(128, 128, 100, good, 0, good, good, 0, good, good, 0, 128, S) == fg.ERR_SHAPE
    assert lib.fp8_mx_gemm_tiled(128, 128, 128, good, 0, P(4100), good, 0, good, good, 0, 128, S) == \
        fg.ERR_ALIGNMENT
    assert lib.fp8_mx_gemm_tiled(128, 128, 128, good, 0, good, good, 0, P(4104), good, 0, 128, S) == \
        fg.ERR_ALIGNMENT
    assert lib.fp8_mx_gemm_tiled(128, 128, 128, good, 2, good, good, 0, good, good, 0, 128, S) == \
        fg.ERR_INVALID_ARG
    assert lib.fp8_mx_gemm_tiled(0, 128, 128, None, 0, None, None, 0, None, good, 0, 128, S) == fg.OK
    assert lib.fp8_selftest_wait_timeout(0, S) == fg.ERR_INVALID_ARG
    assert lib.fp8_device_status(S, None) == fg.ERR_INVALID_ARG


def test_header_is_plain_c(tmp_path):
    """include/fp8fg.h is a C header: it compiles as pedantic C99 with every
    warning an error, and a C caller links nothing but the declarations."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_header.c"
    src.write_text('#include "fp8fg.h"\n'
                   "int main(void)\n{\n"
                   "    fp8_adamw_hparams_t h = {0};\n    fp8_wgrad_err_t e = {0};\n    fp8_stats_t s = {0};\n"
                   "    (void)h; (void)e; (void)s;\n"
                   "    return fp8_abi_version() > 0 ? 0 : 1;\n}\n")
    p = subprocess.run([cc, "-std=c99", "-pedantic", "-Wall", "-Wextra", "-Werror",
                        "-I", os.path.join(ROOT, "include"), "-c", str(src), "-o", str(tmp_path / "use_header.o")],
                       capture_output=True, text=True)
    assert p.returncode == 0, p.stderr


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    """Without the CUDA library every entry point raises: there is no CPU
    fallback behind the binding."""
    monkeypatch.setattr(fg, "LIB_PATH", str(tmp_path / "absent.so"))
    monkeypatch.setattr(fg, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU fallback"):
        fg.lib()
    import torch
    x = torch.zeros((128, 128), dtype=torch.bfloat16)
    with pytest.raises(RuntimeError):
        fg.quant_1x128(x, fg.E4M3, torch.empty((128, 128), dtype=torch.uint8), torch.empty((1, 128)))


def test_binding_refuses_host_memory():
    """The binding checks what the C ABI cannot: a host tensor's address
    would reach a kernel as a device pointer, so it is refused (ValueError)
    before anything is launched; so is a non-tensor where a tensor's shape is
    needed (TypeError)."""
    import torch
    fg.lib()
    x = torch.zeros((128, 128), dtype=torch.bfloat16)
    q, s = torch.empty((128, 128), dtype=torch.uint8), torch.empty((1, 128))
    with pytest.raises(ValueError, match="CUDA tensor"):
        fg.quant_1x128(x, fg.E4M3, q, s)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fg.swiglu_fwd(torch.zeros((128, 256), dtype=torch.bfloat16), x)
    with pytest.raises(ValueError, match="CUDA tensor"):
        fg.blockscaled_gemm(q, fg.E4M3, s, fg.GRAN_1x128, q, fg.E4M3, s, fg.GRAN_1x128,
                            torch.empty((128, 128), dtype=torch.bfloat16))
    with pytest.raises(TypeError, match="torch.Tensor"):
        fg.grouped_gemm_wgrad([0, 128], q, fg.E4M3, s, q, fg.E4M3, s, x)
    with pytest.raises(TypeError, match="torch.Tensor"):
        fg.adamw_step_fp8_states(None, None, None, None, None, None, fg.adamw_hparams(1e-3, 0.9, 0.95, 1e-8, 0, 1))
