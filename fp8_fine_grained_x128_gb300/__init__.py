"""Python binding of libfp8fg.so, the fine-grained FP8 Linear for GB300.

Argument marshalling only: every function passes torch tensors' device
pointers, sizes and the current CUDA stream to the C ABI declared in
``include/fp8fg.h``; all arithmetic runs in the library's sm_103a kernels.
PyTorch provides device memory and streams.  There is no fallback: if the
library is missing or fails to load, every call raises.

BF16 tensors are ``torch.bfloat16`` (or int16/uint16 bit patterns), FP8
tensors are ``torch.uint8`` code arrays (int8 and torch's float8 types are
accepted too), scales are ``torch.float32``, index arrays ``torch.int32``.
Layouts follow the header (1x128 scales are chunk-major ``S[C/128][R]``).

Before a call the binding checks what the C ABI cannot see behind a pointer:
every tensor is on the current CUDA device and of the element type above;
a 2-D input passed with a leading dimension has unit column stride; every
other array is contiguous and at least as large as the header's layout for
the call's sizes.  A failed check raises ValueError / TypeError before anything
is launched.  A plain ``int`` is taken as a raw device pointer, unchecked.
"""
from __future__ import annotations

import ctypes
import os

import torch

E4M3 = 0
E5M2 = 1
GRAN_1x128 = 0
GRAN_128x128 = 1
GRAN_TENSOR = 2
GRAN_128x1 = 3
OUT_BF16 = 0
OUT_F32 = 1
AMAX_MAX = 0
AMAX_MOST_RECENT = 1

OK = 0
ERR_INVALID_ARG = 1
ERR_SHAPE = 2
ERR_ALIGNMENT = 3
ERR_UNSUPPORTED = 4
ERR_CUDA = 5
ERR_NONFINITE = 6
ERR_TIMEOUT = 7
ERR_BOUNDS = 8

_HERE = os.path.dirname(os.path.abspath(__file__))
# FP8FG_DEBUG=1 in the environment selects the index-checked debug build
# (every kernel store checked against its buffer's extent; FP8_ERR_BOUNDS in
# the status word on a miss), built by `python -m fp8_fine_grained_x128_gb300.build --debug`.
DEBUG = os.environ.get("FP8FG_DEBUG", "0") not in ("", "0")
LIB_PATH = os.path.join(_HERE, "libfp8fg_debug.so" if DEBUG else "libfp8fg.so")
_lib = None


class Fp8Error(RuntimeError):
    def __init__(self, name: str, code: int):
        super().__init__(f"{name} failed: {status_string(code) if _lib else code}")
        self.code = code


class Stats(ctypes.Structure):
    _fields_ = [("nonzero", ctypes.c_uint64), ("underflow", ctypes.c_uint64),
                ("saturated", ctypes.c_uint64), ("distinct_in", ctypes.c_uint64),
                ("distinct_out", ctypes.c_uint64)]


class DelayedRecipe(ctypes.Structure):
    _fields_ = [("fmt", ctypes.c_int32), ("history_len", ctypes.c_int32),
                ("margin", ctypes.c_int32), ("algo", ctypes.c_int32)]


class AdamWHparams(ctypes.Structure):
    _fields_ = [(n, ctypes.c_float) for n in ("lr", "beta1", "beta2", "one_minus_beta1", "one_minus_beta2", "eps",
                                              "weight_decay", "bias_correction1", "bias_correction2")]


_I64, _I32, _VP, _INT = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p, ctypes.c_int
_SIGS = {
    "fp8_abi_version": (_INT, []),
    "fp8_status_string": (ctypes.c_char_p, [_INT]),
    "fp8_device_status": (_INT, [_VP, ctypes.POINTER(_INT)]),
    "fp8_selftest_wait_timeout": (_INT, [_INT, _VP]),
    "fp8_debug_build": (_INT, []),
    "fp8_selftest_bounds": (_INT, [_VP, _I64, _I64, _VP]),
    "fp8_quant_1x128": (_INT, [_VP, _I64, _I64, _I64, _INT, _VP, _VP, _VP, _VP, _VP]),
    "fp8_quant_128x128": (_INT, [_VP, _I64, _I64, _I64, _INT, _VP, _VP, _VP, _VP, _VP]),
    "fp8_transpose_128x128": (_INT, [_VP, _VP, _I64, _I64, _VP, _VP, _VP]),
    "fp8_transpose_128x128_batched": (_INT, [_VP, _VP, _INT, _I64, _I64, _VP, _VP, _VP]),
    "fp8_pertensor_workspace_bytes": (ctypes.c_size_t, []),
    "fp8_quant_pertensor_delayed": (_INT, [_VP, _I64, _I64, _I64, ctypes.POINTER(DelayedRecipe),
                                           _VP, _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "fp8_quant_pertensor_delayed_noalloc": (_INT, [_VP, _I64, _I64, _I64, ctypes.POINTER(DelayedRecipe),
                                                   _VP, _VP, _VP, _VP, _VP, _VP, _VP]),
    "fp8_quant_pertensor_current": (_INT, [_VP, _I64, _I64, _I64, _INT, _VP, _VP, _VP, _VP]),
    "fp8_quant_stats": (_INT, [_VP, _I64, _I64, _I64, _VP, _VP, _INT, _INT, _VP, _VP, _VP]),
    "fp8_quant_mx": (_INT, [_VP, _I64, _I64, _I64, _INT, _VP, _VP, _VP]),
    "fp8_quant_mx_tiled": (_INT, [_VP, _I64, _I64, _I64, _INT, _VP, _VP, _VP]),
    "fp8_blockscaled_gemm": (_INT, [_I64, _I64, _I64, _VP, _INT, _VP, _INT, _VP, _INT, _VP, _INT,
                                    _VP, _INT, _I64, _VP]),
    "fp8_mx_gemm": (_INT, [_I64, _I64, _I64, _VP, _INT, _VP, _VP, _INT, _VP, _VP, _INT, _I64, _VP]),
    "fp8_mx_gemm_tiled": (_INT, [_I64, _I64, _I64, _VP, _INT, _VP, _VP, _INT, _VP, _VP, _INT, _I64, _VP]),
    "fp8_grouped_gemm": (_INT, [_INT, _VP, _I64, _I64, _I64, _VP, _VP, _VP, _VP, _VP, _INT, _I64,
                                _VP]),
    "fp8_grouped_gemm_wgrad": (_INT, [_INT, _VP, _I64, _I64, _I64, _VP, _INT, _VP, _VP, _INT, _VP, _VP, _INT,
                                      _I64, _VP]),
    "fp8_wgrad_recompute_error": (_INT, [_I64, _I64, _I64, _VP, _VP, _VP, _I64, _VP, _VP, _VP]),
    "fp8_adamw_step_fp8_states": (_INT, [_VP, _VP, _VP, _VP, _VP, _VP, _I64, ctypes.POINTER(AdamWHparams), _VP]),
    "fp8_moe_route_pad": (_INT, [_VP, _I64, _INT, _INT, _INT, _I64, _VP, _VP, _VP, _VP, _VP, _VP,
                                 _VP, _VP]),
    "fp8_moe_gather": (_INT, [_VP, _VP, _I64, _I64, _VP, _VP, _INT, _I64, _VP, _VP, _VP]),
    "fp8_swiglu_fwd": (_INT, [_VP, _I64, _I64, _VP, _VP]),
    "fp8_swiglu_bwd": (_INT, [_VP, _VP, _I64, _I64, _VP, _VP]),
    "fp8_swiglu_quant_fwd": (_INT, [_VP, _I64, _I64, _INT, _VP, _VP, _VP, _VP, _VP]),
    "fp8_swiglu_bwd_quant": (_INT, [_VP, _VP, _I64, _I64, _INT, _VP, _VP, _VP, _VP, _VP]),
}


def lib() -> ctypes.CDLL:
    """The loaded CUDA library (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            flag = " --debug" if DEBUG else ""
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m fp8_fine_grained_x128_gb300.build{flag}` "
                               "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        if bool(L.fp8_debug_build()) != DEBUG:
            raise RuntimeError(f"{LIB_PATH} is not the {'debug' if DEBUG else 'release'} build")
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().fp8_status_string(int(code)).decode()


_BF16 = (torch.bfloat16, torch.int16, torch.uint16)
_CODES = (torch.uint8, torch.int8, torch.float8_e4m3fn, torch.float8_e5m2)
_F32 = (torch.float32,)
_I32 = (torch.int32,)
_OUT = (torch.bfloat16, torch.float32)


def _on_device(t, name, dtypes):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor, got {type(t).__name__}")
    if t.device.type != "cuda":
        raise ValueError(f"{name}: expected a CUDA tensor, got one on {t.device}")
    cur = torch.cuda.current_device()
    if t.device.index != cur:
        raise ValueError(f"{name}: on {t.device}, but the current device is cuda:{cur}")
    if t.dtype not in dtypes:
        raise TypeError(f"{name}: dtype {t.dtype}, expected one of {tuple(str(d) for d in dtypes)}")


def _buf(t, name, dtypes, numel, optional=False):
    """Device pointer of an array the library reads or writes as `numel`
    contiguous elements."""
    if t is None:
        if optional:
            return None
        raise ValueError(f"{name} is required")
    if isinstance(t, int):
        return t
    _on_device(t, name, dtypes)
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    if t.numel() < numel:
        raise ValueError(f"{name}: holds {t.numel()} elements, the call needs {numel}")
    return t.data_ptr()


def _mat(t, name, dtypes):
    """(pointer, rows, cols, leading dimension) of a row-major 2-D view."""
    _on_device(t, name, dtypes)
    if t.dim() != 2:
        raise ValueError(f"{name}: expected a 2-D tensor, got shape {tuple(t.shape)}")
    R, C = t.shape
    if C > 1 and t.stride(1) != 1:
        raise ValueError(f"{name}: columns must be contiguous (stride {t.stride(1)})")
    ld = t.stride(0) if R > 1 else C
    return t.data_ptr(), R, C, ld


def _shape(t, name, dims):
    if isinstance(t, torch.Tensor) and t.dim() != dims:
        raise ValueError(f"{name}: expected a {dims}-D tensor, got shape {tuple(t.shape)}")
    return tuple(t.shape)


def _gran_scales(gran, rows, cols):
    """Element count of the scale array of a [rows][cols] operand (header layouts)."""
    if gran == GRAN_1x128:
        return (cols // 128) * rows
    if gran == GRAN_128x128:
        return (rows // 128) * (cols // 128)
    if gran == GRAN_128x1:
        return (rows // 128) * cols
    return 1


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(name: str, rc: int) -> None:
    if rc != OK:
        raise Fp8Error(name, rc)


# ------------------------------------------------------------------ utility

def device_status(stream=None) -> int:
    """Synchronize, read and clear the device status word (0 = OK)."""
    out = _INT(0)
    _check("fp8_device_status", lib().fp8_device_status(_stream(stream), ctypes.byref(out)))
    return out.value


def selftest_wait_timeout(timeout_ms: int, stream=None) -> None:
    _check("fp8_selftest_wait_timeout", lib().fp8_selftest_wait_timeout(timeout_ms, _stream(stream)))


def debug_build() -> bool:
    """True when the loaded library is the index-checked debug build."""
    return bool(lib().fp8_debug_build())


def selftest_bounds(buf: torch.Tensor, n_claimed: int, stream=None) -> None:
    """Writes 1.0 to every element of the FP32 device buffer `buf` through the
    checked store, against a claimed extent of `n_claimed` elements: the debug
    build stops at n_claimed and records ERR_BOUNDS, the release build writes
    all of `buf`."""
    if not isinstance(buf, torch.Tensor):
        raise TypeError("buf: expected a torch.Tensor (its size gives n_write)")
    n = buf.numel()
    _check("fp8_selftest_bounds", lib().fp8_selftest_bounds(_buf(buf, "buf", _F32, n), int(n_claimed), n,
                                                             _stream(stream)))


def workspace_bytes() -> int:
    return int(lib().fp8_pertensor_workspace_bytes())


def new_workspace(device="cuda") -> torch.Tensor:
    """A zeroed workspace for the per-tensor reductions (kept zeroed by the library)."""
    n = (workspace_bytes() + 15) // 16 * 16
    return torch.zeros(n, dtype=torch.uint8, device=device)


def new_stats(device="cuda") -> torch.Tensor:
    """A zeroed fp8_stats_t on the device (5 x uint64 as int64)."""
    return torch.zeros(5, dtype=torch.int64, device=device)


# ------------------------------------------------------------------ quantizers

def quant_1x128(x, fmt, q, s, qT=None, sT=None, stream=None):
    L = lib()
    px, R, C, ld = _mat(x, "x", _BF16)
    args = (_buf(q, "q", _CODES, R * C), _buf(s, "s", _F32, (C // 128) * R),
            _buf(qT, "qT", _CODES, C * R, True), _buf(sT, "sT", _F32, (R // 128) * C, True))
    _check("fp8_quant_1x128", L.fp8_quant_1x128(px, R, C, ld, fmt, *args, _stream(stream)))


def quant_128x128(w, fmt, q, s, qT=None, sT=None, stream=None):
    L = lib()
    pw, R, C, ld = _mat(w, "w", _BF16)
    nb = (R // 128) * (C // 128)
    args = (_buf(q, "q", _CODES, R * C), _buf(s, "s", _F32, nb),
            _buf(qT, "qT", _CODES, C * R, True), _buf(sT, "sT", _F32, nb, True))
    _check("fp8_quant_128x128", L.fp8_quant_128x128(pw, R, C, ld, fmt, *args, _stream(stream)))


def transpose_128x128(q, s, qT, sT, stream=None):
    L = lib()
    R, C = _shape(q, "q", 2)
    nb = (R // 128) * (C // 128)
    args = (_buf(q, "q", _CODES, R * C), _buf(s, "s", _F32, nb), R, C,
            _buf(qT, "qT", _CODES, C * R), _buf(sT, "sT", _F32, nb))
    _check("fp8_transpose_128x128", L.fp8_transpose_128x128(*args, _stream(stream)))


def transpose_128x128_batched(q, s, qT, sT, stream=None):
    """q [B, R, C] codes with scales [B, R/128, C/128] -> qT [B, C, R], sT [B, C/128, R/128]."""
    L = lib()
    B, R, C = _shape(q, "q", 3)
    nb = B * (R // 128) * (C // 128)
    args = (_buf(q, "q", _CODES, B * R * C), _buf(s, "s", _F32, nb), B, R, C,
            _buf(qT, "qT", _CODES, B * C * R), _buf(sT, "sT", _F32, nb))
    _check("fp8_transpose_128x128_batched", L.fp8_transpose_128x128_batched(*args, _stream(stream)))


def _delayed_state(recipe, hist, step, scale, R, C, q, qT, stats):
    return (_buf(hist, "amax_history", _F32, max(int(recipe.history_len), 1)), _buf(step, "step", _I32, 1),
            _buf(scale, "scale", _F32, 1), _buf(q, "q", _CODES, R * C), _buf(qT, "qT", _CODES, C * R, True),
            _buf(stats, "stats", (torch.int64,), 5, True))


def quant_pertensor_delayed(x, recipe: DelayedRecipe, hist, step, scale, q, workspace, qT=None,
                            stats=None, stream=None):
    L = lib()
    px, R, C, ld = _mat(x, "x", _BF16)
    st = _delayed_state(recipe, hist, step, scale, R, C, q, qT, stats)
    ws = _buf(workspace, "workspace", (torch.uint8,), workspace_bytes())
    _check("fp8_quant_pertensor_delayed",
           L.fp8_quant_pertensor_delayed(px, R, C, ld, ctypes.byref(recipe), *st, ws, _stream(stream)))


def quant_pertensor_delayed_noalloc(x, recipe: DelayedRecipe, hist, step, scale, q, qT=None, stats=None,
                                    stream=None):
    """The delayed-scaling step without a caller workspace, for callers that
    cannot allocate device memory (the library's own scratch block is used;
    calls that overlap on the GPU race on it)."""
    L = lib()
    px, R, C, ld = _mat(x, "x", _BF16)
    st = _delayed_state(recipe, hist, step, scale, R, C, q, qT, stats)
    _check("fp8_quant_pertensor_delayed_noalloc",
           L.fp8_quant_pertensor_delayed_noalloc(px, R, C, ld, ctypes.byref(recipe), *st, _stream(stream)))


def quant_pertensor_current(x, fmt, scale, q, workspace, stream=None):
    """Per-tensor current scaling: scale (device float[1]) = amax / fmax of x, q = codes."""
    L = lib()
    px, R, C, ld = _mat(x, "x", _BF16)
    args = (_buf(scale, "scale", _F32, 1), _buf(q, "q", _CODES, R * C),
            _buf(workspace, "workspace", (torch.uint8,), workspace_bytes()))
    _check("fp8_quant_pertensor_current", L.fp8_quant_pertensor_current(px, R, C, ld, fmt, *args, _stream(stream)))


def quant_stats(x, q, s, gran, fmt, stats, workspace=None, stream=None):
    L = lib()
    px, R, C, ld = _mat(x, "x", _BF16)
    args = (_buf(q, "q", _CODES, R * C), _buf(s, "s", _F32, _gran_scales(gran, R, C)), gran, fmt,
            _buf(stats, "stats", (torch.int64,), 5),
            _buf(workspace, "workspace", (torch.uint8,), workspace_bytes(), True))
    _check("fp8_quant_stats", L.fp8_quant_stats(px, R, C, ld, *args, _stream(stream)))


def quant_mx(x, fmt, q, e8, stream=None):
    """MXFP8: q [R, C] codes and e8 [R, C/32] uint8 scale codes, X = 2^(e8 - 127)."""
    L = lib()
    px, R, C, ld = _mat(x, "x", _BF16)
    args = (_buf(q, "q", _CODES, R * C), _buf(e8, "e8", (torch.uint8,), R * (C // 32)))
    _check("fp8_quant_mx", L.fp8_quant_mx(px, R, C, ld, fmt, *args, _stream(stream)))


def quant_mx_tiled(x, fmt, q, e8t, stream=None):
    """MXFP8 with the scale codes in the GEMM's 512-byte tile layout (R, C multiples of 128):
    e8t holds R * C / 32 uint8 codes, any shape."""
    L = lib()
    px, R, C, ld = _mat(x, "x", _BF16)
    args = (_buf(q, "q", _CODES, R * C), _buf(e8t, "e8t", (torch.uint8,), R * (C // 32)))
    _check("fp8_quant_mx_tiled", L.fp8_quant_mx_tiled(px, R, C, ld, fmt, *args, _stream(stream)))


# ------------------------------------------------------------------ GEMMs

def _out_mat(D, rows, cols):
    pd, R, C, ld = _mat(D, "D", _OUT)
    if R < rows or C < cols:
        raise ValueError(f"D: shape {(R, C)}, the call writes [{rows}][{cols}]")
    return pd, (OUT_F32 if D.dtype == torch.float32 else OUT_BF16), ld


def blockscaled_gemm(A, fmtA, sA, granA, B, fmtB, sB, granB, D, stream=None):
    L = lib()
    M, K = _shape(A, "A", 2)
    N, KB = _shape(B, "B", 2)
    if KB != K:
        raise ValueError(f"B: shape {(N, KB)}, expected [N][{K}]")
    pA, pB = _buf(A, "A", _CODES, M * K), _buf(B, "B", _CODES, N * K)
    psA = _buf(sA, "sA", _F32, _gran_scales(granA, M, K))
    psB = _buf(sB, "sB", _F32, _gran_scales(granB, N, K))
    pD, out, ldD = _out_mat(D, M, N)
    _check("fp8_blockscaled_gemm",
           L.fp8_blockscaled_gemm(M, N, K, pA, fmtA, psA, granA, pB, fmtB, psB, granB, pD, out, ldD,
                                  _stream(stream)))


def mx_gemm(A, fmtA, eA, B, fmtB, eB, D, stream=None):
    """MXFP8 GEMM: D = A . B^T with codes A [M, K], B [N, K] and scale exponents eA [M, K/32],
    eB [N, K/32] (uint8, X = 2^(e - 127), as quant_mx writes them)."""
    L = lib()
    M, K = _shape(A, "A", 2)
    N, KB = _shape(B, "B", 2)
    if KB != K:
        raise ValueError(f"B: shape {(N, KB)}, expected [N][{K}]")
    pA, pB = _buf(A, "A", _CODES, M * K), _buf(B, "B", _CODES, N * K)
    peA = _buf(eA, "eA", (torch.uint8,), M * (K // 32))
    peB = _buf(eB, "eB", (torch.uint8,), N * (K // 32))
    pD, out, ldD = _out_mat(D, M, N)
    _check("fp8_mx_gemm", L.fp8_mx_gemm(M, N, K, pA, fmtA, peA, pB, fmtB, peB, pD, out, ldD, _stream(stream)))


def mx_gemm_tiled(A, fmtA, eAt, B, fmtB, eBt, D, stream=None):
    """MXFP8 GEMM with the scale codes of A and B in the tiled layout quant_mx_tiled writes
    (M * K / 32 and N * K / 32 uint8 codes, 16-byte aligned)."""
    L = lib()
    M, K = _shape(A, "A", 2)
    N, KB = _shape(B, "B", 2)
    if KB != K:
        raise ValueError(f"B: shape {(N, KB)}, expected [N][{K}]")
    pA, pB = _buf(A, "A", _CODES, M * K), _buf(B, "B", _CODES, N * K)
    peA = _buf(eAt, "eAt", (torch.uint8,), M * (K // 32))
    peB = _buf(eBt, "eBt", (torch.uint8,), N * (K // 32))
    pD, out, ldD = _out_mat(D, M, N)
    _check("fp8_mx_gemm_tiled",
           L.fp8_mx_gemm_tiled(M, N, K, pA, fmtA, peA, pB, fmtB, peB, pD, out, ldD, _stream(stream)))


def grouped_gemm(offsets, A, sA, B, sB, D, stream=None):
    L = lib()
    G, N, K = _shape(B, "B", 3)
    Mcap, KA = _shape(A, "A", 2)
    if KA != K:
        raise ValueError(f"A: shape {(Mcap, KA)}, expected [M_capacity][{K}]")
    args = (_buf(offsets, "offsets", _I32, G + 1), Mcap, N, K, _buf(A, "A", _CODES, Mcap * K),
            _buf(sA, "sA", _F32, (K // 128) * Mcap), _buf(B, "B", _CODES, G * N * K),
            _buf(sB, "sB", _F32, G * (N // 128) * (K // 128)))
    pD, out, ldD = _out_mat(D, Mcap, N)
    _check("fp8_grouped_gemm", L.fp8_grouped_gemm(G, *args, pD, out, ldD, _stream(stream)))


def grouped_gemm_wgrad(offsets, AT, fmtA, sAT, BT, fmtB, sBT, D, stream=None):
    """D [G*N, ldD]: expert g's AT[:, rows_g] . BT[:, rows_g]^T (transposed copies, 1x128 scales)."""
    L = lib()
    if not isinstance(offsets, torch.Tensor):
        raise TypeError("offsets: expected a torch.Tensor (its length gives the number of experts)")
    G = offsets.numel() - 1
    N, Mcap = _shape(AT, "AT", 2)
    K, MB = _shape(BT, "BT", 2)
    if MB != Mcap:
        raise ValueError(f"BT: shape {(K, MB)}, expected [K][{Mcap}]")
    args = (_buf(offsets, "offsets", _I32, G + 1), Mcap, N, K, _buf(AT, "AT", _CODES, N * Mcap), fmtA,
            _buf(sAT, "sAT", _F32, (Mcap // 128) * N), _buf(BT, "BT", _CODES, K * Mcap), fmtB,
            _buf(sBT, "sBT", _F32, (Mcap // 128) * K))
    pD, out, ldD = _out_mat(D, max(G, 0) * N, K)
    _check("fp8_grouped_gemm_wgrad", L.fp8_grouped_gemm_wgrad(G, *args, pD, out, ldD, _stream(stream)))


# ------------------------------------------------------------------ high-precision dw monitor

def wgrad_recompute_error(dY, X, D, ref_workspace, err, stream=None):
    """err (device float64[3] view of fp8_wgrad_err_t: see new_wgrad_err) <- statistics of the FP8
    wgrad D [N, K] against R = dY^T . X recomputed from the BF16 operands into ref_workspace."""
    L = lib()
    M, N = _shape(dY, "dY", 2)
    MX, K = _shape(X, "X", 2)
    if MX != M:
        raise ValueError(f"X: shape {(MX, K)}, expected [{M}][K]")
    pdY, pX = _buf(dY, "dY", _BF16, M * N), _buf(X, "X", _BF16, M * K)
    pD, R, C, ldD = _mat(D, "D", _F32)
    if R < N or C < K:
        raise ValueError(f"D: shape {(R, C)}, expected at least [{N}][{K}]")
    args = (pdY, pX, pD, ldD, _buf(ref_workspace, "ref_workspace", _F32, N * K),
            _buf(err, "err", (torch.float64,), 3))
    _check("fp8_wgrad_recompute_error", L.fp8_wgrad_recompute_error(M, N, K, *args, _stream(stream)))


def new_wgrad_err(device="cuda") -> torch.Tensor:
    """Storage for fp8_wgrad_err_t (24 bytes)."""
    return torch.zeros(3, dtype=torch.float64, device=device)


def wgrad_err_values(err: torch.Tensor):
    """(sum_sq_diff, sum_sq_ref, max_abs_diff, max_abs_ref) from new_wgrad_err storage."""
    h = err.cpu()
    f = h[2:3].view(torch.float32)
    return float(h[0]), float(h[1]), float(f[0]), float(f[1])


# ------------------------------------------------------------------ FP8 optimizer states

def adamw_hparams(lr, beta1, beta2, eps, weight_decay, step) -> AdamWHparams:
    """The binary32 hyper-parameters of AdamW step ``step`` (>= 1)."""
    return AdamWHparams(lr, beta1, beta2, 1.0 - beta1, 1.0 - beta2, eps, weight_decay, 1.0 - beta1 ** step,
                        1.0 - beta2 ** step)


def adamw_step_fp8_states(param, grad, m, m_scales, v, v_scales, hparams: AdamWHparams, stream=None):
    """In place: FP32 ``param`` [n], BF16 ``grad`` [n], E4M3 ``m`` / E5M2 ``v`` codes [n] with
    scales [n/128]."""
    L = lib()
    if not isinstance(param, torch.Tensor):
        raise TypeError("param: expected a torch.Tensor (its size gives n)")
    n = param.numel()
    args = (_buf(param, "param", _F32, n), _buf(grad, "grad", _BF16, n), _buf(m, "m", _CODES, n),
            _buf(m_scales, "m_scales", _F32, n // 128), _buf(v, "v", _CODES, n),
            _buf(v_scales, "v_scales", _F32, n // 128))
    _check("fp8_adamw_step_fp8_states", L.fp8_adamw_step_fp8_states(*args, n, ctypes.byref(hparams),
                                                                    _stream(stream)))


# ------------------------------------------------------------------ MoE glue

def moe_route_pad(logits, topk, align, Mcap, topk_idx, topk_prob, counts, offsets, row_token,
                  row_prob, row_is_pad=None, stream=None):
    L = lib()
    T, E = _shape(logits, "logits", 2)
    args = (_buf(logits, "logits", _F32, T * E), T, E, topk, align, Mcap,
            _buf(topk_idx, "topk_idx", _I32, T * topk), _buf(topk_prob, "topk_prob", _F32, T * topk),
            _buf(counts, "counts", _I32, E), _buf(offsets, "offsets", _I32, E + 1),
            _buf(row_token, "row_token", _I32, Mcap), _buf(row_prob, "row_prob", _F32, Mcap),
            _buf(row_is_pad, "row_is_pad", (torch.uint8, torch.bool), Mcap, True))
    _check("fp8_moe_route_pad", L.fp8_moe_route_pad(*args, _stream(stream)))


def moe_gather(q, s, row_token, offsets, E, Mcap, qg, sg, stream=None):
    L = lib()
    T, K = _shape(q, "q", 2)
    args = (_buf(q, "q", _CODES, T * K), _buf(s, "s", _F32, (K // 128) * T), T, K,
            _buf(row_token, "row_token", _I32, Mcap), _buf(offsets, "offsets", _I32, E + 1), E, Mcap,
            _buf(qg, "qg", _CODES, Mcap * K), _buf(sg, "sg", _F32, (K // 128) * Mcap))
    _check("fp8_moe_gather", L.fp8_moe_gather(*args, _stream(stream)))


def _gu(gu):
    R, F2 = _shape(gu, "gu", 2)
    return _buf(gu, "gu", _BF16, R * F2), R, F2 // 2


def swiglu_fwd(gu, h, stream=None):
    L = lib()
    pg, R, F = _gu(gu)
    _check("fp8_swiglu_fwd", L.fp8_swiglu_fwd(pg, R, F, _buf(h, "h", _BF16, R * F), _stream(stream)))


def swiglu_bwd(gu, dh, dgu, stream=None):
    L = lib()
    pg, R, F = _gu(gu)
    args = (_buf(dh, "dh", _BF16, R * F), R, F, _buf(dgu, "dgu", _BF16, R * 2 * F))
    _check("fp8_swiglu_bwd", L.fp8_swiglu_bwd(pg, *args, _stream(stream)))


def _quant_outs(q, s, qT, sT, R, C):
    return (_buf(q, "q", _CODES, R * C), _buf(s, "s", _F32, (C // 128) * R), _buf(qT, "qT", _CODES, C * R),
            _buf(sT, "sT", _F32, (R // 128) * C))


def swiglu_quant_fwd(gu, fmt, q, s, qT, sT, stream=None):
    """H = SwiGLU(gu) quantized 1x128 (q [R, F], s [F/128, R]) and 128x1 (qT [F, R], sT [R/128, F])."""
    L = lib()
    pg, R, F = _gu(gu)
    _check("fp8_swiglu_quant_fwd", L.fp8_swiglu_quant_fwd(pg, R, F, fmt, *_quant_outs(q, s, qT, sT, R, F),
                                                          _stream(stream)))


def swiglu_bwd_quant(gu, dh, fmt, q, s, qT, sT, stream=None):
    """dGU = SwiGLU'(gu) . dh quantized 1x128 (q [R, 2F], s [2F/128, R]) and 128x1 (qT [2F, R], sT [R/128, 2F])."""
    L = lib()
    pg, R, F = _gu(gu)
    pdh = _buf(dh, "dh", _BF16, R * F)
    _check("fp8_swiglu_bwd_quant", L.fp8_swiglu_bwd_quant(pg, pdh, R, F, fmt, *_quant_outs(q, s, qT, sT, R, 2 * F),
                                                          _stream(stream)))
