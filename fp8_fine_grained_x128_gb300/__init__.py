"""Python binding of libfp8fg.so, the fine-grained FP8 Linear for GB300.

Argument marshalling only: every function passes torch tensors' device
pointers, sizes and the current CUDA stream to the C ABI declared in
``include/fp8fg.h``; all arithmetic runs in the library's sm_103a kernels.
PyTorch provides device memory and streams.  There is no fallback: if the
library is missing or fails to load, every call raises.

BF16 tensors are ``torch.bfloat16`` (or int16/uint16 bit patterns), FP8
tensors are ``torch.uint8`` code arrays, scales are ``torch.float32``.
Layouts follow the header (1x128 scales are chunk-major ``S[C/128][R]``).
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

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libfp8fg.so")
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
    "fp8_blockscaled_gemm": (_INT, [_I64, _I64, _I64, _VP, _INT, _VP, _INT, _VP, _INT, _VP, _INT,
                                    _VP, _INT, _I64, _VP]),
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
            raise RuntimeError(f"{LIB_PATH} is missing: run `python -m fp8_fine_grained_x128_gb300.build` "
                               "(there is no CPU fallback)")
        L = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(code: int) -> str:
    return lib().fp8_status_string(int(code)).decode()


def _p(t):
    if t is None:
        return None
    if isinstance(t, int):
        return t
    return t.data_ptr()


def _stream(stream=None):
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _check(name: str, rc: int) -> None:
    if rc != OK:
        raise Fp8Error(name, rc)


def _rows_cols(t):
    assert t.dim() == 2, "expected a 2-D tensor"
    return t.shape[0], t.shape[1], t.stride(0)


# ------------------------------------------------------------------ utility

def device_status(stream=None) -> int:
    """Synchronize, read and clear the device status word (0 = OK)."""
    out = _INT(0)
    _check("fp8_device_status", lib().fp8_device_status(_stream(stream), ctypes.byref(out)))
    return out.value


def selftest_wait_timeout(timeout_ms: int, stream=None) -> None:
    _check("fp8_selftest_wait_timeout", lib().fp8_selftest_wait_timeout(timeout_ms, _stream(stream)))


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
    R, C, ld = _rows_cols(x)
    _check("fp8_quant_1x128", lib().fp8_quant_1x128(_p(x), R, C, ld, fmt, _p(q), _p(s), _p(qT), _p(sT),
                                                    _stream(stream)))


def quant_128x128(w, fmt, q, s, qT=None, sT=None, stream=None):
    R, C, ld = _rows_cols(w)
    _check("fp8_quant_128x128", lib().fp8_quant_128x128(_p(w), R, C, ld, fmt, _p(q), _p(s), _p(qT),
                                                        _p(sT), _stream(stream)))


def transpose_128x128(q, s, qT, sT, stream=None):
    R, C = q.shape
    _check("fp8_transpose_128x128", lib().fp8_transpose_128x128(_p(q), _p(s), R, C, _p(qT), _p(sT),
                                                                _stream(stream)))


def transpose_128x128_batched(q, s, qT, sT, stream=None):
    """q [B, R, C] codes with scales [B, R/128, C/128] -> qT [B, C, R], sT [B, C/128, R/128]."""
    B, R, C = q.shape
    _check("fp8_transpose_128x128_batched",
           lib().fp8_transpose_128x128_batched(_p(q), _p(s), B, R, C, _p(qT), _p(sT), _stream(stream)))


def quant_pertensor_delayed(x, recipe: DelayedRecipe, hist, step, scale, q, workspace, qT=None,
                            stats=None, stream=None):
    R, C, ld = _rows_cols(x)
    _check("fp8_quant_pertensor_delayed",
           lib().fp8_quant_pertensor_delayed(_p(x), R, C, ld, ctypes.byref(recipe), _p(hist), _p(step),
                                             _p(scale), _p(q), _p(qT), _p(stats), _p(workspace),
                                             _stream(stream)))


def quant_pertensor_delayed_noalloc(x, recipe: DelayedRecipe, hist, step, scale, q, qT=None, stats=None,
                                    stream=None):
    """The delayed-scaling step without a caller workspace, for callers that
    cannot allocate device memory (the library's own scratch block is used;
    calls that overlap on the GPU race on it)."""
    R, C, ld = _rows_cols(x)
    _check("fp8_quant_pertensor_delayed_noalloc",
           lib().fp8_quant_pertensor_delayed_noalloc(_p(x), R, C, ld, ctypes.byref(recipe), _p(hist), _p(step),
                                                     _p(scale), _p(q), _p(qT), _p(stats), _stream(stream)))


def quant_pertensor_current(x, fmt, scale, q, workspace, stream=None):
    """Per-tensor current scaling: scale (device float[1]) = amax / fmax of x, q = codes."""
    R, C, ld = _rows_cols(x)
    _check("fp8_quant_pertensor_current",
           lib().fp8_quant_pertensor_current(_p(x), R, C, ld, fmt, _p(scale), _p(q), _p(workspace),
                                             _stream(stream)))


def quant_stats(x, q, s, gran, fmt, stats, workspace=None, stream=None):
    R, C, ld = _rows_cols(x)
    _check("fp8_quant_stats", lib().fp8_quant_stats(_p(x), R, C, ld, _p(q), _p(s), gran, fmt, _p(stats),
                                                    _p(workspace), _stream(stream)))


# ------------------------------------------------------------------ GEMMs

def blockscaled_gemm(A, fmtA, sA, granA, B, fmtB, sB, granB, D, stream=None):
    M, K = A.shape
    N = B.shape[0]
    out = OUT_F32 if D.dtype == torch.float32 else OUT_BF16
    _check("fp8_blockscaled_gemm",
           lib().fp8_blockscaled_gemm(M, N, K, _p(A), fmtA, _p(sA), granA, _p(B), fmtB, _p(sB), granB,
                                      _p(D), out, D.stride(0), _stream(stream)))


def grouped_gemm(offsets, A, sA, B, sB, D, stream=None):
    G, N, K = B.shape
    Mcap = A.shape[0]
    out = OUT_F32 if D.dtype == torch.float32 else OUT_BF16
    _check("fp8_grouped_gemm",
           lib().fp8_grouped_gemm(G, _p(offsets), Mcap, N, K, _p(A), _p(sA), _p(B), _p(sB), _p(D), out,
                                  D.stride(0), _stream(stream)))


def grouped_gemm_wgrad(offsets, AT, fmtA, sAT, BT, fmtB, sBT, D, stream=None):
    """D [G*N, ldD]: expert g's AT[:, rows_g] . BT[:, rows_g]^T (transposed copies, 1x128 scales)."""
    G = offsets.numel() - 1
    N, Mcap = AT.shape
    K = BT.shape[0]
    out = OUT_F32 if D.dtype == torch.float32 else OUT_BF16
    _check("fp8_grouped_gemm_wgrad",
           lib().fp8_grouped_gemm_wgrad(G, _p(offsets), Mcap, N, K, _p(AT), fmtA, _p(sAT), _p(BT), fmtB, _p(sBT),
                                        _p(D), out, D.stride(0), _stream(stream)))


# ------------------------------------------------------------------ high-precision dw monitor

def wgrad_recompute_error(dY, X, D, ref_workspace, err, stream=None):
    """err (device float64[3] view of fp8_wgrad_err_t: see new_wgrad_err) <- statistics of the FP8
    wgrad D [N, K] against R = dY^T . X recomputed from the BF16 operands into ref_workspace."""
    M, N = dY.shape
    K = X.shape[1]
    _check("fp8_wgrad_recompute_error",
           lib().fp8_wgrad_recompute_error(M, N, K, _p(dY), _p(X), _p(D), D.stride(0), _p(ref_workspace), _p(err),
                                           _stream(stream)))


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
    _check("fp8_adamw_step_fp8_states",
           lib().fp8_adamw_step_fp8_states(_p(param), _p(grad), _p(m), _p(m_scales), _p(v), _p(v_scales),
                                           param.numel(), ctypes.byref(hparams), _stream(stream)))


# ------------------------------------------------------------------ MoE glue

def moe_route_pad(logits, topk, align, Mcap, topk_idx, topk_prob, counts, offsets, row_token,
                  row_prob, row_is_pad=None, stream=None):
    T, E = logits.shape
    _check("fp8_moe_route_pad",
           lib().fp8_moe_route_pad(_p(logits), T, E, topk, align, Mcap, _p(topk_idx), _p(topk_prob),
                                   _p(counts), _p(offsets), _p(row_token), _p(row_prob),
                                   _p(row_is_pad), _stream(stream)))


def moe_gather(q, s, row_token, offsets, E, Mcap, qg, sg, stream=None):
    T, K = q.shape
    _check("fp8_moe_gather", lib().fp8_moe_gather(_p(q), _p(s), T, K, _p(row_token), _p(offsets), E,
                                                  Mcap, _p(qg), _p(sg), _stream(stream)))


def swiglu_fwd(gu, h, stream=None):
    R, F2 = gu.shape
    _check("fp8_swiglu_fwd", lib().fp8_swiglu_fwd(_p(gu), R, F2 // 2, _p(h), _stream(stream)))


def swiglu_bwd(gu, dh, dgu, stream=None):
    R, F2 = gu.shape
    _check("fp8_swiglu_bwd", lib().fp8_swiglu_bwd(_p(gu), _p(dh), R, F2 // 2, _p(dgu), _stream(stream)))


def swiglu_quant_fwd(gu, fmt, q, s, qT, sT, stream=None):
    """H = SwiGLU(gu) quantized 1x128 (q [R, F], s [F/128, R]) and 128x1 (qT [F, R], sT [R/128, F])."""
    R, F2 = gu.shape
    _check("fp8_swiglu_quant_fwd", lib().fp8_swiglu_quant_fwd(_p(gu), R, F2 // 2, fmt, _p(q), _p(s), _p(qT),
                                                              _p(sT), _stream(stream)))


def swiglu_bwd_quant(gu, dh, fmt, q, s, qT, sT, stream=None):
    """dGU = SwiGLU'(gu) . dh quantized 1x128 (q [R, 2F], s [2F/128, R]) and 128x1 (qT [2F, R], sT [R/128, 2F])."""
    R, F2 = gu.shape
    _check("fp8_swiglu_bwd_quant", lib().fp8_swiglu_bwd_quant(_p(gu), _p(dh), R, F2 // 2, fmt, _p(q), _p(s),
                                                              _p(qT), _p(sT), _stream(stream)))
