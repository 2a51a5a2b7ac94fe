"""CPU oracle for the fine-grained FP8 Linear -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (the CUDA library and its
binding) never loads it, and it shares no code with that path: the arithmetic
lives in ``fp8fg_oracle.c`` (plain C, FP64 where the definition is real
valued), compiled with gcc, no fast-math, no FP contraction, and for MXFP8 in
``mx.py`` (plain numpy around the C encoder and decoders).

Each wrapper below takes and returns numpy arrays (BF16 as uint16 bit
patterns, FP8 as uint8 codes).  Citations and the readings taken where the
pages are silent are in the C file's header.

Every function is pinned by ``tests/test_oracle_*.py`` to something other than
itself (library routines, hand-worked examples from the pages, closed forms,
brute force); the monitors' definitions have no formula on the pages, so their
parity rests on the hand-worked examples and a brute-force recount.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

E4M3 = 0
E5M2 = 1
GRAN_1x128 = 0
GRAN_128x128 = 1
GRAN_TENSOR = 2
GRAN_128x1 = 3
ALGO_MAX = 0
ALGO_MOST_RECENT = 1

OK = 0
NONFINITE = 1
BADARG = 2

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8fg_oracle.c")
_LIB = os.path.join(_HERE, "_build", "liboracle_fp8fg.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (OpenMP, strict IEEE).  Returns the .so path."""
    os.makedirs(os.path.dirname(_LIB), exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".{os.getpid()}.tmp"
        cmd = ["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-Wall", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _P(t):
    return ctypes.POINTER(t)


def _load(path: str):
    """The oracle library at `path`, with every entry point's signature set."""
    L = ctypes.CDLL(path)
    i64, i32, f32, f64, u8, u16 = (ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                                   ctypes.c_double, ctypes.c_uint8, ctypes.c_uint16)
    vp = ctypes.c_void_p
    sig = {
        "orc_version": (ctypes.c_int, []),
        "orc_bf16_to_f32": (f32, [u16]),
        "orc_fmax": (f32, [ctypes.c_int]),
        "orc_fp8_decode": (f64, [u8, ctypes.c_int]),
        "orc_fp8_encode": (u8, [f32, ctypes.c_int]),
        "orc_fp8_encode_array": (None, [vp, i64, ctypes.c_int, vp]),
        "orc_fp8_encode_bits_range": (None, [ctypes.c_uint32, i64, ctypes.c_int, vp]),
        "orc_f64_to_bf16": (u16, [f64]),
        "orc_quant_1x128": (ctypes.c_int, [vp, i64, i64, i64, ctypes.c_int, vp, vp]),
        "orc_quant_128x1_transposed": (ctypes.c_int, [vp, i64, i64, i64, ctypes.c_int, vp, vp]),
        "orc_quant_128x128": (ctypes.c_int, [vp, i64, i64, i64, ctypes.c_int, vp, vp]),
        "orc_fp8_transpose": (None, [vp, i64, i64, vp]),
        "orc_f32_transpose": (None, [vp, i64, i64, vp]),
        "orc_quant_stats": (ctypes.c_int, [vp, i64, i64, i64, vp, vp, ctypes.c_int,
                                           ctypes.c_int, vp]),
        "orc_delayed_step": (ctypes.c_int, [vp, i64, i64, i64, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, vp, vp, vp, vp, vp]),
        "orc_gemm_points": (ctypes.c_int, [i64, i64, i64, vp, i64, ctypes.c_int, vp,
                                           ctypes.c_int, i64, vp, i64, ctypes.c_int, vp,
                                           ctypes.c_int, i64, i64, vp, vp, vp]),
        "orc_grouped_gemm_points": (ctypes.c_int, [ctypes.c_int, vp, i64, i64, vp, vp, i64,
                                                   vp, vp, i64, vp, vp, vp]),
        "orc_grouped_wgrad_points": (ctypes.c_int, [ctypes.c_int, vp, i64, i64, i64, vp, ctypes.c_int,
                                                    vp, vp, ctypes.c_int, vp, i64, vp, vp, vp, vp]),
        "orc_quant_pertensor_current": (ctypes.c_int, [vp, i64, i64, i64, ctypes.c_int, vp, vp]),
        "orc_wgrad_recompute_error": (ctypes.c_int, [i64, i64, i64, vp, vp, vp, i64, vp]),
        "orc_adam_fp8_step": (ctypes.c_int, [i64, vp, vp, vp, vp, vp, vp] + [ctypes.c_float] * 9),
        "orc_moe_route": (ctypes.c_int, [i64, ctypes.c_int, ctypes.c_int, ctypes.c_int, vp,
                                         vp, vp, vp, vp, vp, i64, vp, vp, vp, vp]),
        "orc_moe_gather": (None, [vp, vp, i64, i64, vp, i64, i64, vp, vp]),
        "orc_swiglu_fwd": (None, [vp, i64, i64, vp]),
        "orc_swiglu_bwd": (None, [vp, vp, i64, i64, vp]),
    }
    for name, (res, args) in sig.items():
        fn = getattr(L, name)
        fn.restype = res
        fn.argtypes = args
    return L


def lib():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _load(build())
    return _lib


def use_library(path: str) -> None:
    """Tests only: route every wrapper below through the oracle library built
    at `path` -- a modified copy of fp8fg_oracle.c with a planted mistake,
    which the pins in tests/ must catch."""
    global _lib
    with _lock:
        _lib = _load(path)


def _ptr(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"] or a.ndim == 0
    return a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------
# Formats
# ---------------------------------------------------------------------------

def fmax(fmt: int) -> float:
    return float(lib().orc_fmax(fmt))


def fp8_decode(codes, fmt: int) -> np.ndarray:
    codes = np.asarray(codes, dtype=np.uint8)
    f = lib().orc_fp8_decode
    return np.array([f(int(c), fmt) for c in codes.ravel()], dtype=np.float64).reshape(codes.shape)


def fp8_decode_table(fmt: int) -> np.ndarray:
    return fp8_decode(np.arange(256, dtype=np.uint8), fmt)


def fp8_encode(values, fmt: int) -> np.ndarray:
    v = _c(values, np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib().orc_fp8_encode_array(_ptr(v), v.size, fmt, _ptr(out))
    return out


def fp8_encode_bits_range(first: int, count: int, fmt: int) -> np.ndarray:
    out = np.empty(count, dtype=np.uint8)
    lib().orc_fp8_encode_bits_range(first, count, fmt, _ptr(out))
    return out


def bf16_to_f32(bits) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16)
    f = lib().orc_bf16_to_f32
    return np.array([f(int(x)) for x in b.ravel()], dtype=np.float32).reshape(b.shape)


def f64_to_bf16(values) -> np.ndarray:
    v = np.asarray(values, dtype=np.float64)
    f = lib().orc_f64_to_bf16
    return np.array([f(float(x)) for x in v.ravel()], dtype=np.uint16).reshape(v.shape)


# ---------------------------------------------------------------------------
# Quantizers
# ---------------------------------------------------------------------------

def quant_1x128(x_bits: np.ndarray, fmt: int = E4M3):
    """1x128 tiles along rows: returns (q [R,C] uint8, s [C/128, R] float32, status)."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty((C // 128, R), np.float32)
    st = lib().orc_quant_1x128(_ptr(x), R, C, C, fmt, _ptr(q), _ptr(s))
    return q, s, st


def quant_128x1_transposed(x_bits: np.ndarray, fmt: int = E4M3):
    """Per-128-row column groups: returns (qT [C,R] uint8, sT [R/128, C] float32, status)."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    qT = np.empty((C, R), np.uint8)
    sT = np.empty((R // 128, C), np.float32)
    st = lib().orc_quant_128x1_transposed(_ptr(x), R, C, C, fmt, _ptr(qT), _ptr(sT))
    return qT, sT, st


def quant_128x128(w_bits: np.ndarray, fmt: int = E4M3):
    """128x128 blocks: returns (q [R,C] uint8, s [R/128, C/128] float32, status)."""
    w = _c(w_bits, np.uint16)
    R, C = w.shape
    q = np.empty((R, C), np.uint8)
    s = np.empty((R // 128, C // 128), np.float32)
    st = lib().orc_quant_128x128(_ptr(w), R, C, C, fmt, _ptr(q), _ptr(s))
    return q, s, st


def fp8_transpose(q: np.ndarray) -> np.ndarray:
    q = _c(q, np.uint8)
    R, C = q.shape
    out = np.empty((C, R), np.uint8)
    lib().orc_fp8_transpose(_ptr(q), R, C, _ptr(out))
    return out


def scale_grid_transpose(s: np.ndarray) -> np.ndarray:
    s = _c(s, np.float32)
    R, C = s.shape
    out = np.empty((C, R), np.float32)
    lib().orc_f32_transpose(_ptr(s), R, C, _ptr(out))
    return out


def quant_stats(x_bits, q, s, gran: int, fmt: int = E4M3) -> np.ndarray:
    """Monitors: uint64 [nonzero, underflow, saturated, distinct_in, distinct_out]."""
    x = _c(x_bits, np.uint16)
    q = _c(q, np.uint8)
    s = _c(np.atleast_1d(s), np.float32)
    R, C = x.shape
    out = np.zeros(5, np.uint64)
    st = lib().orc_quant_stats(_ptr(x), R, C, C, _ptr(q), _ptr(s), gran, fmt, _ptr(out))
    if st != OK:
        raise ValueError(f"orc_quant_stats status {st}")
    return out


class DelayedState:
    """Caller-owned per-tensor delayed-scaling state (history, step, scale)."""

    def __init__(self, history_len: int = 16):
        self.hist = np.zeros(history_len, np.float32)
        self.step = np.zeros(1, np.int32)
        self.scale = np.ones(1, np.float32)

    def copy(self) -> "DelayedState":
        c = DelayedState(len(self.hist))
        c.hist[:] = self.hist
        c.step[:] = self.step
        c.scale[:] = self.scale
        return c


def delayed_step(x_bits, state: DelayedState, fmt: int, margin: int = 0, algo: int = ALGO_MAX,
                 want_stats: bool = True):
    """One delayed-scaling step: returns (q, scale_used, stats or None, status); updates state."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    used = float(state.scale[0])
    stats = np.zeros(5, np.uint64) if want_stats else None
    st = lib().orc_delayed_step(_ptr(x), R, C, C, fmt, len(state.hist), margin, algo,
                                _ptr(state.hist), _ptr(state.step), _ptr(state.scale), _ptr(q),
                                _ptr(stats) if want_stats else None)
    return q, used, stats, st


# ---------------------------------------------------------------------------
# GEMMs
# ---------------------------------------------------------------------------

def gemm_points(A, fmtA, sA, granA, B, fmtB, sB, granB, pm, pn, ldsA=None, ldsB=None):
    """Unrounded FP64 D[m, n] = (A . B^T)[m, n] with the operands' scales, at points (pm, pn)."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    M, K = A.shape
    N = B.shape[0]
    sA = _c(np.atleast_1d(sA), np.float32)
    sB = _c(np.atleast_1d(sB), np.float32)
    if ldsA is None:
        ldsA = M if granA == GRAN_1x128 else K // 128
    if ldsB is None:
        ldsB = N if granB == GRAN_1x128 else K // 128
    pm = _c(pm, np.int64)
    pn = _c(pn, np.int64)
    out = np.empty(pm.shape, np.float64)
    st = lib().orc_gemm_points(M, N, K, _ptr(A), K, fmtA, _ptr(sA), granA, ldsA,
                               _ptr(B), K, fmtB, _ptr(sB), granB, ldsB, pm.size, _ptr(pm), _ptr(pn),
                               _ptr(out))
    if st != OK:
        raise ValueError(f"orc_gemm_points status {st}")
    return out


def gemm_full(A, fmtA, sA, granA, B, fmtB, sB, granB, ldsA=None, ldsB=None):
    M, N = A.shape[0], B.shape[0]
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    return gemm_points(A, fmtA, sA, granA, B, fmtB, sB, granB, mm.ravel(), nn.ravel(),
                       ldsA, ldsB).reshape(M, N)


def grouped_gemm_points(offsets, A, sA, ldsA, B, sB, pm, pn):
    """Grouped expert GEMM at points; B [G,N,K], sB [G,N/128,K/128], A scales S[K/128][ldsA]."""
    off = _c(offsets, np.int32)
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    G, N, K = B.shape
    sA = _c(sA, np.float32)
    sB = _c(sB, np.float32)
    pm = _c(pm, np.int64)
    pn = _c(pn, np.int64)
    out = np.empty(pm.shape, np.float64)
    st = lib().orc_grouped_gemm_points(G, _ptr(off), N, K, _ptr(A), _ptr(sA), ldsA, _ptr(B),
                                       _ptr(sB), pm.size, _ptr(pm), _ptr(pn), _ptr(out))
    if st != OK:
        raise ValueError(f"orc_grouped_gemm_points status {st}")
    return out


def grouped_wgrad_points(offsets, AT, fmtA, sA, BT, fmtB, sB, pg, pn, pk):
    """MoE grouped wgrad at points (g, n, k): D_g = AT[:, rows of g] . BT[:, rows of g]^T
    with 1x128 scales along the rows, S[ldt/128][N] and S[ldt/128][K]; 0 for an empty group."""
    off = _c(offsets, np.int32)
    AT = _c(AT, np.uint8)
    BT = _c(BT, np.uint8)
    N, ldt = AT.shape
    K = BT.shape[0]
    sA = _c(sA, np.float32)
    sB = _c(sB, np.float32)
    pg, pn, pk = (_c(np.ravel(v), np.int64) for v in (pg, pn, pk))
    out = np.empty(pg.size, np.float64)
    st = lib().orc_grouped_wgrad_points(len(off) - 1, _ptr(off), N, K, ldt, _ptr(AT), fmtA, _ptr(sA), _ptr(BT),
                                        fmtB, _ptr(sB), pg.size, _ptr(pg), _ptr(pn), _ptr(pk), _ptr(out))
    if st != OK:
        raise ValueError(f"orc_grouped_wgrad_points status {st}")
    return out


def grouped_wgrad_full(offsets, AT, fmtA, sA, BT, fmtB, sB):
    """All of D [G][N][K] of grouped_wgrad_points."""
    G, N, K = len(offsets) - 1, AT.shape[0], BT.shape[0]
    gg, nn, kk = np.meshgrid(np.arange(G), np.arange(N), np.arange(K), indexing="ij")
    return grouped_wgrad_points(offsets, AT, fmtA, sA, BT, fmtB, sB, gg, nn, kk).reshape(G, N, K)


# ---------------------------------------------------------------------------
# MoE routing and glue
# ---------------------------------------------------------------------------

def moe_route(logits, topk: int = 8, align: int = 128, cap: int | None = None):
    z = _c(logits, np.float32)
    T, E = z.shape
    if cap is None:
        cap = T * topk + E * (align - 1)
    topk_idx = np.empty((T, topk), np.int32)
    topk_prob = np.empty((T, topk), np.float64)
    counts = np.empty(E, np.int32)
    padded = np.empty(E, np.int32)
    offsets = np.empty(E + 1, np.int32)
    row_token = np.full(cap, -1, np.int32)
    row_prob = np.zeros(cap, np.float64)
    row_is_pad = np.zeros(cap, np.uint8)
    total = np.zeros(1, np.int64)
    st = lib().orc_moe_route(T, E, topk, align, _ptr(z), _ptr(topk_idx), _ptr(topk_prob),
                             _ptr(counts), _ptr(padded), _ptr(offsets), cap, _ptr(row_token),
                             _ptr(row_prob), _ptr(row_is_pad), _ptr(total))
    if st != OK:
        raise ValueError(f"orc_moe_route status {st}")
    return dict(topk_idx=topk_idx, topk_prob=topk_prob, counts=counts, padded=padded,
                offsets=offsets, row_token=row_token, row_prob=row_prob, row_is_pad=row_is_pad,
                total=int(total[0]), cap=cap)


def moe_gather(q, s, row_token, total: int, cap: int):
    q = _c(q, np.uint8)
    s = _c(s, np.float32)
    T, K = q.shape
    rt = _c(row_token, np.int32)
    qg = np.zeros((cap, K), np.uint8)
    sg = np.zeros((K // 128, cap), np.float32)
    lib().orc_moe_gather(_ptr(q), _ptr(s), T, K, _ptr(rt), total, cap, _ptr(qg), _ptr(sg))
    return qg, sg


def swiglu_fwd(gu_bits):
    gu = _c(gu_bits, np.uint16)
    R, F2 = gu.shape
    h = np.empty((R, F2 // 2), np.uint16)
    lib().orc_swiglu_fwd(_ptr(gu), R, F2 // 2, _ptr(h))
    return h


def swiglu_bwd(gu_bits, dh_bits):
    gu = _c(gu_bits, np.uint16)
    dh = _c(dh_bits, np.uint16)
    R, F2 = gu.shape
    dgu = np.empty((R, F2), np.uint16)
    lib().orc_swiglu_bwd(_ptr(gu), _ptr(dh), R, F2 // 2, _ptr(dgu))
    return dgu


# ---------------------------------------------------------------------------
# FP8 optimizer states
# ---------------------------------------------------------------------------

def adam_hyper(lr, beta1, beta2, eps, wd, step):
    """The binary32 constants of one AdamW step (bias corrections from the step number)."""
    f = np.float32
    return dict(lr=f(lr), b1=f(beta1), b2=f(beta2), omb1=f(1.0 - beta1), omb2=f(1.0 - beta2), eps=f(eps), wd=f(wd),
                bc1=f(1.0 - beta1 ** step), bc2=f(1.0 - beta2 ** step))


def adam_fp8_step(p, g_bits, qm, sm, qv, sv, h):
    """One AdamW step with FP8 moments (in place on copies): returns (p, qm, sm, qv, sv)."""
    p = np.array(p, np.float32, copy=True)
    qm, qv = np.array(qm, np.uint8, copy=True), np.array(qv, np.uint8, copy=True)
    sm, sv = np.array(sm, np.float32, copy=True), np.array(sv, np.float32, copy=True)
    g = _c(g_bits, np.uint16)
    st = lib().orc_adam_fp8_step(p.size, _ptr(p), _ptr(g), _ptr(qm), _ptr(sm), _ptr(qv), _ptr(sv), h["lr"], h["b1"],
                                 h["b2"], h["omb1"], h["omb2"], h["eps"], h["wd"], h["bc1"], h["bc2"])
    if st != OK:
        raise ValueError(f"orc_adam_fp8_step status {st}")
    return p, qm, sm, qv, sv


def quant_pertensor_current(x_bits, fmt=E4M3):
    """Per-tensor current scaling (the whole tensor one group): returns (q, scale, status)."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    s = np.zeros(1, np.float32)
    st = lib().orc_quant_pertensor_current(_ptr(x), R, C, C, fmt, _ptr(s), _ptr(q))
    return q, s[0], st


def wgrad_recompute_error(dY_bits, X_bits, D):
    """High-precision dw recompute monitor: {sum (D-R)^2, sum R^2, max|D-R|, max|R|} with
    R = dY^T . X of the BF16 operands (exact products, FP64 sums)."""
    dY, X = _c(dY_bits, np.uint16), _c(X_bits, np.uint16)
    D = _c(D, np.float32)
    M, N = dY.shape
    K = X.shape[1]
    out = np.zeros(4, np.float64)
    lib().orc_wgrad_recompute_error(M, N, K, _ptr(dY), _ptr(X), _ptr(D), D.shape[1], _ptr(out))
    return out
