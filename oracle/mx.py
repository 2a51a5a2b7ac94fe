"""MXFP8 (micro-scaled FP8) oracle -- TEST INFRASTRUCTURE ONLY.

Source: [Infra] "FP8 training infrastructure" guide, sections "Hardware
requirements for FP8 training" (Blackwell adds MXFP8, micro-scaled FP8),
"Scaling strategies and stability" (per-block scaling: each block inside a
tensor gets its own scale factor, which follows local value distributions
more closely than one per-tensor scale) and "Blackwell MXFP8 and NVFP4:
looking ahead" (hardware-accelerated block scaling replaces per-tensor
scaling).

The pages name the format but give neither the block size nor the scale
encoding.  Readings:
  R13  A block is 32 consecutive elements along a row (the contraction
       dimension of the GEMM that consumes it), the block of the
       micro-scaling format the pages call MXFP8.
  R14  A block's scale X is a power of two, stored as an unsigned 8-bit
       exponent code e8 (X = 2^(e8 - 127), e8 in 0..254): the smallest power
       of two with amax / X <= fmax, i.e. the R2 scale amax / fmax rounded up
       to a power of two, so no element of the block saturates.  A block whose
       amax is 0 gets X = 1.  A block holding Inf/NaN is reported
       (NONFINITE) and its codes are unspecified.
  R15  The element codes are enc(x / X) with R1 (round to nearest even,
       saturating); x / X is exact because X is a power of two.
  R16  MXFP8 GEMM: D[m, n] = sum_b X_A[m, b] * X_B[n, b] * (sum over the 32-block b
       of qA * qB), in FP64, rounded once at the end.

Plain numpy around the C oracle's FP8 encoder / decoder; no blocking or
reordering beyond the definition.
"""
from __future__ import annotations

import numpy as np

from . import E4M3, NONFINITE, OK, bf16_to_f32, fmax, fp8_decode_table, fp8_encode

MX_BLOCK = 32
E8_BIAS = 127

_tables = {}


def _bf16_table() -> np.ndarray:
    # every BF16 pattern through the C oracle's decoder, once
    if "bf16" not in _tables:
        _tables["bf16"] = bf16_to_f32(np.arange(65536, dtype=np.uint16)).astype(np.float64)
    return _tables["bf16"]


def _fp8_table(fmt: int) -> np.ndarray:
    if fmt not in _tables:
        _tables[fmt] = fp8_decode_table(fmt)
    return _tables[fmt]


def _dec(q, fmt: int) -> np.ndarray:
    return _fp8_table(fmt)[np.asarray(q, np.uint8)]


def mx_scale_exponents(amax: np.ndarray, fmt: int) -> np.ndarray:
    """R14: for each finite amax >= 0, the smallest integer e with
    fmax * 2^e >= amax (0 for amax == 0), clamped to [-127, 127]."""
    fm = float(fmax(fmt))
    a = np.asarray(amax, np.float64)
    pos = a > 0
    with np.errstate(divide="ignore"):
        e = np.ceil(np.log2(np.where(pos, a, fm) / fm)).astype(np.int64)
    # log2 is only approximately correctly rounded: settle e by exact comparisons
    e = e + (np.ldexp(fm, e) < a)
    e = e - ((np.ldexp(fm, e - 1) >= a) & pos)
    e = np.where(pos, e, 0)
    return np.clip(e, -E8_BIAS, E8_BIAS)


def quant_mx(x_bits: np.ndarray, fmt: int = E4M3):
    """MXFP8 quantization of a BF16 [R, C] tensor (C % 32 == 0) in 1x32 blocks
    along rows.  Returns (q [R, C] uint8 codes, e8 [R, C/32] uint8 scale codes
    with X = 2^(e8 - 127), status)."""
    x = _bf16_table()[np.asarray(x_bits, np.uint16)]
    R, C = x.shape
    if C % MX_BLOCK:
        raise ValueError("columns must be a multiple of 32")
    xb = x.reshape(R, C // MX_BLOCK, MX_BLOCK)
    amax = np.abs(xb).max(axis=2) if C else np.zeros((R, 0))
    if not np.all(np.isfinite(amax)):
        return np.zeros((R, C), np.uint8), np.full((R, C // MX_BLOCK), E8_BIAS, np.uint8), NONFINITE
    e = mx_scale_exponents(amax, fmt)
    quot = xb / np.ldexp(1.0, e)[..., None]           # exact: division by a power of two
    # binary32 holds the quotient exactly down to 2^-126; anything smaller is
    # far below half the smallest FP8 subnormal and encodes to a zero either way
    q = fp8_encode(quot.astype(np.float32).reshape(R, C), fmt)
    return q, (e + E8_BIAS).astype(np.uint8), OK


def dequant_mx(q: np.ndarray, e8: np.ndarray, fmt: int = E4M3) -> np.ndarray:
    """x_hat = dec(q) * 2^(e8 - 127) in FP64."""
    R, C = q.shape
    d = _dec(q, fmt).reshape(R, C // MX_BLOCK, MX_BLOCK)
    return (d * np.ldexp(1.0, e8.astype(np.int64) - E8_BIAS)[..., None]).reshape(R, C)


def mx_tile_scales(e8: np.ndarray) -> np.ndarray:
    """The library's GEMM-ready arrangement of MXFP8 scale codes (a layout of
    its own; the pages fix none): e8 [R, KB] with R % 128 == 0 and KB % 4 ==
    0 becomes R * KB bytes in which the codes of rows 128 rb .. 128 rb + 127
    and 32-blocks 4 kc .. 4 kc + 3 form the 512-byte tile number
    kc * (R / 128) + rb, and the code of row r, block b sits at byte
    16 (r % 32) + 4 ((r % 128) // 32) + b % 4 inside its tile.  A pure
    permutation of the codes."""
    e8 = np.asarray(e8, np.uint8)
    R, KB = e8.shape
    if R % 128 or KB % 4:
        raise ValueError("rows must be a multiple of 128 and blocks a multiple of 4")
    t = e8.reshape(R // 128, 4, 32, KB // 4, 4)          # [rb][(r % 128) // 32][r % 32][kc][b % 4]
    return np.ascontiguousarray(t.transpose(3, 0, 2, 1, 4)).reshape(-1)


def mx_untile_scales(tiled: np.ndarray, R: int, KB: int) -> np.ndarray:
    """Inverse of mx_tile_scales."""
    t = np.asarray(tiled, np.uint8).reshape(KB // 4, R // 128, 32, 4, 4)
    return np.ascontiguousarray(t.transpose(1, 3, 2, 0, 4)).reshape(R, KB)


def mx_gemm_points(qA, eA, fmtA, qB, eB, fmtB, pm, pn, chunk: int = 2048) -> np.ndarray:
    """R16 at the output points (pm, pn): A [M, K] and B [N, K] MXFP8 (scale
    codes [M, K/32] and [N, K/32]); unrounded FP64 values."""
    dA, dB = _dec(qA, fmtA), _dec(qB, fmtB)
    eA, eB = np.asarray(eA, np.int64), np.asarray(eB, np.int64)
    K = dA.shape[1]
    nb = K // MX_BLOCK
    pm, pn = np.asarray(pm, np.int64), np.asarray(pn, np.int64)
    out = np.empty(pm.shape, np.float64)
    for i in range(0, pm.size, chunk):
        m, n = pm[i:i + chunk], pn[i:i + chunk]
        part = (dA[m] * dB[n]).reshape(m.size, nb, MX_BLOCK).sum(axis=2)
        out[i:i + chunk] = np.ldexp(part, eA[m] + eB[n] - 2 * E8_BIAS).sum(axis=1)
    return out


def mx_gemm_full(qA, eA, fmtA, qB, eB, fmtB) -> np.ndarray:
    M, N = qA.shape[0], qB.shape[0]
    mm, nn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    return mx_gemm_points(qA, eA, fmtA, qB, eB, fmtB, mm.ravel(), nn.ravel()).reshape(M, N)
