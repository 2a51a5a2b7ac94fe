"""Pins for the oracle's block-scaled / per-tensor / grouped GEMM.

Independent references: exact rational arithmetic (fractions) on tiny shapes,
an integer matmul when the FP8 values are small integers and all scales are 1,
and numpy's FP64 matmul of the dequantized operands (the dequantise-then-
multiply brute force), with FP8 codes decoded by torch, not by the oracle.
"""
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth

TORCH_FP8 = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def tdec(codes, fmt):
    t = torch.from_numpy(np.ascontiguousarray(codes, np.uint8))
    return t.view(TORCH_FP8[fmt]).to(torch.float64).numpy()


def rand_codes(shape, seed, fmt):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    bad = np.isnan(tdec(c, fmt)) | np.isinf(tdec(c, fmt))
    c[bad] = 0x38
    return c


def rand_scales(shape, seed):
    rng = np.random.default_rng(seed)
    return (np.exp(rng.uniform(-6, 2, size=shape))).astype(np.float32)


def dequant(codes, fmt, s, gran, rows_are_M):
    """Dequantized operand [R, K] (float64) for the scale layouts the GEMM reads."""
    v = tdec(codes, fmt)
    R, K = v.shape
    if gran == oracle.GRAN_TENSOR:
        return v * np.float64(np.atleast_1d(s)[0])
    if gran == oracle.GRAN_1x128:       # S[K/128][R]
        full = np.repeat(s.astype(np.float64).T, 128, axis=1)
    else:                                # S[R/128][K/128]
        full = np.repeat(np.repeat(s.astype(np.float64), 128, 0), 128, 1)
    return v * full


def test_exact_rational_bruteforce_tiny():
    fmtA, fmtB = oracle.E4M3, oracle.E4M3
    M, N, K = 3, 130, 256
    A = rand_codes((M, K), 1, fmtA)
    B = rand_codes((N, K), 2, fmtB)
    sA = rand_scales((K // 128, M), 3)                 # 1x128
    sB = rand_scales(((N + 127) // 128, K // 128), 4)  # 128x128 (N=130: 2 row blocks)
    B = np.concatenate([B, np.zeros((256 - N, K), np.uint8)])  # pad to whole blocks
    Nb = 256
    pm, pn = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    got = oracle.gemm_points(A, fmtA, sA, oracle.GRAN_1x128, B, fmtB, sB, oracle.GRAN_128x128,
                             pm.ravel(), pn.ravel()).reshape(M, N)
    da, db = tdec(A, fmtA), tdec(B, fmtB)
    for m in range(M):
        for n in range(N):
            exact = Fraction(0)
            for kb in range(K // 128):
                p = sum(Fraction(float(da[m, k])) * Fraction(float(db[n, k]))
                        for k in range(kb * 128, kb * 128 + 128))
                exact += Fraction(float(sA[kb, m])) * Fraction(float(sB[n // 128, kb])) * p
            assert abs(Fraction(float(got[m, n])) - exact) <= abs(exact) * Fraction(1, 2 ** 50)
    assert Nb == 256


def test_integer_special_case():
    rng = np.random.default_rng(7)
    M, N, K = 128, 128, 384
    ia = rng.integers(-8, 9, size=(M, K))
    ib = rng.integers(-8, 9, size=(N, K))
    enc = lambda v: torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    A, B = enc(ia), enc(ib)
    ones_a = np.ones((K // 128, M), np.float32)
    ones_b = np.ones((N // 128, K // 128), np.float32)
    got = oracle.gemm_full(A, oracle.E4M3, ones_a, oracle.GRAN_1x128, B, oracle.E4M3, ones_b,
                           oracle.GRAN_128x128)
    assert np.array_equal(got, (ia @ ib.T).astype(np.float64))


CASES = [
    # (fmtA, granA, fmtB, granB)   fprop / dgrad / wgrad / per-tensor HYBRID
    (oracle.E4M3, oracle.GRAN_1x128, oracle.E4M3, oracle.GRAN_128x128),
    (oracle.E4M3, oracle.GRAN_1x128, oracle.E4M3, oracle.GRAN_1x128),
    (oracle.E4M3, oracle.GRAN_128x128, oracle.E4M3, oracle.GRAN_1x128),
    (oracle.E4M3, oracle.GRAN_TENSOR, oracle.E4M3, oracle.GRAN_TENSOR),
    (oracle.E5M2, oracle.GRAN_TENSOR, oracle.E4M3, oracle.GRAN_TENSOR),
]


@pytest.mark.parametrize("fmtA,granA,fmtB,granB", CASES)
def test_matches_dequantize_then_multiply(fmtA, granA, fmtB, granB):
    M, N, K = 256, 384, 512
    A = rand_codes((M, K), 11, fmtA)
    B = rand_codes((N, K), 12, fmtB)
    shape = lambda g, R: (K // 128, R) if g == oracle.GRAN_1x128 else \
        ((R // 128, K // 128) if g == oracle.GRAN_128x128 else (1,))
    sA = rand_scales(shape(granA, M), 13)
    sB = rand_scales(shape(granB, N), 14)
    got = oracle.gemm_full(A, fmtA, sA, granA, B, fmtB, sB, granB)
    a, b = dequant(A, fmtA, sA, granA, True), dequant(B, fmtB, sB, granB, False)
    ref = a @ b.T
    bound = 1e-12 * (np.abs(a) @ np.abs(b).T) + 1e-300
    assert np.all(np.abs(got - ref) <= bound)


def test_transposed_operand_mixups_are_detected():
    # wrong scale layout (transpose) gives a visibly different result
    M, N, K = 128, 256, 256
    A = rand_codes((M, K), 21, oracle.E4M3)
    B = rand_codes((N, K), 22, oracle.E4M3)
    sA = rand_scales((K // 128, M), 23)
    sB = rand_scales((N // 128, K // 128), 24)
    good = oracle.gemm_full(A, oracle.E4M3, sA, oracle.GRAN_1x128, B, oracle.E4M3, sB,
                            oracle.GRAN_128x128)
    bad = oracle.gemm_full(A, oracle.E4M3, sA, oracle.GRAN_1x128, B, oracle.E4M3,
                           np.ascontiguousarray(sB.T), oracle.GRAN_128x128)
    assert not np.allclose(good, bad)


def test_grouped_equals_per_group_gemm():
    G, N, K = 4, 256, 256
    offs = np.array([0, 128, 128, 384, 512], np.int32)   # group 1 empty
    cap = 640
    A = rand_codes((cap, K), 31, oracle.E4M3)
    sA = rand_scales((K // 128, cap), 32)
    B = rand_codes((G, N, K), 33, oracle.E4M3)
    sB = rand_scales((G, N // 128, K // 128), 34)
    pm, pn = np.meshgrid(np.arange(cap), np.arange(N), indexing="ij")
    got = oracle.grouped_gemm_points(offs, A, sA, cap, B, sB, pm.ravel(), pn.ravel()).reshape(cap, N)
    for g in range(G):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            continue
        a = dequant(A[lo:hi], oracle.E4M3, np.ascontiguousarray(sA[:, lo:hi]), oracle.GRAN_1x128, True)
        b = dequant(B[g], oracle.E4M3, sB[g], oracle.GRAN_128x128, False)
        ref = a @ b.T
        assert np.all(np.abs(got[lo:hi] - ref) <= 1e-12 * (np.abs(a) @ np.abs(b).T) + 1e-300)
    assert np.all(np.isnan(got[offs[-1]:]))


def test_grouped_wgrad_matches_dequantize_then_multiply():
    """MoE wgrad per expert: D_g = dequant(AT[:, rows_g]) . dequant(BT[:, rows_g])^T with the
    1x128 scales of the transposed copies (one per 128 rows and per column of the copy);
    an expert without rows gets exactly zero."""
    offs = np.array([0, 256, 256, 640, 768], np.int32)    # expert 1 has no rows
    ldt, N, K = 896, 256, 384                              # capacity past the last expert
    fa, fb = oracle.E5M2, oracle.E4M3                      # gradient x activation
    AT = rand_codes((N, ldt), 41, fa)
    BT = rand_codes((K, ldt), 42, fb)
    sA = rand_scales((ldt // 128, N), 43)
    sB = rand_scales((ldt // 128, K), 44)
    got = oracle.grouped_wgrad_full(offs, AT, fa, sA, BT, fb, sB)
    deqA = tdec(AT, fa) * np.repeat(sA.astype(np.float64).T, 128, axis=1)   # [N, ldt]
    deqB = tdec(BT, fb) * np.repeat(sB.astype(np.float64).T, 128, axis=1)   # [K, ldt]
    for g in range(len(offs) - 1):
        lo, hi = offs[g], offs[g + 1]
        if hi == lo:
            assert np.all(got[g] == 0.0)
            continue
        ref = deqA[:, lo:hi] @ deqB[:, lo:hi].T
        bound = 1e-12 * (np.abs(deqA[:, lo:hi]) @ np.abs(deqB[:, lo:hi]).T) + 1e-300
        assert np.all(np.abs(got[g] - ref) <= bound)
    # reading the scales with the row index instead of the chunk index is caught
    wrong = oracle.grouped_wgrad_full(offs, AT, fa, np.ascontiguousarray(sA[::-1]), BT, fb, sB)
    assert not np.allclose(wrong[3], got[3])


def test_wgrad_recompute_error_closed_forms():
    """With small-integer BF16 operands R = dY^T X is an exact integer matrix: D = R gives
    zero error; one entry off by delta gives delta^2 and delta; D = 0 gives sum (D-R)^2 =
    sum R^2 and max |D-R| = max |R|; D = 2R gives the same."""
    rng = np.random.default_rng(7)
    M, N, K = 64, 24, 40
    dyi = rng.integers(-8, 9, size=(M, N))
    xi = rng.integers(-8, 9, size=(M, K))
    to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)   # exact for small ints
    dy, x = to_bf16(dyi), to_bf16(xi)
    R = (dyi.T @ xi).astype(np.float64)                      # integer matmul
    out = oracle.wgrad_recompute_error(dy, x, R.astype(np.float32))
    assert out[0] == 0.0 and out[2] == 0.0
    assert out[1] == float((R * R).sum()) and out[3] == float(np.abs(R).max())
    D = R.astype(np.float32).copy()
    D[3, 5] += 0.5
    out = oracle.wgrad_recompute_error(dy, x, D)
    assert out[0] == 0.25 and out[2] == 0.5
    for D in (np.zeros_like(R, np.float32), (2 * R).astype(np.float32)):
        out = oracle.wgrad_recompute_error(dy, x, D)
        assert out[0] == out[1] and out[2] == out[3]
