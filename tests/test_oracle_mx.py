"""Pins for the MXFP8 oracle (oracle/mx.py): 1x32 blocks with power-of-two
(UE8M0) scales, the smallest that keeps every element of a block unsaturated.

Independent references: the hand-worked 1x128 tile (its first 32 elements
form one block whose scale is the tile's), torch's own FP8 conversion of the
power-of-two-scaled values, the round-to-nearest error bound, the reduction to
the C oracle's 1x128 quantizer and block-scaled GEMM when every block scale is
the same power of two, exact rational brute force and a numpy
dequantise-then-multiply for the GEMM, and the pages' statement that block
scaling loses less than per-tensor scaling (checked on the wide-range
gradient distribution of the delayed-scaling workload)."""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
import synth
from oracle import mx

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
TORCH_FP8 = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def f32_to_bf16_bits(a):
    return torch.from_numpy(np.asarray(a, np.float32)).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_hand_tile():
    """The hand-worked tile: block 0 holds 896, -1, 0.30078125, 0.000999451
    and zeros, so amax / 448 = 2 is already a power of two: X = 2 (e8 = 128)
    and the codes are the tile's 0x7E, 0xB0, 0x22, 0x00; the three all-zero
    blocks get X = 1 (e8 = 127) and zero codes."""
    g = json.load(open(os.path.join(GOLDEN, "hand_1x128_tile.json")))
    x = np.zeros((1, 128), np.uint16)
    for i, b in g["tile_bf16_first_values"].items():
        x[0, int(i)] = int(b, 16)
    q, e8, st = mx.quant_mx(x, oracle.E4M3)
    assert st == oracle.OK
    assert list(e8[0]) == [128, 127, 127, 127]
    want = np.zeros(128, np.uint8)
    for i, c in g["expected_codes"].items():
        want[int(i)] = int(c, 16)
    assert np.array_equal(q[0], want)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_codes_equal_torch_conversion(fmt):
    xb = synth.bf16_normal((64, 512), 91, 1.0, 1e-3, 50.0)
    q, e8, _ = mx.quant_mx(xb, fmt)
    x = synth.bf16_bits_to_f32(xb).astype(np.float64).reshape(64, 16, 32)
    scaled = (x * np.ldexp(1.0, 127 - e8.astype(np.int64))[..., None]).astype(np.float32).reshape(64, 512)
    want = torch.from_numpy(scaled).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(q, want)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_smallest_unsaturated_power_of_two(fmt):
    """Every element is within half an FP8 spacing of x / X (so nothing
    saturated), and each nonzero block uses the top binade [fmax/2, fmax]
    (so X / 2 would have saturated its largest element)."""
    xb = synth.delayed_step_inputs(3, m=64, hidden=512, n_out=512)[1]       # wide-range gradients
    q, e8, _ = mx.quant_mx(xb, fmt)
    fm = oracle.fmax(fmt)
    dec = oracle.fp8_decode_table(fmt)[q]
    X = np.ldexp(1.0, np.repeat(e8.astype(np.int64) - 127, 32, axis=1))
    v = np.abs(synth.bf16_bits_to_f32(xb).astype(np.float64)) / X
    mant, sub = (3, -6) if fmt == oracle.E4M3 else (2, -14)
    binade = np.maximum(np.floor(np.log2(np.maximum(v, 1e-300))), sub).astype(np.int64)
    spacing = np.ldexp(1.0, binade - mant)
    assert np.all(np.abs(v - np.abs(dec)) <= spacing / 2)
    top = np.abs(dec).reshape(64, 16, 32).max(axis=2)
    nonzero = v.reshape(64, 16, 32).max(axis=2) > 0
    assert np.all(top[nonzero] >= fm / 2) and np.all(top <= fm)


def test_power_of_two_rescaling_shifts_only_the_scale():
    xb = synth.bf16_normal((32, 256), 92, 1.0, 1e-3, 20.0)
    q, e8, _ = mx.quant_mx(xb)
    for j in (-5, 3):
        x2 = f32_to_bf16_bits(synth.bf16_bits_to_f32(xb) * np.float32(2.0 ** j))
        q2, e82, _ = mx.quant_mx(x2)
        assert np.array_equal(q2, q) and np.array_equal(e82.astype(int), e8.astype(int) + j)


def test_reduces_to_the_1x128_quantizer_when_block_scales_agree():
    """Each 128-element tile whose four 32-blocks all have amax = 448 * 2^j:
    the 1x128 scale amax / 448 = 2^j is the MX scale of every block, so the
    codes are the C oracle's 1x128 codes."""
    rng = np.random.default_rng(93)
    R, C = 16, 512
    x = rng.normal(0, 1, (R, C)).astype(np.float32)
    j = rng.integers(-20, 8, (R, C // 128))
    for r in range(R):
        for t in range(C // 128):
            peak = np.float32(448.0 * 2.0 ** j[r, t])
            seg = x[r, t * 128:(t + 1) * 128]
            seg *= peak / np.abs(seg).max() * np.float32(0.9)
            for b in range(4):
                seg[b * 32 + rng.integers(0, 32)] = peak * (1 if rng.random() < 0.5 else -1)
    xb = f32_to_bf16_bits(x)
    q, e8, _ = mx.quant_mx(xb)
    q1, s1, _ = oracle.quant_1x128(xb)
    assert np.array_equal(q, q1)
    assert np.array_equal(np.ldexp(1.0, e8.astype(np.int64) - 127), np.repeat(s1.T.astype(np.float64), 4, axis=1))


def test_less_loss_than_per_tensor_on_wide_range_gradients():
    """The pages: per-block scale factors lose less than one per-tensor scale.
    On the delayed-scaling workload's gradients (signed lognormal, sigma 2.5)
    per-tensor scaling flushes a quarter of the nonzeros to zero; the MX
    blocks keep almost all of them and the mean relative error drops."""
    xb = synth.delayed_step_inputs(0, m=256, hidden=1024, n_out=1024)[1]
    x = synth.bf16_bits_to_f32(xb).astype(np.float64)
    nz = x != 0
    q, e8, _ = mx.quant_mx(xb)
    dm = mx.dequant_mx(q, e8)
    qp, sp, _ = oracle.quant_pertensor_current(xb)
    dp = oracle.fp8_decode_table(oracle.E4M3)[qp] * float(sp)
    under = lambda d: float(np.mean(d[nz] == 0))
    mrel = lambda d: float(np.mean(np.abs(d[nz] - x[nz]) / np.abs(x[nz])))
    assert under(dm) < 0.1 * under(dp) and under(dp) > 0.1
    assert mrel(dm) < 0.5 * mrel(dp)


def test_nonfinite_block_is_reported():
    xb = synth.bf16_normal((4, 64), 94)
    xb[2, 40] = 0x7F80
    assert mx.quant_mx(xb)[2] == oracle.NONFINITE


def test_gemm_exact_rational_bruteforce_tiny():
    rng = np.random.default_rng(95)
    M, N, K = 3, 2, 96
    qa, qb = rng.integers(0, 256, (M, K)).astype(np.uint8), rng.integers(0, 256, (N, K)).astype(np.uint8)
    qa[(qa & 0x7F) == 0x7F] = 0x38
    qb[(qb & 0x7F) == 0x7F] = 0x38
    # E4M3 values are multiples of 2^-9 below 2^9, so with block scales 2^-1..2^1
    # every term is a multiple of 2^-20 below 2^27: the FP64 sums are exact
    ea, eb = rng.integers(126, 129, (M, K // 32)).astype(np.uint8), rng.integers(126, 129, (N, K // 32)).astype(np.uint8)
    got = mx.mx_gemm_full(qa, ea, oracle.E4M3, qb, eb, oracle.E4M3)
    dec = torch.from_numpy(np.arange(256, dtype=np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    for m in range(M):
        for n in range(N):
            acc = Fraction(0)
            for k in range(K):
                b = k // 32
                acc += (Fraction(dec[qa[m, k]]) * Fraction(dec[qb[n, k]])
                        * Fraction(2) ** (int(ea[m, b]) - 127) * Fraction(2) ** (int(eb[n, b]) - 127))
            assert got[m, n] == float(acc)


def test_gemm_equals_dequantize_then_multiply_and_catches_a_block_mixup():
    xa = synth.bf16_normal((64, 256), 96, 1.0, 1e-3, 30.0)
    xw = synth.bf16_normal((48, 256), 97, 0.02)
    w = synth.bf16_bits_to_f32(xw)
    w[:, 32:64] *= np.float32(8.0)          # block 1 of every row sits 3 binades above block 0
    xw = f32_to_bf16_bits(w)
    qa, ea, _ = mx.quant_mx(xa, oracle.E5M2)
    qb, eb, _ = mx.quant_mx(xw, oracle.E4M3)
    got = mx.mx_gemm_full(qa, ea, oracle.E5M2, qb, eb, oracle.E4M3)
    ref = mx.dequant_mx(qa, ea, oracle.E5M2) @ mx.dequant_mx(qb, eb, oracle.E4M3).T
    assert np.allclose(got, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    eb_bad = eb.copy()
    eb_bad[:, [0, 1]] = eb_bad[:, [1, 0]]
    assert not np.allclose(mx.mx_gemm_full(qa, ea, oracle.E5M2, qb, eb_bad, oracle.E4M3), ref, rtol=1e-6)


def test_gemm_reduces_to_the_block_scaled_gemm_when_scales_agree():
    """With every 32-block scale inside a 128-chunk equal, the MX GEMM is the
    C oracle's 1x128 x 1x128 block-scaled GEMM with scales 2^(e8 - 127)."""
    rng = np.random.default_rng(98)
    M, N, K = 32, 24, 384
    qa = rng.integers(0, 0x7E, (M, K)).astype(np.uint8) | (rng.integers(0, 2, (M, K)).astype(np.uint8) << 7)
    qb = rng.integers(0, 0x7E, (N, K)).astype(np.uint8)
    ca, cb = rng.integers(115, 135, (M, K // 128)), rng.integers(115, 135, (N, K // 128))
    ea, eb = np.repeat(ca, 4, axis=1).astype(np.uint8), np.repeat(cb, 4, axis=1).astype(np.uint8)
    got = mx.mx_gemm_full(qa, ea, oracle.E4M3, qb, eb, oracle.E4M3)
    sa = np.ldexp(1.0, ca - 127).T.astype(np.float32).copy()     # S[K/128][M]
    sb = np.ldexp(1.0, cb - 127).T.astype(np.float32).copy()     # S[K/128][N]
    ref = oracle.gemm_full(qa, oracle.E4M3, sa, oracle.GRAN_1x128, qb, oracle.E4M3, sb, oracle.GRAN_1x128)
    assert np.allclose(got, ref, rtol=1e-13, atol=1e-13 * np.abs(ref).max())


def test_tile_scales_structure_and_inverse():
    """The GEMM-ready scale layout (mx_tile_scales): every 512-byte tile holds
    the codes of exactly one rectangle of 128 rows x 4 blocks, the tiles of one
    group of four blocks next to each other in row order; inside a tile the
    16-byte row j holds the four-block words of rows j, j + 32, j + 64, j + 96
    in that order (what a 32-row copy to all four lane quarters of the tensor
    memory needs); mx_untile_scales inverts it."""
    R, KB = 256, 12
    rr, kk = np.meshgrid(np.arange(R), np.arange(KB), indexing="ij")
    tr = mx.mx_tile_scales(rr.astype(np.uint8)).astype(int).reshape(KB // 4, R // 128, 32, 4, 4)
    tk = mx.mx_tile_scales(kk.astype(np.uint8)).astype(int).reshape(KB // 4, R // 128, 32, 4, 4)
    j = np.arange(32)[:, None, None]
    q = np.arange(4)[None, :, None]
    b = np.arange(4)[None, None, :]
    for kc in range(KB // 4):
        for rb in range(R // 128):
            assert set(tr[kc, rb].ravel()) == set(range(128 * rb, 128 * rb + 128))
            assert set(tk[kc, rb].ravel()) == set(range(4 * kc, 4 * kc + 4))
            assert np.array_equal(tr[kc, rb], np.broadcast_to(128 * rb + 32 * q + j, (32, 4, 4)))
            assert np.array_equal(tk[kc, rb], np.broadcast_to(4 * kc + b, (32, 4, 4)))
    e = np.random.default_rng(3).integers(0, 255, (384, 8), dtype=np.uint8)
    t = mx.mx_tile_scales(e)
    assert t.size == e.size and np.array_equal(np.sort(t), np.sort(e.ravel()))
    assert np.array_equal(mx.mx_untile_scales(t, 384, 8), e)
    with pytest.raises(ValueError):
        mx.mx_tile_scales(np.zeros((100, 8), np.uint8))
