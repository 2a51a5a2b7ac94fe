"""GPU parity of the high-precision dw recompute monitor: exact on small-integer
operands (zero error for the exact wgrad), and on the FP8 wgrad of random
operands the statistics match the oracle's FP64 ones within the FP32
accumulation of the BF16 reference."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import assert_status_ok, dev_bf16, guarded

pytestmark = pytest.mark.gpu


def monitor(dy_bits, x_bits, D):
    M, N = dy_bits.shape
    K = x_bits.shape[1]
    R = guarded((N, K), torch.float32)
    err = fg.new_wgrad_err()
    fg.wgrad_recompute_error(dev_bf16(dy_bits), dev_bf16(x_bits), D, R, err)
    assert_status_ok()
    return fg.wgrad_err_values(err), R


def test_exact_wgrad_has_zero_error():
    rng = np.random.default_rng(3)
    M, N, K = 256, 128, 384
    dyi, xi = rng.integers(-8, 9, size=(M, N)), rng.integers(-8, 9, size=(M, K))
    to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    R = (dyi.T @ xi).astype(np.float32)
    (sdd, srr, mdd, mrr), Rg = monitor(to_bf16(dyi), to_bf16(xi), torch.from_numpy(R).cuda())
    assert np.array_equal(Rg.cpu().numpy(), R)
    assert sdd == 0.0 and mdd == 0.0
    assert srr == float((R.astype(np.float64) ** 2).sum()) and mrr == float(np.abs(R).max())


@pytest.mark.parametrize("M,N,K", [(256, 128, 384), (1000, 256, 512), (64, 384, 256), (8200, 128, 128)],
                         ids=["bn128", "ragged_tokens_bn256", "one_stage", "long_ragged"])
def test_exact_integer_reference_shapes(M, N, K):
    """Small-integer operands make every product and partial sum exact in
    FP32, so R must equal the integer matmul whatever the reduction order:
    both tile widths, token counts that are not a multiple of the 64-token
    stage (zero-filled), one stage, many stages."""
    rng = np.random.default_rng(M + N + K)
    dyi, xi = rng.integers(-8, 9, size=(M, N)), rng.integers(-8, 9, size=(M, K))
    to_bf16 = lambda a: (a.astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    R = (dyi.T.astype(np.int64) @ xi.astype(np.int64)).astype(np.float32)
    D = torch.from_numpy(R + 1.0).cuda()
    (sdd, srr, mdd, mrr), Rg = monitor(to_bf16(dyi), to_bf16(xi), D)
    assert np.array_equal(Rg.cpu().numpy(), R)
    assert sdd == float(N * K) and mdd == 1.0
    assert mrr == float(np.abs(R).max())


def test_fp8_wgrad_error_matches_oracle():
    M, N, K = 1024, 256, 384
    dy = synth.bf16_normal((M, N), 71, 1e-3, 1e-3, 30.0)
    x = synth.bf16_normal((M, K), 72, 1.0, 1e-3, 50.0)
    ops = []
    for bits, fmt in ((dy, fg.E5M2), (x, fg.E4M3)):
        R_, C_ = bits.shape
        q, s = torch.empty((R_, C_), dtype=torch.uint8, device="cuda"), torch.empty((C_ // 128, R_), device="cuda")
        qT, sT = torch.empty((C_, R_), dtype=torch.uint8, device="cuda"), torch.empty((R_ // 128, C_), device="cuda")
        fg.quant_1x128(dev_bf16(bits), fmt, q, s, qT, sT)
        ops.append((qT, sT, fmt))
    (a, sa, fa), (b, sb, fb) = ops
    D = torch.empty((N, K), dtype=torch.float32, device="cuda")
    fg.blockscaled_gemm(a, fa, sa, fg.GRAN_1x128, b, fb, sb, fg.GRAN_1x128, D)
    assert_status_ok()
    got, _ = monitor(dy, x, D)
    ref = oracle.wgrad_recompute_error(dy, x, D.cpu().numpy())
    assert ref[0] > 0
    for g, r in zip(got, ref):
        assert abs(g - r) <= 1e-3 * abs(r), (got, ref)
    rel = np.sqrt(got[0] / got[1])
    assert 0 < rel < 0.1                     # the FP8 wgrad is close to the BF16 one


def test_no_rows_gives_zero_reference():
    N, K = 128, 256
    D = torch.ones((N, K), dtype=torch.float32, device="cuda")
    (sdd, srr, mdd, mrr), R = monitor(np.zeros((0, N), np.uint16), np.zeros((0, K), np.uint16), D)
    assert srr == 0.0 and mrr == 0.0 and sdd == float(N * K) and mdd == 1.0


def test_full_size_exact_properties():
    """The benchmarked size: dW_down [4096, 14336] recomputed over 8192 tokens.
    Small-integer operands make every product and partial sum exact in FP32
    (|R| <= 8192 * 64 < 2^24), so R is the integer matmul whatever the GEMM's
    reduction order: sampled entries equal int64 dot products, D = 0 gives
    sum (D-R)^2 = sum R^2 and max|D-R| = max|R|, and D = R gives zero error."""
    M, N, K = 8192, 4096, 14336
    g = torch.Generator(device="cuda").manual_seed(11)
    dy = torch.randint(-8, 9, (M, N), generator=g, device="cuda").to(torch.bfloat16)
    x = torch.randint(-8, 9, (M, K), generator=g, device="cuda").to(torch.bfloat16)
    R = torch.empty((N, K), dtype=torch.float32, device="cuda")
    D = torch.zeros((N, K), dtype=torch.float32, device="cuda")
    err = fg.new_wgrad_err()
    fg.wgrad_recompute_error(dy, x, D, R, err)
    assert_status_ok()
    sdd, srr, mdd, mrr = fg.wgrad_err_values(err)
    assert srr > 0 and abs(sdd - srr) <= 1e-12 * srr and mdd == mrr
    rng = np.random.default_rng(12)
    pn, pk = rng.integers(0, N, 4096), rng.integers(0, K, 4096)
    dyc = dy[:, torch.from_numpy(pn).cuda()].float().cpu().numpy().astype(np.int64)
    xc = x[:, torch.from_numpy(pk).cuda()].float().cpu().numpy().astype(np.int64)
    want = (dyc * xc).sum(axis=0)
    got = R[torch.from_numpy(pn).cuda(), torch.from_numpy(pk).cuda()].cpu().numpy()
    assert np.array_equal(got.astype(np.int64), want) and np.all(got == want)
    assert mrr == float(R.abs().max().item())
    fg.wgrad_recompute_error(dy, x, R.clone(), R, err)
    assert_status_ok()
    sdd2, srr2, mdd2, mrr2 = fg.wgrad_err_values(err)
    assert sdd2 == 0.0 and mdd2 == 0.0 and srr2 == srr and mrr2 == mrr
