"""GPU parity of the tcgen05 FP8 GEMMs against the oracle's FP64 values.

Bar: |err| <= 1e-3 * max(|ref|, 1) on every compared output, plus the
stricter gate 1e-3 * max(|ref|, rms(ref)) that still bites on the small
dgrad / wgrad outputs; BF16 outputs get half a BF16 ulp of ref on top (the
rounding of the FP32 result).  BF16 outputs must also equal
the round-to-nearest-even of the FP32 outputs bit for bit."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import (CANARY_BYTE, assert_status_ok, bf16_to_f64, dev_f32, dev_u8, gemm_tolerance_check,
                         guarded, host_u16, sample_points_dense)

pytestmark = pytest.mark.gpu


def quantized_operand(rows, K, seed, gran, fmt=oracle.E4M3, std=1.0, outliers=True):
    xb = synth.bf16_normal((rows, K), seed, std, 1e-3 if outliers else 0.0, 50.0)
    if gran == oracle.GRAN_1x128:
        q, s, _ = oracle.quant_1x128(xb, fmt)
    elif gran == oracle.GRAN_128x128:
        q, s, _ = oracle.quant_128x128(xb, fmt)
    else:
        st = oracle.DelayedState()
        st.scale[0] = np.float32(np.abs(synth.bf16_bits_to_f32(xb)).max() / oracle.fmax(fmt))
        q, used, _, _ = oracle.delayed_step(xb, st, fmt, want_stats=False)
        s = np.array([used], np.float32)
    return q, s


def run_gemm(qa, fa, sa, ga, qb, fb, sb, gb, out_dtype):
    M, N = qa.shape[0], qb.shape[0]
    D = guarded((M, N), out_dtype)
    fg.blockscaled_gemm(dev_u8(qa), fa, dev_f32(sa), ga, dev_u8(qb), fb, dev_f32(sb), gb, D)
    assert_status_ok()
    return D


def to_f64(D):
    if D.dtype == torch.float32:
        return D.cpu().numpy().astype(np.float64)
    return bf16_to_f64(host_u16(D))


CASES = [
    # name, M, N, K, (fmtA, granA), (fmtB, granB)
    ("tiny_fprop", 256, 256, 512, (oracle.E4M3, oracle.GRAN_1x128), (oracle.E4M3, oracle.GRAN_128x128)),
    ("bn128_tail", 384, 384, 640, (oracle.E4M3, oracle.GRAN_1x128), (oracle.E4M3, oracle.GRAN_128x128)),
    ("multi_wave", 1024, 1536, 1024, (oracle.E4M3, oracle.GRAN_1x128), (oracle.E4M3, oracle.GRAN_128x128)),
    ("wgrad_like", 512, 768, 1024, (oracle.E4M3, oracle.GRAN_1x128), (oracle.E4M3, oracle.GRAN_1x128)),
    ("wgrad_bn128", 256, 384, 512, (oracle.E4M3, oracle.GRAN_1x128), (oracle.E4M3, oracle.GRAN_1x128)),
    ("weight_as_A", 256, 512, 384, (oracle.E4M3, oracle.GRAN_128x128), (oracle.E4M3, oracle.GRAN_1x128)),
    ("tensor_e4m3", 512, 512, 1024, (oracle.E4M3, oracle.GRAN_TENSOR), (oracle.E4M3, oracle.GRAN_TENSOR)),
    ("tensor_hybrid", 256, 384, 2048, (oracle.E5M2, oracle.GRAN_TENSOR), (oracle.E4M3, oracle.GRAN_TENSOR)),
    ("tensor_e5m2_b", 256, 256, 512, (oracle.E4M3, oracle.GRAN_TENSOR), (oracle.E5M2, oracle.GRAN_TENSOR)),
    ("e5m2_blocks", 256, 512, 512, (oracle.E5M2, oracle.GRAN_1x128), (oracle.E4M3, oracle.GRAN_128x128)),
]


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_gemm_full_compare(case):
    name, M, N, K, (fa, ga), (fb, gb) = case
    qa, sa = quantized_operand(M, K, 11, ga, fa)
    qb, sb = quantized_operand(N, K, 12, gb, fb, std=0.5)
    ref = oracle.gemm_full(qa, fa, sa, ga, qb, fb, sb, gb)
    d32 = run_gemm(qa, fa, sa, ga, qb, fb, sb, gb, torch.float32)
    gemm_tolerance_check(to_f64(d32), ref, bf16_out=False)
    d16 = run_gemm(qa, fa, sa, ga, qb, fb, sb, gb, torch.bfloat16)
    gemm_tolerance_check(to_f64(d16), ref, bf16_out=True)
    # the BF16 output is the RNE rounding of the FP32 one
    assert torch.equal(d16, d32.to(torch.bfloat16))


def test_gemm_qkv_fprop_full_size_sampled():
    # Dense attention QKV projection: X [8192,4096] 1x128, W [6144,4096] 128x128
    xb, wb = synth.qkv_fprop()
    qa, sa, _ = oracle.quant_1x128(xb)
    qb, sb, _ = oracle.quant_128x128(wb)
    D = run_gemm(qa, oracle.E4M3, sa, oracle.GRAN_1x128, qb, oracle.E4M3, sb, oracle.GRAN_128x128,
                 torch.bfloat16)
    pm, pn = sample_points_dense(8192, 6144, seed=1)
    ref = oracle.gemm_points(qa, oracle.E4M3, sa, oracle.GRAN_1x128, qb, oracle.E4M3, sb,
                             oracle.GRAN_128x128, pm, pn)
    got = bf16_to_f64(host_u16(D))[pm, pn]
    gemm_tolerance_check(got, ref, bf16_out=True)


@pytest.mark.parametrize("fa", [oracle.E4M3, oracle.E5M2], ids=["e4m3", "hybrid_e5m2"])
def test_gemm_pertensor_full_size_sampled(fa):
    """Per-tensor scaling at its benchmarked size: X [16384,4096] (E4M3, or
    E5M2 for the HYBRID gradient side) x W [4096,4096] E4M3, whole-K
    accumulation on the tensor cores and one scale product, BF16 out."""
    M, N, K = 16384, 4096, 4096
    qa, sa = quantized_operand(M, K, 31, oracle.GRAN_TENSOR, fa)
    qb, sb = quantized_operand(N, K, 32, oracle.GRAN_TENSOR, oracle.E4M3, std=0.02)
    D = run_gemm(qa, fa, sa, oracle.GRAN_TENSOR, qb, oracle.E4M3, sb, oracle.GRAN_TENSOR, torch.bfloat16)
    pm, pn = sample_points_dense(M, N, seed=3)
    ref = oracle.gemm_points(qa, fa, sa, oracle.GRAN_TENSOR, qb, oracle.E4M3, sb, oracle.GRAN_TENSOR, pm, pn)
    got = bf16_to_f64(host_u16(D))[pm, pn]
    gemm_tolerance_check(got, ref, bf16_out=True)


def test_gemm_k_zero_gives_zeros_and_empty_is_no_op():
    D = torch.full((256, 256), 7.0, dtype=torch.float32, device="cuda")
    z = torch.empty(0, dtype=torch.uint8, device="cuda")
    zf = torch.empty(0, dtype=torch.float32, device="cuda")
    rc = fg.lib().fp8_blockscaled_gemm(256, 256, 0, None, 0, None, 0, None, 0, None, 1, D.data_ptr(), 1, 256,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == fg.OK
    assert_status_ok()
    assert torch.count_nonzero(D).item() == 0
    rc = fg.lib().fp8_blockscaled_gemm(0, 256, 128, z.data_ptr(), 0, zf.data_ptr(), 0, z.data_ptr(), 0,
                                       zf.data_ptr(), 1, D.data_ptr(), 1, 256,
                                       torch.cuda.current_stream().cuda_stream)
    assert rc == fg.OK


def test_gemm_repeated_calls_are_deterministic():
    qa, sa = quantized_operand(512, 1024, 21, oracle.GRAN_1x128)
    qb, sb = quantized_operand(512, 1024, 22, oracle.GRAN_128x128)
    d1 = run_gemm(qa, 0, sa, 0, qb, 0, sb, 1, torch.float32)
    d2 = run_gemm(qa, 0, sa, 0, qb, 0, sb, 1, torch.float32)
    assert torch.equal(d1, d2)


LD_CASES = [
    # name, M, N, K, ldD - N, out dtype: the BF16 tile leaves through shared memory and TMA
    # stores (BN = 256, K <= 8192), straight from registers (BN = 256, K > 8192; BN = 128), FP32
    ("bf16_tma_store_bn256", 384, 512, 1024, 64, torch.bfloat16),
    ("bf16_direct_long_k", 256, 512, 8320, 64, torch.bfloat16),
    ("bf16_bn128", 384, 384, 640, 32, torch.bfloat16),
    ("f32_bn256", 256, 512, 512, 8, torch.float32),
]


@pytest.mark.parametrize("case", LD_CASES, ids=[c[0] for c in LD_CASES])
def test_gemm_output_leading_dimension(case):
    """D given as a column slice of a wider matrix (ldD > N): the N columns of
    every row match the oracle and the padding columns keep their sentinel,
    whichever store path the output takes."""
    name, M, N, K, pad, dt = case
    qa, sa = quantized_operand(M, K, 41, oracle.GRAN_1x128)
    qb, sb = quantized_operand(N, K, 42, oracle.GRAN_128x128, std=0.5)
    ref = oracle.gemm_full(qa, 0, sa, oracle.GRAN_1x128, qb, 0, sb, oracle.GRAN_128x128)
    full = guarded((M, N + pad), dt)
    D = full[:, :N]
    fg.blockscaled_gemm(dev_u8(qa), 0, dev_f32(sa), fg.GRAN_1x128, dev_u8(qb), 0, dev_f32(sb), fg.GRAN_128x128, D)
    assert_status_ok()
    gemm_tolerance_check(to_f64(D.contiguous()), ref, bf16_out=dt == torch.bfloat16)
    padding = full[:, N:].contiguous().view(torch.uint8)
    assert bool((padding == CANARY_BYTE).all()), "the GEMM wrote into the padding columns of D"
