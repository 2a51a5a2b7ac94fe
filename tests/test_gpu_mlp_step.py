"""GPU parity of the dense SwiGLU MLP training step at its full size (8192
tokens, hidden 4096, FFN 14336), run exactly as the benchmark times it: one
pass of ``bench.MlpStep`` (14 launches, the same kernels, shapes, layouts and
launch configuration).

Every one of the six GEMMs is compared with the oracle's unrounded FP64 value
on a stratified sample of at least 2^20 outputs that hits every 128x128
output tile at least 16 times (its four corners among them), computed from
the FP8 operands the step itself produced.
Those operands are pinned separately: the quantizations of X, dY and W_gu
equal the oracle's on whole 128-row blocks, and the on-demand weight
transposes equal the byte / scale-grid transposes bit for bit.  (The SwiGLU-
fused quantizations of H and dGU are compared with the oracle at this size in
the SwiGLU tests.)"""
import numpy as np
import pytest
import torch

import bench
import fp8_fine_grained_x128_gb300 as fg
import oracle
from gpu_helpers import assert_status_ok, bf16_to_f64, gemm_tolerance_check, host_u16, sample_points_dense

pytestmark = pytest.mark.gpu

B1, BB = oracle.GRAN_1x128, oracle.GRAN_128x128


@pytest.fixture(scope="module")
def step():
    s = bench.MlpStep(torch.device("cuda", 0), seed=0)
    s.run()
    assert_status_ok()
    return s


def host(t):
    return t.cpu().numpy()


def sampled(D, pm, pn):
    got = D[torch.from_numpy(pm).cuda(), torch.from_numpy(pn).cuda()]
    if D.dtype == torch.float32:
        return got.cpu().numpy().astype(np.float64)
    return bf16_to_f64(host_u16(got))


# name, A, sA, granA, B, sB, granB, D (attribute names of MlpStep)
GEMMS = [
    ("fprop_gate_up", "qX", "sX", B1, "qWgu", "sWgu", BB, "GU"),
    ("fprop_down", "qH", "sH", B1, "qWd", "sWd", BB, "Y"),
    ("dgrad_down", "qdY", "sdY", B1, "qWdT", "sWdT", BB, "dH"),
    ("dgrad_gate_up", "qdGU", "sdGU", B1, "qWguT", "sWguT", BB, "dX"),
    ("wgrad_down", "qdYT", "sdYT", B1, "qHT", "sHT", B1, "dWd"),
    ("wgrad_gate_up", "qdGUT", "sdGUT", B1, "qXT", "sXT", B1, "dWgu"),
]


@pytest.mark.parametrize("i", range(len(GEMMS)), ids=[g[0] for g in GEMMS])
def test_step_gemm_sampled(step, i):
    name, a, sa, ga, b, sb, gb, d = GEMMS[i]
    A, B, D = getattr(step, a), getattr(step, b), getattr(step, d)
    M, K = A.shape
    N = B.shape[0]
    assert B.shape[1] == K and tuple(D.shape) == (M, N)
    pm, pn = sample_points_dense(M, N, per_tile=16, total=1 << 20, seed=100 + i)
    assert pm.size >= 1 << 20
    ref = oracle.gemm_points(host(A), oracle.E4M3, host(getattr(step, sa)), ga,
                             host(B), oracle.E4M3, host(getattr(step, sb)), gb, pm, pn)
    gemm_tolerance_check(sampled(D, pm, pn), ref, bf16_out=D.dtype == torch.bfloat16)


@pytest.mark.parametrize("src,q,s,qT,sT", [("X", "qX", "sX", "qXT", "sXT"), ("dY", "qdY", "sdY", "qdYT", "sdYT")])
@pytest.mark.parametrize("mb", [0, 41, 63])
def test_step_activation_quant_blocks(step, src, q, s, qT, sT, mb):
    r0, r1 = mb * 128, mb * 128 + 128
    xb = host_u16(getattr(step, src)[r0:r1])
    rq, rs, _ = oracle.quant_1x128(xb, oracle.E4M3)
    rqT, rsT, _ = oracle.quant_128x1_transposed(xb, oracle.E4M3)
    assert np.array_equal(host(getattr(step, q)[r0:r1]), rq)
    assert np.array_equal(host(getattr(step, s)[:, r0:r1]).view(np.uint32), rs.view(np.uint32))
    assert np.array_equal(host(getattr(step, qT)[:, r0:r1]), rqT)
    assert np.array_equal(host(getattr(step, sT)[mb:mb + 1]).view(np.uint32), rsT.view(np.uint32))


@pytest.mark.parametrize("nb", [0, 101, 223])
def test_step_weight_quant_blocks(step, nb):
    n0, n1 = nb * 128, nb * 128 + 128
    wb = host_u16(step.Wgu[n0:n1])
    rq, rs, _ = oracle.quant_128x128(wb, oracle.E4M3)
    assert np.array_equal(host(step.qWgu[n0:n1]), rq)
    assert np.array_equal(host(step.sWgu[nb:nb + 1]).view(np.uint32), rs.reshape(1, -1).view(np.uint32))


def test_step_weight_transposes_are_exact(step):
    for q, s, qT, sT in (("qWgu", "sWgu", "qWguT", "sWguT"), ("qWd", "sWd", "qWdT", "sWdT")):
        assert torch.equal(getattr(step, qT), getattr(step, q).t())
        assert torch.equal(getattr(step, sT).view(torch.int32), getattr(step, s).t().contiguous().view(torch.int32))
