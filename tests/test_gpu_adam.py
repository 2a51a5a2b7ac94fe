"""GPU parity of the AdamW step with FP8 moments: parameters, E4M3 / E5M2
moment codes and their block scales bit-exact against the oracle, over
consecutive steps from zero moments (with blocks whose gradient stays zero)
and on a 117M-parameter tensor."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import assert_status_ok, dev_bf16

pytestmark = pytest.mark.gpu

HP = dict(lr=1e-3, beta1=0.9, beta2=0.95, eps=1e-8, weight_decay=0.1)


def hyper(step):
    return oracle.adam_hyper(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"], step)


def gpu_state(p, n):
    return dict(p=torch.from_numpy(p.copy()).cuda(), m=torch.zeros(n, dtype=torch.uint8, device="cuda"),
                sm=torch.ones(n // 128, device="cuda"), v=torch.zeros(n, dtype=torch.uint8, device="cuda"),
                sv=torch.ones(n // 128, device="cuda"))


def gpu_step(st, g_bits, step):
    h = fg.adamw_hparams(HP["lr"], HP["beta1"], HP["beta2"], HP["eps"], HP["weight_decay"], step)
    fg.adamw_step_fp8_states(st["p"], dev_bf16(g_bits), st["m"], st["sm"], st["v"], st["sv"], h)
    assert_status_ok()


def same(gpu, ref, view=None):
    a = gpu.cpu().numpy()
    return np.array_equal(a.view(view), ref.view(view)) if view else np.array_equal(a, ref)


def test_adamw_fp8_three_steps_bit_exact():
    n = 128 * 300
    p = np.random.default_rng(1).normal(0, 0.02, n).astype(np.float32)
    st = gpu_state(p, n)
    ref = (p, np.zeros(n, np.uint8), np.ones(n // 128, np.float32), np.zeros(n, np.uint8), np.ones(n // 128, np.float32))
    for step in (1, 2, 3):
        g = synth.bf16_normal((n,), 10 + step, 1e-3, 1e-3, 30.0)
        g[: 128 * 5] = 0                                 # blocks whose gradient stays zero
        gpu_step(st, g, step)
        ref = oracle.adam_fp8_step(ref[0], g, ref[1], ref[2], ref[3], ref[4], hyper(step))
        assert same(st["p"], ref[0], np.uint32)
        assert same(st["m"], ref[1]) and same(st["v"], ref[3])
        assert same(st["sm"], ref[2], np.uint32) and same(st["sv"], ref[4], np.uint32)
    assert np.all(st["sm"].cpu().numpy()[:5] == 1.0)


def test_adamw_fp8_full_size_one_step():
    n = 28672 * 4096
    rng = np.random.default_rng(2)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = synth.bf16_normal((n,), 3, 1e-3, 1e-3, 30.0)
    st = gpu_state(p, n)
    # a second step, so that the moments read back are non-trivial codes
    gpu_step(st, g, 1)
    ref = oracle.adam_fp8_step(p, g, np.zeros(n, np.uint8), np.ones(n // 128, np.float32), np.zeros(n, np.uint8),
                               np.ones(n // 128, np.float32), hyper(1))
    g2 = synth.bf16_normal((n,), 4, 1e-3, 1e-3, 30.0)
    gpu_step(st, g2, 2)
    ref = oracle.adam_fp8_step(ref[0], g2, ref[1], ref[2], ref[3], ref[4], hyper(2))
    assert same(st["p"], ref[0], np.uint32)
    assert same(st["m"], ref[1]) and same(st["v"], ref[3])
    assert same(st["sm"], ref[2], np.uint32) and same(st["sv"], ref[4], np.uint32)


@pytest.mark.parametrize("step", [1, 7, 100, 5000])
def test_adamw_fp8_random_moments_bit_exact(step):
    """One step from random moment codes and scales (magnitudes over many
    binades, both signs of m, zero codes and zero blocks among them) at step
    numbers whose bias corrections run from 0.1 / 0.05 to 1: the bias-corrected
    moments m / bc1 and v / bc2 are divided through the corrections'
    reciprocals, and must match the oracle's IEEE quotients bit for bit."""
    n = 128 * 2048
    rng = np.random.default_rng(100 + step)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    qm = rng.integers(0, 256, n, dtype=np.uint8)
    qm[(qm & 0x7F) == 0x7F] = 0x7E                       # no NaN codes in the state (E4M3 S.1111.111)
    qv = rng.integers(0, 0x7C, n, dtype=np.uint8)        # E5M2 v >= 0: finite codes, zeros included
    qm[:128 * 3] = 0
    qv[:128 * 3] = 0
    sm = (2.0 ** rng.uniform(-40, 2, n // 128)).astype(np.float32)
    sv = (2.0 ** rng.uniform(-60, 0, n // 128)).astype(np.float32)
    g = synth.bf16_normal((n,), 200 + step, 1e-3, 1e-3, 30.0)
    st = dict(p=torch.from_numpy(p.copy()).cuda(), m=torch.from_numpy(qm.copy()).cuda(),
              sm=torch.from_numpy(sm.copy()).cuda(), v=torch.from_numpy(qv.copy()).cuda(),
              sv=torch.from_numpy(sv.copy()).cuda())
    gpu_step(st, g, step)
    ref = oracle.adam_fp8_step(p, g, qm, sm, qv, sv, hyper(step))
    assert same(st["p"], ref[0], np.uint32)
    assert same(st["m"], ref[1]) and same(st["v"], ref[3])
    assert same(st["sm"], ref[2], np.uint32) and same(st["sv"], ref[4], np.uint32)
