"""Pins for the oracle's AdamW step with FP8 moments (m in E4M3, v in E5M2,
one scale per 128 consecutive parameters).

Independent references: the closed form of a step with zero gradient and zero
moments (pure decoupled weight decay), torch.optim.AdamW run from the
dequantized moments (its own operation order, so parameters agree within a
few binary32 ulps and the re-quantized moments within FP8 precision), and the
scale rule's invariant that each non-empty block holds a full-scale code."""
import numpy as np
import torch

import oracle
import synth

TORCH_FP8 = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def tdec(codes, fmt):
    return torch.from_numpy(np.ascontiguousarray(codes, np.uint8)).view(TORCH_FP8[fmt]).to(torch.float32).numpy()


def quantize_blocks(x, fmt):
    """Moments as the optimizer stores them, built with torch's FP8 conversion."""
    fm = 448.0 if fmt == oracle.E4M3 else 57344.0
    xb = x.reshape(-1, 128)
    amax = np.abs(xb).max(axis=1)
    s = np.where(amax == 0, np.float32(1), (amax / np.float32(fm)).astype(np.float32)).astype(np.float32)
    q = torch.from_numpy((xb / s[:, None]).astype(np.float32)).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    return q.reshape(-1), s


def state(n, seed):
    rng = np.random.default_rng(seed)
    p = rng.normal(0, 0.02, n).astype(np.float32)
    g = synth.bf16_normal((n,), seed + 1, 1e-3, 1e-3, 20.0)
    qm, sm = quantize_blocks(rng.normal(0, 1e-3, n).astype(np.float32), oracle.E4M3)
    qv, sv = quantize_blocks((rng.normal(0, 1e-3, n) ** 2).astype(np.float32), oracle.E5M2)
    return p, g, qm, sm, qv, sv


def test_zero_gradient_and_moments_is_pure_weight_decay():
    n = 512
    p = np.random.default_rng(3).normal(0, 1, n).astype(np.float32)
    z8, one = np.zeros(n, np.uint8), np.ones(n // 128, np.float32)
    h = oracle.adam_hyper(3e-4, 0.9, 0.95, 1e-8, 0.1, 7)
    p1, qm, sm, qv, sv = oracle.adam_fp8_step(p, np.zeros(n, np.uint16), z8, one, z8, one, h)
    assert np.array_equal(p1, p - h["lr"] * (h["wd"] * p))          # binary32 closed form
    assert not np.any(qm) and not np.any(qv) and np.all(sm == 1) and np.all(sv == 1)


def test_matches_torch_adamw():
    n, t = 4096, 5
    lr, b1, b2, eps, wd = 1e-3, 0.9, 0.95, 1e-8, 0.1
    p, g, qm, sm, qv, sv = state(n, 11)
    h = oracle.adam_hyper(lr, b1, b2, eps, wd, t)
    p1, qm1, sm1, qv1, sv1 = oracle.adam_fp8_step(p, g, qm, sm, qv, sv, h)

    m0 = (tdec(qm, oracle.E4M3).reshape(-1, 128) * sm[:, None]).reshape(-1)
    v0 = (tdec(qv, oracle.E5M2).reshape(-1, 128) * sv[:, None]).reshape(-1)
    param = torch.nn.Parameter(torch.from_numpy(p.copy()))
    opt = torch.optim.AdamW([param], lr=lr, betas=(b1, b2), eps=eps, weight_decay=wd, foreach=False)
    param.grad = torch.from_numpy(synth.bf16_bits_to_f32(g).astype(np.float32))
    opt.state[param] = {"step": torch.tensor(float(t - 1)), "exp_avg": torch.from_numpy(m0.copy()),
                        "exp_avg_sq": torch.from_numpy(v0.copy())}
    opt.step()
    pt = param.detach().numpy()
    mt = opt.state[param]["exp_avg"].numpy()
    vt = opt.state[param]["exp_avg_sq"].numpy()

    ulp = np.spacing(np.abs(pt)).astype(np.float64)
    upd = np.abs(p.astype(np.float64) - pt)
    assert np.all(np.abs(p1.astype(np.float64) - pt) <= 4 * ulp + 1e-5 * upd)
    m1 = (tdec(qm1, oracle.E4M3).reshape(-1, 128) * sm1[:, None]).reshape(-1)
    v1 = (tdec(qv1, oracle.E5M2).reshape(-1, 128) * sv1[:, None]).reshape(-1)
    sm_e, sv_e = np.repeat(sm1, 128), np.repeat(sv1, 128)
    assert np.all(np.abs(m1 - mt) <= 2.0 ** -4 * np.abs(mt) + sm_e * 2.0 ** -9 + 1e-12)   # E4M3 half ulp
    assert np.all(np.abs(v1 - vt) <= 2.0 ** -3 * np.abs(vt) + sv_e * 2.0 ** -16 + 1e-20)  # E5M2 half ulp
    # a wrong momentum coefficient is caught
    bad = dict(h, omb1=h["b1"])
    assert not np.array_equal(oracle.adam_fp8_step(p, g, qm, sm, qv, sv, bad)[1], qm1)


def test_every_nonempty_block_holds_a_full_scale_code():
    p, g, qm, sm, qv, sv = state(2048, 21)
    _, qm1, sm1, qv1, sv1 = oracle.adam_fp8_step(p, g, qm, sm, qv, sv, oracle.adam_hyper(1e-3, 0.9, 0.95, 1e-8, 0, 2))
    assert np.all(np.any((qm1.reshape(-1, 128) & 0x7F) == 0x7E, axis=1))
    assert np.all(np.any((qv1.reshape(-1, 128) & 0x7F) == 0x7B, axis=1))
