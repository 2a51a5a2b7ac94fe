"""GPU parity of SwiGLU fused into the 1x128 quantizer with its transposed
128x1 copy (forward H = SwiGLU(GU), backward dGU from GU and dH).

The fused kernels never store the BF16 H / dGU, so parity is a chain:
the standalone SwiGLU kernels are within one BF16 ulp of the oracle's SwiGLU
(their own test), and the fused outputs equal, bit for bit, both the unfused
GPU composition (SwiGLU kernel, then the fused 1x128 + 128x1 quantizer) and
the oracle's 1x128 / 128x1 quantization of the GPU's BF16 SwiGLU values."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import assert_status_ok, dev_bf16, empty_f32, empty_u8, host_u16

pytestmark = pytest.mark.gpu


def quant_outputs(R, C):
    return empty_u8(R, C), empty_f32(C // 128, R), empty_u8(C, R), empty_f32(R // 128, C)


def unfused(gu, dh, fmt):
    R, F = gu.shape[0], gu.shape[1] // 2
    if dh is None:
        v = torch.empty((R, F), dtype=torch.bfloat16, device="cuda")
        fg.swiglu_fwd(gu, v)
    else:
        v = torch.empty((R, 2 * F), dtype=torch.bfloat16, device="cuda")
        fg.swiglu_bwd(gu, dh, v)
    out = quant_outputs(*v.shape)
    fg.quant_1x128(v, fmt, *out)
    return v, out


def fused(gu, dh, fmt):
    R, F = gu.shape[0], gu.shape[1] // 2
    out = quant_outputs(R, F if dh is None else 2 * F)
    if dh is None:
        fg.swiglu_quant_fwd(gu, fmt, *out)
    else:
        fg.swiglu_bwd_quant(gu, dh, fmt, *out)
    return out


def same_bits(a, b):
    if a.dtype == torch.float32:
        return torch.equal(a.view(torch.int32), b.view(torch.int32))
    return torch.equal(a, b)


@pytest.mark.parametrize("bwd", [False, True])
@pytest.mark.parametrize("fmt", [fg.E4M3, fg.E5M2])
def test_fused_equals_unfused_and_oracle(bwd, fmt):
    R, F = 384, 384                     # 3 x 3 (forward) / 3 x 6 (backward) tiles
    gu_h = synth.bf16_normal((R, 2 * F), 51, 2.0, 1e-3, 20.0)
    dh_h = synth.bf16_normal((R, F), 52, 1e-3, 1e-3, 50.0)
    gu, dh = dev_bf16(gu_h), (dev_bf16(dh_h) if bwd else None)
    v, ref = unfused(gu, dh, fmt)
    got = fused(gu, dh, fmt)
    assert_status_ok()
    for a, b in zip(got, ref):
        assert same_bits(a, b)
    # the oracle's quantizers on the GPU's SwiGLU values
    vb = host_u16(v)
    q, s, _ = oracle.quant_1x128(vb, fmt)
    qT, sT, _ = oracle.quant_128x1_transposed(vb, fmt)
    assert np.array_equal(got[0].cpu().numpy(), q)
    assert np.array_equal(got[1].cpu().numpy().view(np.uint32), s.view(np.uint32))
    assert np.array_equal(got[2].cpu().numpy(), qT)
    assert np.array_equal(got[3].cpu().numpy().view(np.uint32), sT.view(np.uint32))


@pytest.mark.parametrize("bwd", [False, True])
def test_fused_equals_unfused_at_mlp_size(bwd):
    """The MLP block's shapes: 8192 tokens, FFN 14336 (GU is [8192][28672]);
    forward H quantized E4M3, backward dGU quantized E5M2.  Everything is
    compared with the unfused GPU path, and one 128-row block with the oracle."""
    R, F = 8192, 14336
    g = torch.Generator(device="cuda").manual_seed(7)
    gu = (torch.randn((R, 2 * F), generator=g, device="cuda") * 2).to(torch.bfloat16)
    dh = (torch.randn((R, F), generator=g, device="cuda") * 1e-3).to(torch.bfloat16) if bwd else None
    fmt = fg.E5M2 if bwd else fg.E4M3
    v, ref = unfused(gu, dh, fmt)
    got = fused(gu, dh, fmt)
    assert_status_ok()
    for a, b in zip(got, ref):
        assert same_bits(a, b)
    # against the oracle on one 128-row block (whole 1x128 and 128x1 groups):
    # the GPU's SwiGLU within one BF16 ulp of the oracle's, the fused codes and
    # scales equal to the oracle's quantization of those GPU values
    mb = 37
    r0, r1 = mb * 128, mb * 128 + 128
    gu_h = host_u16(gu[r0:r1])
    want_v = oracle.swiglu_fwd(gu_h) if dh is None else oracle.swiglu_bwd(gu_h, host_u16(dh[r0:r1]))
    vb = host_u16(v[r0:r1])
    si = lambda b: np.where(b & 0x8000, -(b & 0x7FFF).astype(np.int64), (b & 0x7FFF).astype(np.int64))
    assert np.max(np.abs(si(vb) - si(want_v))) <= 1
    q, s, _ = oracle.quant_1x128(vb, fmt)
    qT, sT, _ = oracle.quant_128x1_transposed(vb, fmt)
    assert np.array_equal(got[0][r0:r1].cpu().numpy(), q)
    assert np.array_equal(got[1][:, r0:r1].cpu().numpy().view(np.uint32), s.view(np.uint32))
    assert np.array_equal(got[2][:, r0:r1].cpu().numpy(), qT)
    assert np.array_equal(got[3][mb:mb + 1].cpu().numpy().view(np.uint32), sT.view(np.uint32))


def test_nonfinite_gate_is_reported():
    R, F = 128, 128
    gu_h = synth.bf16_normal((R, 2 * F), 61, 1.0)
    gu_h[5, 7] = 0x7F80                 # +Inf gate: SwiGLU gives Inf
    out = quant_outputs(R, F)
    fg.swiglu_quant_fwd(dev_bf16(gu_h), fg.E4M3, *out)
    assert fg.device_status() == fg.ERR_NONFINITE


def test_empty_is_a_no_op():
    gu = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    fg.swiglu_quant_fwd(gu, fg.E4M3, *quant_outputs(0, 128))
    fg.swiglu_bwd_quant(gu, torch.empty((0, 128), dtype=torch.bfloat16, device="cuda"), fg.E5M2,
                        *quant_outputs(0, 256))
    assert_status_ok()


def test_zero_inputs_give_zero_codes_and_unit_scales():
    """SwiGLU(0, u) = +-0 and dGU(g, u, 0) = +-0: every group's amax is 0, so
    s = 1 and every code is a zero (0x00 or 0x80, the sign of the product)."""
    R, F = 256, 256
    gu = dev_bf16(synth.bf16_normal((R, 2 * F), 71, 1.0))
    zero_gate = gu.clone()
    zero_gate[:, :F] = 0
    for dh in (None, torch.zeros((R, F), dtype=torch.bfloat16, device="cuda")):
        out = fused(zero_gate if dh is None else gu, dh, fg.E4M3)
        assert_status_ok()
        assert not torch.any(out[0] & 0x7F) and not torch.any(out[2] & 0x7F)
        assert torch.all(out[1] == 1.0) and torch.all(out[3] == 1.0)
