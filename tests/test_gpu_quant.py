"""GPU parity of the quantizers against the oracle: bit-exact FP8 codes and
scales (1x128, fused 1x128 + transposed 128x1, 128x128 with and without the
fused transpose, the on-demand FP8 transpose), on seeded inputs with the
benchmark's laws, small shapes spanning several tiles with a ragged row tail,
the full benchmark shapes, and the degenerate cases."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import assert_status_ok, dev_bf16, empty_f32, empty_u8

pytestmark = pytest.mark.gpu

FMTS = [oracle.E4M3, oracle.E5M2]


def gpu_quant_1x128(xb, fmt, transposed=False):
    R, C = xb.shape
    x = dev_bf16(xb)
    q, s = empty_u8(R, C), empty_f32(C // 128, R)
    qT = sT = None
    if transposed:
        qT, sT = empty_u8(C, R), empty_f32(R // 128, C)
    fg.quant_1x128(x, fmt, q, s, qT, sT)
    assert_status_ok()
    out = [q.cpu().numpy(), s.cpu().numpy()]
    if transposed:
        out += [qT.cpu().numpy(), sT.cpu().numpy()]
    return out


def same_f32(a, b):
    return np.array_equal(np.asarray(a, np.float32).view(np.uint32), np.asarray(b, np.float32).view(np.uint32))


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(256, 512), (1000, 384), (3, 128)])
def test_1x128_rows_small(fmt, shape):
    xb = synth.bf16_normal(shape, 0, 1.0, 1e-3, 100.0)
    q, s = gpu_quant_1x128(xb, fmt)
    q_ref, s_ref, st = oracle.quant_1x128(xb, fmt)
    assert st == oracle.OK
    assert np.array_equal(q, q_ref)
    assert same_f32(s, s_ref)


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("shape", [(256, 512), (384, 256), (128, 128)])
def test_1x128_fused_transposed_small(fmt, shape):
    xb = synth.bf16_normal(shape, 1, 1.0, 1e-3, 50.0)
    q, s, qT, sT = gpu_quant_1x128(xb, fmt, transposed=True)
    q_ref, s_ref, _ = oracle.quant_1x128(xb, fmt)
    qT_ref, sT_ref, _ = oracle.quant_128x1_transposed(xb, fmt)
    assert np.array_equal(q, q_ref) and same_f32(s, s_ref)
    assert np.array_equal(qT, qT_ref) and same_f32(sT, sT_ref)


def test_1x128_full_size_activation_and_gradient():
    # X of the dense layers: [8192, 4096], N(0,1) + 0.1% outliers x50
    xb = synth.bf16_normal((8192, 4096), 0, 1.0, 1e-3, 50.0)
    q, s, qT, sT = gpu_quant_1x128(xb, oracle.E4M3, transposed=True)
    q_ref, s_ref, _ = oracle.quant_1x128(xb, oracle.E4M3)
    assert np.array_equal(q, q_ref) and same_f32(s, s_ref)
    qT_ref, sT_ref, _ = oracle.quant_128x1_transposed(xb, oracle.E4M3)
    assert np.array_equal(qT, qT_ref) and same_f32(sT, sT_ref)
    q2, s2 = gpu_quant_1x128(xb, oracle.E4M3)          # the rows-only kernel agrees
    assert np.array_equal(q2, q_ref) and same_f32(s2, s_ref)
    # dY: N(0, 1e-3)
    db = synth.bf16_normal((8192, 4096), 3000, 1e-3)
    q, s = gpu_quant_1x128(db, oracle.E4M3)
    q_ref, s_ref, _ = oracle.quant_1x128(db, oracle.E4M3)
    assert np.array_equal(q, q_ref) and same_f32(s, s_ref)


@pytest.mark.parametrize("fmt", FMTS)
def test_every_bf16_value_against_many_scales(fmt):
    """Each 1x128 tile holds one amax A (fixing s = A/fmax) and 127 BF16 values
    with |x| <= A drawn from all 65536 patterns, for 256 scales spread over
    the whole binary32 range (including subnormal s): the per-element division
    must round exactly like IEEE x / s."""
    rng = np.random.default_rng(4)
    allv = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    finite = allv[(allv & 0x7F80) != 0x7F80]
    amax_bits = np.concatenate([rng.integers(0x0001, 0x7F7F, 250), [0x0001, 0x0080, 0x7F7F, 0x3F80, 0x4360, 0x0400]])
    tiles = []
    for a in amax_bits.astype(np.uint16):
        ok = finite[(finite & 0x7FFF) <= a]
        n_t = max(1, (len(ok) + 126) // 127)
        vals = np.resize(rng.permutation(ok), n_t * 127).reshape(n_t, 127)
        t = np.concatenate([np.full((n_t, 1), a, np.uint16), vals], axis=1)
        tiles.append(t)
    x = np.concatenate(tiles).astype(np.uint16)
    x = x[: (len(x) // 2) * 2].reshape(-1, 256)      # two tiles per row
    q, s = gpu_quant_1x128(x, fmt)
    q_ref, s_ref, st = oracle.quant_1x128(x, fmt)
    assert st == oracle.OK
    assert same_f32(s, s_ref)
    bad = np.count_nonzero(q != q_ref)
    assert bad == 0, f"{bad} codes differ"


@pytest.mark.parametrize("fmt", FMTS)
@pytest.mark.parametrize("transposed", [False, True])
@pytest.mark.parametrize("shape", [(256, 512), (6144, 4096)])
def test_128x128(fmt, transposed, shape):
    wb = synth.bf16_normal(shape, 1000, 0.02)
    if shape[0] == 256:
        wb = synth.bf16_normal(shape, 1000, 1.0, 1e-3, 100.0)
    R, C = shape
    w = dev_bf16(wb)
    q, s = empty_u8(R, C), empty_f32(R // 128, C // 128)
    qT, sT = (empty_u8(C, R), empty_f32(C // 128, R // 128)) if transposed else (None, None)
    fg.quant_128x128(w, fmt, q, s, qT, sT)
    assert_status_ok()
    q_ref, s_ref, st = oracle.quant_128x128(wb, fmt)
    assert np.array_equal(q.cpu().numpy(), q_ref) and same_f32(s.cpu().numpy(), s_ref)
    if transposed:
        assert np.array_equal(qT.cpu().numpy(), oracle.fp8_transpose(q_ref))
        assert same_f32(sT.cpu().numpy(), oracle.scale_grid_transpose(s_ref))


def test_on_demand_transpose():
    wb = synth.bf16_normal((1024, 768), 5, 0.02)
    q_ref, s_ref, _ = oracle.quant_128x128(wb)
    qT, sT = empty_u8(768, 1024), empty_f32(6, 8)
    fg.transpose_128x128(torch.from_numpy(q_ref).cuda(), torch.from_numpy(s_ref).cuda(), qT, sT)
    assert_status_ok()
    assert np.array_equal(qT.cpu().numpy(), oracle.fp8_transpose(q_ref))
    assert same_f32(sT.cpu().numpy(), oracle.scale_grid_transpose(s_ref))


def test_degenerate_tiles():
    x = np.zeros((128, 256), np.uint16)
    x[1, :] = 0x8000                     # -0 everywhere
    x[2, 0] = 0x0001                     # smallest subnormal: subnormal scale
    x[3, 5] = 0x7F7F                     # largest finite BF16
    x[4, :128] = 0x3F80                  # constant tile
    x[5, 130] = 0xC2C8                   # lone -100
    for fmt in FMTS:
        q, s, qT, sT = gpu_quant_1x128(x, fmt, transposed=True)
        q_ref, s_ref, _ = oracle.quant_1x128(x, fmt)
        qT_ref, sT_ref, _ = oracle.quant_128x1_transposed(x, fmt)
        assert np.array_equal(q, q_ref) and same_f32(s, s_ref)
        assert np.array_equal(qT, qT_ref) and same_f32(sT, sT_ref)


def test_nonfinite_is_reported():
    x = synth.bf16_normal((128, 256), 2)
    x[7, 9] = 0x7FC0   # NaN
    xd = dev_bf16(x)
    q, s = empty_u8(128, 256), empty_f32(2, 128)
    fg.quant_1x128(xd, fg.E4M3, q, s)
    assert fg.device_status() == fg.ERR_NONFINITE
    assert fg.device_status() == fg.OK      # reading clears it


def test_empty_is_a_no_op():
    x = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    fg.quant_1x128(x, fg.E4M3, empty_u8(0, 256), empty_f32(2, 0))
    assert_status_ok()
