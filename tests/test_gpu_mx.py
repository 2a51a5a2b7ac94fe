"""GPU parity of the MXFP8 quantizer (1x32 blocks, power-of-two scales):
codes and scale exponents bit-exact against the oracle (oracle/mx.py) on
ragged and strided shapes, blocks at the edges of the exponent rule (amax
exactly fmax * 2^j and just above, subnormal BF16 amax, all-zero blocks,
values near the BF16 maximum, signed zeros), a tensor holding Inf/NaN
(reported) and the 8192 x 4096 activation of the MLP step."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import assert_status_ok, dev_bf16
from oracle import mx

pytestmark = pytest.mark.gpu


def run(xb, fmt, ldx=None):
    R, C = xb.shape
    if ldx is None:
        x = dev_bf16(xb)
    else:
        full = np.zeros((R, ldx), np.uint16)
        full[:, :C] = xb
        x = dev_bf16(full)[:, :C]
    q = torch.full((R, C), 0x55, dtype=torch.uint8, device="cuda")
    e8 = torch.full((R, C // 32), 0x55, dtype=torch.uint8, device="cuda")
    fg.quant_mx(x, fmt, q, e8)
    return q.cpu().numpy(), e8.cpu().numpy()


def edge_cases(fmt):
    """Rows of 32-blocks built to sit on the exponent rule's edges."""
    rng = np.random.default_rng(7)
    fm = oracle.fmax(fmt)
    blocks, bump = [], []
    for j in (-30, -3, 0, 5, 100):
        peak = fm * 2.0 ** j
        for above in (False, True):
            b = rng.normal(0, peak / 4, 32).clip(-peak / 2, peak / 2)
            b[3] = -peak if above else peak           # amax exactly fmax * 2^j: X = 2^j
            if above:                                 # ... and one BF16 step above it: X = 2^(j+1)
                bump.append(len(blocks) * 32 + 3)
            blocks.append(b)
    blocks.append(np.zeros(32))                       # all zero: X = 1
    blocks.append(np.full(32, -0.0))                  # signed zeros
    blocks.append(rng.normal(0, 1, 32) * 2.0 ** -130)  # subnormal BF16 amax
    blocks.append(rng.normal(0, 1, 32) * 5e37)        # near the BF16 maximum
    x = np.concatenate(blocks).astype(np.float32)
    bits = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16).copy()
    bits[bump] += 1
    return np.tile(bits, (3, 1))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("shape,ldx", [((256, 1024), None), ((37, 96), None), ((5, 160), 200), ((1, 32), None)])
def test_mx_quant_bit_exact(fmt, shape, ldx):
    xb = synth.bf16_normal(shape, 41, 1.0, 1e-3, 50.0)
    q, e8 = run(xb, fmt, ldx)
    assert_status_ok()
    rq, re8, st = mx.quant_mx(xb, fmt)
    assert st == oracle.OK
    assert np.array_equal(e8, re8) and np.array_equal(q, rq)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_mx_quant_exponent_edges(fmt):
    xb = edge_cases(fmt)
    q, e8 = run(xb, fmt)
    assert_status_ok()
    rq, re8, _ = mx.quant_mx(xb, fmt)
    assert np.array_equal(e8, re8) and np.array_equal(q, rq)


def test_mx_quant_nonfinite_is_reported_and_empty_is_a_no_op():
    xb = synth.bf16_normal((4, 64), 42)
    xb[1, 33] = 0x7FC0
    run(xb, oracle.E4M3)
    assert fg.device_status() == fg.ERR_NONFINITE
    fg.quant_mx(torch.empty((0, 64), dtype=torch.bfloat16, device="cuda"), fg.E4M3,
                torch.empty((0, 64), dtype=torch.uint8, device="cuda"), torch.empty((0, 2), dtype=torch.uint8, device="cuda"))
    assert_status_ok()


def test_mx_quant_mlp_activation_full_size():
    """X of the MLP step, 8192 tokens x 4096, E4M3, every code and exponent."""
    xb = synth.bf16_normal((8192, 4096), 43, 1.0, 1e-3, 50.0)
    q, e8 = run(xb, oracle.E4M3)
    assert_status_ok()
    rq, re8, _ = mx.quant_mx(xb, oracle.E4M3)
    assert np.array_equal(e8, re8) and np.array_equal(q, rq)
