"""GPU parity of per-tensor current scaling (the FP8 KV-cache calibration):
codes and the device-written scale bit-exact against the oracle, on ragged
shapes, strided rows, an all-zero tensor, a tensor holding Inf/NaN (reported,
workspace left clean) and a 32k-token KV-cache layer."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import assert_status_ok, dev_bf16

pytestmark = pytest.mark.gpu


def run(xb, fmt, ws, ldx=None):
    R, C = xb.shape
    if ldx is None:
        x = dev_bf16(xb)
    else:
        full = np.zeros((R, ldx), np.uint16)
        full[:, :C] = xb
        x = dev_bf16(full)[:, :C]
    scale = torch.full((1,), float("nan"), device="cuda")
    q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    fg.quant_pertensor_current(x, fmt, scale, q, ws)
    return q, scale


@pytest.mark.parametrize("fmt", [fg.E4M3, fg.E5M2])
@pytest.mark.parametrize("shape,ldx", [((1000, 1024), None), ((3, 128), 136), ((4096, 8), None)])
def test_current_scaling_bit_exact(fmt, shape, ldx):
    ws = fg.new_workspace()
    xb = synth.bf16_normal(shape, 61, 0.5, 1e-3, 40.0)
    q, scale = run(xb, fmt, ws, ldx)
    assert_status_ok()
    rq, rs, st = oracle.quant_pertensor_current(xb, fmt)
    assert st == oracle.OK
    assert np.array_equal(q.cpu().numpy(), rq)
    assert scale.cpu().numpy().view(np.uint32)[0] == np.float32(rs).view(np.uint32)


def test_zero_tensor_and_nonfinite_then_clean_workspace():
    ws = fg.new_workspace()
    q, scale = run(np.zeros((64, 256), np.uint16), fg.E4M3, ws)
    assert_status_ok()
    assert float(scale.item()) == 1.0 and not q.any()
    bad = synth.bf16_normal((64, 256), 62)
    bad[5, 7] = 0x7FC0
    run(bad, fg.E4M3, ws)
    assert fg.device_status() == fg.ERR_NONFINITE
    xb = synth.bf16_normal((64, 256), 63)               # the workspace was left zeroed
    q, scale = run(xb, fg.E4M3, ws)
    assert_status_ok()
    rq, rs, _ = oracle.quant_pertensor_current(xb)
    assert np.array_equal(q.cpu().numpy(), rq) and np.float32(scale.item()) == np.float32(rs)


def test_kv_cache_layer_full_size():
    """One layer's K cache: 32768 tokens x 8 heads x 128, E4M3."""
    ws = fg.new_workspace()
    xb = synth.bf16_normal((32768, 1024), 64, 1.0, 1e-4, 20.0)
    q, scale = run(xb, fg.E4M3, ws)
    assert_status_ok()
    rq, rs, _ = oracle.quant_pertensor_current(xb)
    assert np.array_equal(q.cpu().numpy(), rq) and np.float32(scale.item()) == np.float32(rs)


@pytest.mark.parametrize("offset", [0, 8, 24])
def test_alignment_paths_agree(offset):
    """A contiguous tensor that starts on a 128-byte line is read with an L2
    evict_last policy in pass 1 and reset line by line in pass 2; one that is
    only 16-byte aligned (offset 8 or 24 BF16 elements) is read plainly.  Both
    give the oracle's codes and scale."""
    R, C = 1536, 640
    ws = fg.new_workspace()
    xb = synth.bf16_normal((R, C), 65 + offset, 2.0, 1e-3, 30.0)
    flat = torch.zeros(R * C + 128, dtype=torch.int16, device="cuda")
    flat[offset:offset + R * C] = torch.from_numpy(xb.reshape(-1).view(np.int16)).cuda()
    x = flat[offset:offset + R * C].view(torch.bfloat16).view(R, C)
    assert (x.data_ptr() % 128 == 0) == (offset == 0)
    scale = torch.full((1,), float("nan"), device="cuda")
    q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    fg.quant_pertensor_current(x, fg.E4M3, scale, q, ws)
    assert_status_ok()
    rq, rs, _ = oracle.quant_pertensor_current(xb)
    assert np.array_equal(q.cpu().numpy(), rq) and np.float32(scale.item()) == np.float32(rs)
