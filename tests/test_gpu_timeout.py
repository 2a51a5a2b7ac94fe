"""The bounded wait gives up with FP8_ERR_TIMEOUT instead of hanging, and the
CUDA context stays usable afterwards.  The wait runs on a barrier that
nothing arrives at; no fault, trap or endless loop is involved."""
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_and_context_survives():
    assert fg.device_status() == fg.OK
    fg.selftest_wait_timeout(20)
    assert fg.device_status() == fg.ERR_TIMEOUT
    assert fg.device_status() == fg.OK
    x = torch.ones((128, 128), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((128, 128), dtype=torch.uint8, device="cuda")
    s = torch.empty((1, 128), dtype=torch.float32, device="cuda")
    fg.quant_1x128(x, fg.E4M3, q, s)
    assert fg.device_status() == fg.OK
    assert int(q[0, 0]) == 0x7E and float(s[0, 0]) == float(torch.tensor(1.0) / torch.tensor(448.0))
