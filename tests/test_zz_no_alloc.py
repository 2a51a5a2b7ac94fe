"""The no-allocation delayed-scaling entry point gives the same results as the
regular one.

Some callers cannot allocate device memory (code running inside another
framework's fixed memory plan, plugins that are handed buffers but no
allocator), so fp8_quant_pertensor_delayed_noalloc keeps its scratch in the
library's own device block instead of a caller workspace.  This test calls it
through the C ABI twice in a row -- the second call must not be disturbed by
what the first left in the shared block -- and compares every output and the
delayed-scaling state with fp8_quant_pertensor_delayed run on copies of the
same state.  The comparison is bit-exact, like every quantizer parity test.

The file name makes pytest collect it last, so a run that stops at the first
failure has already run every other test."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import synth

pytestmark = pytest.mark.gpu


def _dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


class _State:
    def __init__(self, fmt):
        self.recipe = fg.DelayedRecipe(fmt, 16, 0, fg.AMAX_MAX)
        self.hist = torch.zeros(16, dtype=torch.float32, device="cuda")
        self.step = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.scale = torch.ones(1, dtype=torch.float32, device="cuda")


@pytest.mark.parametrize("fmt", [fg.E4M3, fg.E5M2])
def test_noalloc_matches_workspace_entry_point_two_calls(fmt):
    R, C = 512, 384
    ref, new = _State(fmt), _State(fmt)
    ws = fg.new_workspace()
    for t in (0, 8):                       # two calls in a row, the second after a x1.5 drift
        x_bits, dy_bits = synth.delayed_step_inputs(t, m=R, hidden=C, n_out=C)
        x = _dev_bf16(x_bits if fmt == fg.E4M3 else dy_bits)
        outs = []
        for st, noalloc in ((ref, False), (new, True)):
            q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
            qT = torch.empty((C, R), dtype=torch.uint8, device="cuda")
            stats = fg.new_stats()
            if noalloc:
                fg.quant_pertensor_delayed_noalloc(x, st.recipe, st.hist, st.step, st.scale, q, qT, stats)
            else:
                fg.quant_pertensor_delayed(x, st.recipe, st.hist, st.step, st.scale, q, ws, qT, stats)
            assert fg.device_status() == fg.OK
            outs.append((q, qT, stats))
        (q0, qT0, s0), (q1, qT1, s1) = outs
        assert torch.equal(q0, q1) and torch.equal(qT0, qT1) and torch.equal(s0, s1)
        assert torch.equal(ref.hist, new.hist)
        assert torch.equal(ref.scale, new.scale) and torch.equal(ref.step, new.step)
    assert int(new.step.item()) == 2
