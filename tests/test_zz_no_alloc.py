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


def _run(st, x, noalloc, ws, want_T, want_stats):
    R, C = x.shape
    q = torch.empty((R, C), dtype=torch.uint8, device="cuda")
    qT = torch.empty((C, R), dtype=torch.uint8, device="cuda") if want_T else None
    stats = fg.new_stats() if want_stats else None
    if noalloc:
        fg.quant_pertensor_delayed_noalloc(x, st.recipe, st.hist, st.step, st.scale, q, qT, stats)
    else:
        fg.quant_pertensor_delayed(x, st.recipe, st.hist, st.step, st.scale, q, ws, qT, stats)
    return q, qT, stats


def _same_state(a, b):
    return torch.equal(a.hist, b.hist) and torch.equal(a.scale, b.scale) and torch.equal(a.step, b.step)


@pytest.mark.parametrize("want_stats", [True, False], ids=["stats", "no_stats"])
@pytest.mark.parametrize("want_T", [True, False], ids=["qT", "no_qT"])
@pytest.mark.parametrize("fmt", [fg.E4M3, fg.E5M2])
def test_noalloc_matches_workspace_entry_point_two_calls(fmt, want_T, want_stats):
    R, C = 512, 384
    ref, new = _State(fmt), _State(fmt)
    ws = fg.new_workspace()
    for t in (0, 8):                       # two calls in a row, the second after a x1.5 drift
        x_bits, dy_bits = synth.delayed_step_inputs(t, m=R, hidden=C, n_out=C)
        x = _dev_bf16(x_bits if fmt == fg.E4M3 else dy_bits)
        outs = []
        for st, noalloc in ((ref, False), (new, True)):
            outs.append(_run(st, x, noalloc, ws, want_T, want_stats))
            assert fg.device_status() == fg.OK
        (q0, qT0, s0), (q1, qT1, s1) = outs
        assert torch.equal(q0, q1)
        if want_T:
            assert torch.equal(qT0, qT1)
        if want_stats:
            assert torch.equal(s0, s1)
        assert _same_state(ref, new)
    assert int(new.step.item()) == 2


def test_noalloc_zero_rows_updates_state_like_the_workspace_entry_point():
    """A tensor with no rows still advances the delayed-scaling state (amax 0
    goes into the history); this path uses the scratch's last-CTA ticket."""
    ref, new = _State(fg.E4M3), _State(fg.E4M3)
    ws = fg.new_workspace()
    x_bits, _ = synth.delayed_step_inputs(0, m=256, hidden=256, n_out=256)
    x = _dev_bf16(x_bits)
    empty = torch.empty((0, 256), dtype=torch.bfloat16, device="cuda")
    for xx in (x, empty, x):
        _run(ref, xx, False, ws, False, True)
        _run(new, xx, True, ws, False, True)
        assert fg.device_status() == fg.OK
        assert _same_state(ref, new)
    assert int(new.step.item()) == 3


def test_noalloc_after_a_nonfinite_step():
    """A step whose tensor holds an Inf reports FP8_ERR_NONFINITE and leaves the
    state alone; the next call must start from a clean scratch (the entry
    point clears what it uses before every call) and match the workspace
    entry point bit for bit."""
    ref, new = _State(fg.E4M3), _State(fg.E4M3)
    ws = fg.new_workspace()
    R, C = 256, 384
    good = [synth.delayed_step_inputs(t, m=R, hidden=C, n_out=C)[0] for t in (0, 1)]
    bad = good[0].copy()
    bad[5, 7] = 0x7F80                    # +Inf
    for bits, expect in ((good[0], fg.OK), (bad, fg.ERR_NONFINITE), (good[1], fg.OK)):
        x = _dev_bf16(bits)
        outs = []
        for st, noalloc in ((ref, False), (new, True)):
            outs.append(_run(st, x, noalloc, ws, True, True))
            assert fg.device_status() == expect
        if expect == fg.OK:
            (q0, qT0, s0), (q1, qT1, s1) = outs
            assert torch.equal(q0, q1) and torch.equal(qT0, qT1) and torch.equal(s0, s1)
        assert _same_state(ref, new)
    assert int(new.step.item()) == 2
