"""GPU parity of the per-tensor delayed-scaling step (codes, transposed codes,
amax history, scale, step counter, fused monitors -- all bit-exact) over the
32-step drifting workload, the checkpoint-split invariant on the device, the
HYBRID per-tensor GEMMs, and the standalone monitors of the fine-grained
quantizations."""
import numpy as np
import pytest
import torch

import fp8_fine_grained_x128_gb300 as fg
import oracle
import synth
from gpu_helpers import (assert_status_ok, bf16_to_f64, dev_bf16, dev_f32, dev_u8, empty_f32, empty_u8,
                         gemm_tolerance_check, host_u16)

pytestmark = pytest.mark.gpu


class GpuDelayed:
    """Device-resident delayed-scaling state for one tensor."""

    def __init__(self, fmt, history_len=16, margin=0, algo=fg.AMAX_MAX):
        self.recipe = fg.DelayedRecipe(fmt, history_len, margin, algo)
        self.hist = torch.zeros(history_len, dtype=torch.float32, device="cuda")
        self.step = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.scale = torch.ones(1, dtype=torch.float32, device="cuda")
        self.ws = fg.new_workspace()

    def run(self, xb, want_T=True, want_stats=True):
        R, C = xb.shape
        x = dev_bf16(xb)
        q = empty_u8(R, C)
        qT = empty_u8(C, R) if want_T else None
        stats = fg.new_stats() if want_stats else None
        fg.quant_pertensor_delayed(x, self.recipe, self.hist, self.step, self.scale, q, self.ws, qT, stats)
        assert_status_ok()
        return q, qT, stats


def check_against_oracle(g: GpuDelayed, st: oracle.DelayedState, xb, fmt, margin=0, algo=0):
    q, qT, stats = g.run(xb)
    q_ref, used, stats_ref, code = oracle.delayed_step(xb, st, fmt, margin, algo)
    assert code == oracle.OK
    assert np.array_equal(q.cpu().numpy(), q_ref)
    assert np.array_equal(qT.cpu().numpy(), q_ref.T)
    assert np.array_equal(stats.cpu().numpy().astype(np.uint64), stats_ref)
    assert np.array_equal(g.hist.cpu().numpy().view(np.uint32), st.hist.view(np.uint32))
    assert g.scale.cpu().numpy().view(np.uint32)[0] == st.scale.view(np.uint32)[0]
    assert int(g.step.item()) == int(st.step[0])
    return q_ref, used, stats_ref


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_delayed_32_steps_small(fmt):
    g = GpuDelayed(fmt)
    st = oracle.DelayedState(16)
    for t in range(32):
        xb, dyb = synth.delayed_step_inputs(t, m=512, hidden=384, n_out=384)
        check_against_oracle(g, st, xb if fmt == oracle.E4M3 else dyb, fmt)


def test_delayed_knobs():
    for margin, algo, L in [(2, fg.AMAX_MAX, 4), (-1, fg.AMAX_MOST_RECENT, 1), (0, fg.AMAX_MAX, 1024)]:
        g = GpuDelayed(oracle.E4M3, L, margin, algo)
        st = oracle.DelayedState(L)
        for t in range(5):
            xb, _ = synth.delayed_step_inputs(3 * t, m=256, hidden=256, n_out=256)
            check_against_oracle(g, st, xb, oracle.E4M3, margin, algo)


def test_delayed_full_size_32_steps():
    """The delayed-scaling workload exactly as stated: a 16384 x 4096 Linear
    over 32 steps of drifting signed-lognormal X (E4M3) and dY (E5M2), history
    length 16, max algorithm, margin 0.  At every step codes, transposed
    codes, the 16-slot history, the next scale, the step counter and the
    fused monitor counts equal the oracle's; the drift steps (8, 16, 24)
    saturate and the history window wraps at step 16."""
    gx, gd = GpuDelayed(oracle.E4M3), GpuDelayed(oracle.E5M2)
    sx, sd = oracle.DelayedState(16), oracle.DelayedState(16)
    sat = {}
    for t in range(32):
        xb, dyb = synth.delayed_step_inputs(t)
        sat[t] = int(check_against_oracle(gx, sx, xb, oracle.E4M3)[2][2])
        check_against_oracle(gd, sd, dyb, oracle.E5M2)
    assert all(sat[t] > 0 for t in (8, 16, 24)), sat       # the drift outruns the delayed scale
    assert int(gx.step.item()) == 32 and int(gd.step.item()) == 32
    assert np.all(sx.hist > 0) and np.all(sd.hist > 0)        # every slot of the window written


def test_delayed_checkpoint_split_on_device():
    xs = [synth.delayed_step_inputs(t, m=256, hidden=384, n_out=384)[0] for t in range(10)]
    a = GpuDelayed(oracle.E4M3)
    qa = [a.run(x)[0].cpu().numpy() for x in xs]
    b = GpuDelayed(oracle.E4M3)
    qb = [b.run(x)[0].cpu().numpy() for x in xs[:4]]
    c = GpuDelayed(oracle.E4M3)            # fresh buffers, state copied in
    c.hist.copy_(b.hist)
    c.step.copy_(b.step)
    c.scale.copy_(b.scale)
    qb += [c.run(x)[0].cpu().numpy() for x in xs[4:]]
    assert all(np.array_equal(u, v) for u, v in zip(qa, qb))
    assert torch.equal(a.hist, c.hist) and torch.equal(a.scale, c.scale) and torch.equal(a.step, c.step)


def test_delayed_ragged_rows_no_transpose():
    g = GpuDelayed(oracle.E4M3)
    st = oracle.DelayedState(16)
    for t in range(3):
        xb, _ = synth.delayed_step_inputs(t, m=300, hidden=256, n_out=256)
        q, _, stats = g.run(xb, want_T=False)
        q_ref, _, stats_ref, _ = oracle.delayed_step(xb, st, oracle.E4M3)
        assert np.array_equal(q.cpu().numpy(), q_ref)
        assert np.array_equal(stats.cpu().numpy().astype(np.uint64), stats_ref)
        assert g.scale.cpu().numpy().view(np.uint32)[0] == st.scale.view(np.uint32)[0]


def test_delayed_nonfinite_leaves_state_untouched():
    g = GpuDelayed(oracle.E4M3)
    xb, _ = synth.delayed_step_inputs(0, m=256, hidden=256, n_out=256)
    g.run(xb)
    hist, scale, step = g.hist.clone(), g.scale.clone(), g.step.clone()
    bad = xb.copy()
    bad[3, 3] = 0x7F80   # +Inf
    x = dev_bf16(bad)
    q = empty_u8(256, 256)
    fg.quant_pertensor_delayed(x, g.recipe, g.hist, g.step, g.scale, q, g.ws)
    assert fg.device_status() == fg.ERR_NONFINITE
    assert torch.equal(hist, g.hist) and torch.equal(scale, g.scale) and torch.equal(step, g.step)
    # the workspace was left clean: the next good step matches the oracle
    st = oracle.DelayedState(16)
    oracle.delayed_step(xb, st, oracle.E4M3)
    check_against_oracle(g, st, xb, oracle.E4M3)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_delayed_overflowing_quotients_saturate(fmt):
    """A scale carried over from a step with a tiny amax can make x / s overflow
    binary32 this step: such elements saturate like the IEEE quotient says
    (Inf -> +-fmax), they are counted as saturated, and the step's state update
    still follows the oracle."""
    R, C = 256, 384
    xb = synth.bf16_signed_lognormal((R, C), 17, 0.0, 2.0)      # |x| up to ~1e4
    for s0 in (2.0 ** -124, 2.0 ** -118, 1e-30):
        g = GpuDelayed(fmt)
        g.scale.fill_(s0)
        st = oracle.DelayedState(16)
        st.scale[:] = np.float32(s0)
        q_ref, _, _ = check_against_oracle(g, st, xb, fmt)
        assert (q_ref & 0x7F == (0x7E if fmt == oracle.E4M3 else 0x7B)).sum() > 0


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("nans", [(0x7FC1,), (0xFFC1,), (0x7FC1, 0xFFC1, 0xFF81)], ids=["pos_nan", "neg_nan", "both_nans"])
def test_delayed_nonfinite_codes_follow_ieee_quotients(fmt, nans):
    """A step holding Inf and NaN still writes its codes and monitors like the
    IEEE quotients say (Inf -> +-fmax, NaN of either sign -> the NaN code 0x7F)."""
    g = GpuDelayed(fmt)
    xb, _ = synth.delayed_step_inputs(0, m=256, hidden=256, n_out=256)
    g.run(xb)
    st = oracle.DelayedState(16)
    oracle.delayed_step(xb, st, fmt)
    bad = xb.copy()
    bad[3, 3], bad[7, 200] = 0x7F80, 0xFF80                          # +Inf, -Inf
    for i, nb in enumerate(nans):
        bad[100 + i, 5 + 7 * i] = nb
    q = empty_u8(256, 256)
    qT = empty_u8(256, 256)
    stats = fg.new_stats()
    fg.quant_pertensor_delayed(dev_bf16(bad), g.recipe, g.hist, g.step, g.scale, q, g.ws, qT, stats)
    assert fg.device_status() == fg.ERR_NONFINITE
    q_ref, _, stats_ref, code = oracle.delayed_step(bad, st, fmt)
    assert code == oracle.NONFINITE
    assert np.array_equal(q.cpu().numpy(), q_ref) and np.array_equal(qT.cpu().numpy(), q_ref.T)
    assert np.array_equal(stats.cpu().numpy().astype(np.uint64), stats_ref)


def test_hybrid_per_tensor_gemms():
    """fprop E4M3 x E4M3, dgrad E5M2 x E4M3 (W^T), wgrad E5M2 x E4M3 (both transposed copies)."""
    M, H, N = 1024, 512, 384
    gx, gw, gd = GpuDelayed(oracle.E4M3), GpuDelayed(oracle.E4M3), GpuDelayed(oracle.E5M2)
    for t in range(3):   # run a few steps so the scales come from history
        xb, dyb = synth.delayed_step_inputs(t, m=M, hidden=H, n_out=N)
        wb = synth.bf16_normal((N, H), 7, 0.02)
        qx, qxT, _ = gx.run(xb)
        sx = gx.hist.new_empty(1)
        qw, qwT, _ = gw.run(wb)
        qd, qdT, _ = gd.run(dyb)
    # scales used at the last step are the ones before the step's update:
    # recompute them through the oracle state machine
    stx, stw, std = oracle.DelayedState(16), oracle.DelayedState(16), oracle.DelayedState(16)
    for t in range(3):
        xb, dyb = synth.delayed_step_inputs(t, m=M, hidden=H, n_out=N)
        wb = synth.bf16_normal((N, H), 7, 0.02)
        qx_r, s_x, _, _ = oracle.delayed_step(xb, stx, oracle.E4M3)
        qw_r, s_w, _, _ = oracle.delayed_step(wb, stw, oracle.E4M3)
        qd_r, s_d, _, _ = oracle.delayed_step(dyb, std, oracle.E5M2)
    assert np.array_equal(qx.cpu().numpy(), qx_r) and np.array_equal(qd.cpu().numpy(), qd_r)
    T = oracle.GRAN_TENSOR
    cases = [
        ("fprop", qx_r, oracle.E4M3, s_x, qw_r, oracle.E4M3, s_w),
        ("dgrad", qd_r, oracle.E5M2, s_d, np.ascontiguousarray(qw_r.T), oracle.E4M3, s_w),
        ("wgrad", np.ascontiguousarray(qd_r.T), oracle.E5M2, s_d, np.ascontiguousarray(qx_r.T), oracle.E4M3, s_x),
    ]
    for name, A, fa, sa, B, fb, sb in cases:
        sa_, sb_ = np.float32([sa]), np.float32([sb])
        ref = oracle.gemm_full(A, fa, sa_, T, B, fb, sb_, T)
        D = torch.empty((A.shape[0], B.shape[0]), dtype=torch.float32, device="cuda")
        fg.blockscaled_gemm(dev_u8(A), fa, dev_f32(sa_), T, dev_u8(B), fb, dev_f32(sb_), T, D)
        assert_status_ok()
        gemm_tolerance_check(D.cpu().numpy().astype(np.float64), ref, bf16_out=False)


# ------------------------------------------------------------- standalone stats

@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_quant_stats_all_granularities(fmt):
    R, C = 384, 512
    xb = synth.bf16_signed_lognormal((R, C), 4, -2.0, 3.0)
    xb[0, :64] = 0
    xb[1, :7] = 0x8000
    x = dev_bf16(xb)
    cases = []
    q, s, _ = oracle.quant_1x128(xb, fmt)
    cases.append((oracle.GRAN_1x128, q, s))
    q, s, _ = oracle.quant_128x128(xb, fmt)
    cases.append((oracle.GRAN_128x128, q, s))
    q, s, _ = oracle.quant_128x1_transposed(xb, fmt)
    cases.append((oracle.GRAN_128x1, q, s))
    cases.append((oracle.GRAN_TENSOR, oracle.fp8_encode(synth.bf16_bits_to_f32(xb) / np.float32(0.01), fmt),
                  np.float32([0.01])))
    ws = fg.new_workspace()
    for gran, q, s in cases:
        stats = fg.new_stats()
        fg.quant_stats(x, dev_u8(q), dev_f32(np.atleast_1d(s)), gran, fmt, stats, ws)
        assert_status_ok()
        ref = oracle.quant_stats(xb, q, s, gran, fmt)
        assert np.array_equal(stats.cpu().numpy().astype(np.uint64), ref), (gran, stats, ref)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("gran", [oracle.GRAN_1x128, oracle.GRAN_128x1, oracle.GRAN_128x128])
def test_quant_stats_saturation_boundary_and_odd_scales(gran, fmt):
    """Scales that put |x / s| within a few ulps of fmax (the saturation count
    is decided by the exact binary32 quotient), and scales far outside the
    normal range (0, -0, subnormal, huge, FLT_MAX, Inf, NaN, negative, 2^-125
    where x / s overflows); x holds +-Inf, NaN and -0 among its values."""
    R, C = 256, 512
    fm = np.float32(oracle.fmax(fmt))
    rng = np.random.default_rng(5 + fmt)
    xb = synth.bf16_signed_lognormal((R, C), 23, 0.0, 1.5)
    specials = np.array([0x7F80, 0xFF80, 0x7FC0, 0x8000, 0x7F7F, 0x0001], np.uint16)   # Inf, -Inf, NaN, -0, max, min subnormal
    where = rng.choice(R * C, size=64, replace=False)
    xb.ravel()[where] = specials[np.arange(64) % len(specials)]
    xf = synth.bf16_bits_to_f32(xb)
    if gran == oracle.GRAN_1x128:
        shape, pick = (C // 128, R), lambda i, j: xf[j, i * 128:(i + 1) * 128]
    elif gran == oracle.GRAN_128x1:
        shape, pick = (R // 128, C), lambda i, j: xf[i * 128:(i + 1) * 128, j]
    else:
        shape, pick = (R // 128, C // 128), lambda i, j: xf[i * 128:(i + 1) * 128, j * 128:(j + 1) * 128]
    s = np.empty(shape, np.float32)
    for i in range(shape[0]):
        for j in range(shape[1]):
            grp = np.abs(pick(i, j)).ravel()
            grp = grp[np.isfinite(grp)]
            v = grp[rng.integers(0, grp.size)]                  # one element of the group at |x/s| ~ fmax
            s[i, j] = np.float32(v) / fm
            s[i, j] = np.nextafter(s[i, j], np.float32(rng.choice([-1, 1]) * np.inf), dtype=np.float32) \
                if rng.random() < 0.5 else s[i, j]
            if rng.random() < 0.25:
                s[i, j] = -s[i, j]                              # |x / s| does not see the sign of s
    odd = np.float32([0.0, 1e-40, 2.0 ** -125, 2.0 ** -124, 3e37, np.inf, -0.0, np.nan, np.finfo(np.float32).max,
                      -2.0 ** -130])
    n = min(len(odd), s.size)
    s.ravel()[:n] = odd[:n]
    q = rng.integers(0, 256, size=(C, R) if gran == oracle.GRAN_128x1 else (R, C), dtype=np.uint8)
    stats = fg.new_stats()
    fg.quant_stats(dev_bf16(xb), dev_u8(q), dev_f32(s), gran, fmt, stats)
    assert_status_ok()
    ref = oracle.quant_stats(xb, q, s, gran, fmt)
    assert ref[2] > 0
    assert np.array_equal(stats.cpu().numpy().astype(np.uint64), ref), (stats, ref)


def test_quant_stats_full_size_1x128():
    xb = synth.bf16_normal((8192, 4096), 0, 1.0, 1e-3, 50.0)
    q, s, _ = oracle.quant_1x128(xb)
    stats = fg.new_stats()
    fg.quant_stats(dev_bf16(xb), dev_u8(q), dev_f32(s), fg.GRAN_1x128, fg.E4M3, stats)
    assert_status_ok()
    assert np.array_equal(stats.cpu().numpy().astype(np.uint64), oracle.quant_stats(xb, q, s, oracle.GRAN_1x128))


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
@pytest.mark.parametrize("s0", [0.0, float("inf")], ids=["zero", "inf"])
def test_delayed_zero_and_infinite_carried_scale(fmt, s0):
    """A carried-over scale of 0 (x / 0 = +-Inf saturates, 0 / 0 is NaN) or +Inf
    (every finite x / Inf is +-0): codes, monitors (the distinct codes then
    come from the key-by-key path) and the state update follow the oracle."""
    R, C = 256, 384
    xb = synth.bf16_signed_lognormal((R, C), 19, 0.0, 2.0)
    xb[:4, :7] = 0x0000
    xb[4:6, :5] = 0x8000                                        # +-0 among the values
    g = GpuDelayed(fmt)
    g.scale.fill_(s0)
    st = oracle.DelayedState(16)
    st.scale[:] = np.float32(s0)
    check_against_oracle(g, st, xb, fmt)
