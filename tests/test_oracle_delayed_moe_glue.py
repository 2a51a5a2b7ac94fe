"""Pins for the oracle's per-tensor delayed-scaling state machine, MoE routing
with the padded routing map, and the SwiGLU glue.

Independent references: the hand-worked delayed sequence (tests/golden), the
checkpoint-split invariant, numpy's stable argsort and scipy's softmax for the
router, brute-force re-derivation of the padding rule, and torch autograd for
the SwiGLU derivative.
"""
import json
import os
from fractions import Fraction

import numpy as np
import pytest
import scipy.special
import torch

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def tensor_with_amax(a, seed):
    x = synth.bf16_normal((128, 256), seed, 1.0)
    xv = synth.bf16_bits_to_f32(x)
    xv = np.clip(xv, -a / 2, a / 2) if a > 0 else np.zeros_like(xv)
    xv[5, 7] = -a
    return synth.f32_to_bf16_bits(xv)


def test_hand_delayed_sequence():
    g = json.load(open(os.path.join(GOLD, "hand_delayed_sequence.json")))
    st = oracle.DelayedState(g["history_len"])
    used = []
    for t, a in enumerate(g["amax_per_step"]):
        x = tensor_with_amax(a, t)
        q, s_used, stats, code = oracle.delayed_step(x, st, oracle.E4M3, g["margin"])
        assert code == oracle.OK
        used.append(s_used)
        # the quantization used exactly the scale in force before the step
        xv = synth.bf16_bits_to_f32(x)
        assert np.array_equal(q, oracle.fp8_encode(xv / np.float32(s_used), oracle.E4M3))
        # the history window after the step, slot by slot
        assert st.hist.tolist() == g["expected_history_after_each_step"][t]
    ev = lambda e: float(np.float32(Fraction(e)) if "/" not in e else
                         np.float32(np.float32(float(e.split('/')[0])) / np.float32(448.0)))
    assert used == [ev(e) for e in g["expected_scale_used_per_step"]]
    assert float(st.scale[0]) == ev(g["expected_scale_after_last_step"])
    assert int(st.step[0]) == 5


def test_all_zero_history_keeps_the_scale():
    """Reading R5's degenerate case: while every amax in the window is 0 the
    scale in force is kept (here the initial 1), and the first nonzero amax
    sets it from the window's maximum."""
    st = oracle.DelayedState(4)
    zero = np.zeros((128, 256), np.uint16)
    for t in range(3):
        q, s_used, _, code = oracle.delayed_step(zero, st, oracle.E4M3)
        assert code == oracle.OK and s_used == 1.0 and float(st.scale[0]) == 1.0
        assert not q.any()
    oracle.delayed_step(tensor_with_amax(8.0, 3), st, oracle.E4M3)
    assert float(st.scale[0]) == np.float32(np.float32(8.0) / np.float32(448.0))


def test_delayed_knobs_margin_and_most_recent():
    st = oracle.DelayedState(4)
    for t, a in enumerate([8.0, 2.0]):
        oracle.delayed_step(tensor_with_amax(a, t), st, oracle.E4M3, margin=2)
    assert float(st.scale[0]) == np.float32(np.float32(8.0 * 4) / np.float32(448.0))
    st2 = oracle.DelayedState(4)
    for t, a in enumerate([8.0, 2.0]):
        oracle.delayed_step(tensor_with_amax(a, t), st2, oracle.E5M2, algo=oracle.ALGO_MOST_RECENT)
    assert float(st2.scale[0]) == np.float32(np.float32(2.0) / np.float32(57344.0))


def test_checkpoint_split_invariant():
    steps = 12
    xs = [synth.bf16_signed_lognormal((128, 384), t, 0.0, 1.5, 1.5 ** (t // 4)) for t in range(steps)]
    a = oracle.DelayedState(16)
    qa = [oracle.delayed_step(x, a, oracle.E4M3)[0] for x in xs]
    b = oracle.DelayedState(16)
    qb = [oracle.delayed_step(x, b, oracle.E4M3)[0] for x in xs[:5]]
    c = b.copy()                                # "checkpoint" into fresh buffers
    qb += [oracle.delayed_step(x, c, oracle.E4M3)[0] for x in xs[5:]]
    assert all(np.array_equal(u, v) for u, v in zip(qa, qb))
    assert np.array_equal(a.hist, c.hist) and a.scale[0] == c.scale[0] and a.step[0] == c.step[0]


def test_nonfinite_step_leaves_state_unchanged():
    st = oracle.DelayedState(4)
    oracle.delayed_step(tensor_with_amax(3.0, 0), st, oracle.E4M3)
    before = st.copy()
    x = tensor_with_amax(5.0, 1)
    x[0, 0] = 0x7FC0                      # NaN
    _, _, _, code = oracle.delayed_step(x, st, oracle.E4M3)
    assert code == oracle.NONFINITE
    assert np.array_equal(st.hist, before.hist) and st.scale[0] == before.scale[0] and st.step[0] == before.step[0]


def test_drift_saturates_then_recovers():
    # the scale is one step late: a x1.5 jump saturates the elements above the
    # old amax / 1.5 once, and the next step (same magnitude) saturates nothing
    x0 = synth.bf16_normal((128, 256), 0, 1.0)
    v0 = synth.bf16_bits_to_f32(x0)
    x1 = synth.f32_to_bf16_bits(v0 * np.float32(1.5))
    st = oracle.DelayedState(16)
    sat = [int(oracle.delayed_step(x, st, oracle.E4M3)[2][2]) for x in (x0, x1, x1)]
    s1 = np.float32(np.abs(v0).max()) / np.float32(448.0)
    v1 = synth.bf16_bits_to_f32(x1)
    expect = int(np.count_nonzero(np.abs(v1 / s1) > np.float32(448.0)))
    assert expect > 10 and sat[1] == expect and sat[2] == 0


# ------------------------------------------------------------------- routing

def small_logits(T=512, E=16, seed=5):
    z = synth.f32_normal((T, E), seed)
    z[3, :] = 0.25          # a row of exact ties
    z[4, 2] = z[4, E - 1]   # a single tie
    return z


def test_topk_matches_stable_argsort_and_softmax():
    z = small_logits()
    r = oracle.moe_route(z, topk=4, align=8)
    ref = np.argsort(-z, axis=1, kind="stable")[:, :4]
    assert np.array_equal(r["topk_idx"], ref)
    p = scipy.special.softmax(z.astype(np.float64), axis=1)
    assert np.allclose(r["topk_prob"], np.take_along_axis(p, ref, 1), rtol=1e-13, atol=0)


@pytest.mark.parametrize("align", [1, 8, 128])
def test_padding_rule_bruteforce(align):
    z = small_logits(T=1024, E=16)
    topk = 4
    r = oracle.moe_route(z, topk=topk, align=align)
    T, E = z.shape
    routed = np.zeros((T, E), bool)
    np.put_along_axis(routed, np.argsort(-z, axis=1, kind="stable")[:, :topk], True, 1)
    counts = routed.sum(0)
    assert np.array_equal(r["counts"], counts)
    padded = -(-counts // align) * align
    assert np.array_equal(r["padded"], padded)
    assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(padded)]))
    for e in range(E):
        lo, hi = r["offsets"][e], r["offsets"][e + 1]
        toks = r["row_token"][lo:hi]
        assert np.all(np.diff(toks) > 0)                      # ascending, no repeats
        free = np.nonzero(~routed[:, e])[0][: padded[e] - counts[e]]
        expect = np.sort(np.concatenate([np.nonzero(routed[:, e])[0], free]))
        assert np.array_equal(toks, expect)
        ispad = r["row_is_pad"][lo:hi].astype(bool)
        assert np.array_equal(ispad, ~routed[toks, e])
        assert np.all(r["row_prob"][lo:hi][ispad] == 0.0)
    assert r["total"] == int(padded.sum())


def test_quantize_then_gather_equals_gather_then_quantize():
    T, K = 512, 256
    x = synth.bf16_normal((T, K), 2, 1.0, 1e-3, 50.0)
    r = oracle.moe_route(small_logits(T=T, E=16), topk=4, align=128)
    q, s, _ = oracle.quant_1x128(x, oracle.E4M3)
    qg, sg = oracle.moe_gather(q, s, r["row_token"], r["total"], r["cap"])
    tot = r["total"]
    q2, s2, _ = oracle.quant_1x128(x[r["row_token"][:tot]], oracle.E4M3)
    assert np.array_equal(qg[:tot], q2)
    assert np.array_equal(sg[:, :tot], s2)


def test_padding_is_mathematically_equivalent_for_real_rows():
    T, K, N, E = 512, 256, 256, 8
    x = synth.bf16_normal((T, K), 3, 1.0, 1e-3, 50.0)
    r = oracle.moe_route(small_logits(T=T, E=E, seed=8), topk=2, align=128)
    q, s, _ = oracle.quant_1x128(x, oracle.E4M3)
    qg, sg = oracle.moe_gather(q, s, r["row_token"], r["total"], r["cap"])
    w = synth.bf16_normal((E * N, K), 4, 0.02).reshape(E, N, K)
    qw = np.empty((E, N, K), np.uint8)
    sw = np.empty((E, N // 128, K // 128), np.float32)
    for e in range(E):
        qw[e], sw[e], _ = oracle.quant_128x128(w[e])
    pm, pn = np.meshgrid(np.arange(r["total"]), np.arange(N), indexing="ij")
    padded_out = oracle.grouped_gemm_points(r["offsets"], qg, sg, r["cap"], qw, sw,
                                            pm.ravel(), pn.ravel()).reshape(-1, N)
    for e in range(E):
        lo, hi = r["offsets"][e], r["offsets"][e + 1]
        real = ~r["row_is_pad"][lo:hi].astype(bool)
        toks = r["row_token"][lo:hi][real]
        if len(toks) == 0:
            continue
        # the unpadded expert GEMM on the same FP8 bytes and scales
        qa = q[toks]
        sa = np.ascontiguousarray(s[:, toks])
        ref = oracle.gemm_full(qa, oracle.E4M3, sa, oracle.GRAN_1x128, qw[e], oracle.E4M3, sw[e],
                               oracle.GRAN_128x128)
        assert np.array_equal(padded_out[lo:hi][real], ref)


# ------------------------------------------------------------------- SwiGLU

def test_swiglu_forward_and_backward_against_torch_autograd():
    R, F = 64, 256
    gu = synth.bf16_normal((R, 2 * F), 9, 2.0)
    dh = synth.bf16_normal((R, F), 10, 1.0)
    g = torch.from_numpy(synth.bf16_bits_to_f32(gu[:, :F]).astype(np.float64)).requires_grad_()
    u = torch.from_numpy(synth.bf16_bits_to_f32(gu[:, F:]).astype(np.float64)).requires_grad_()
    h = torch.nn.functional.silu(g) * u
    h.backward(torch.from_numpy(synth.bf16_bits_to_f32(dh).astype(np.float64)))
    ours = synth.bf16_bits_to_f32(oracle.swiglu_fwd(gu)).astype(np.float64)
    ulp = lambda v: np.maximum(np.abs(v), 1e-30) * 2.0 ** -8
    ref = h.detach().numpy()
    assert np.all(np.abs(ours - ref) <= ulp(ref) * 1.0001)
    dgu = synth.bf16_bits_to_f32(oracle.swiglu_bwd(gu, dh)).astype(np.float64)
    for got, want in ((dgu[:, :F], g.grad.numpy()), (dgu[:, F:], u.grad.numpy())):
        assert np.all(np.abs(got - want) <= ulp(want) * 1.0001)
