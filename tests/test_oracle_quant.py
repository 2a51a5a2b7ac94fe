"""Pins for the oracle's quantizers (1x128 tiles, the transposed 128x1 copy,
128x128 blocks, the FP8 transpose) and its monitors.

Independent evidence used: hand-worked examples (tests/golden), numpy
recounts, the scaling invariance x -> 2x, the per-element error bound of
round-to-nearest FP8, and identities between layouts.
"""
import json
import os

import numpy as np
import pytest

import oracle
import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as f:
        return json.load(f)


def bits_of(values):
    return synth.f32_to_bf16_bits(np.asarray(values, np.float32))


# ---------------------------------------------------------------- hand examples

def hand_tile():
    g = load("hand_1x128_tile.json")
    x = np.zeros((1, 128), np.uint16)
    for k, b in g["tile_bf16_first_values"].items():
        x[0, int(k)] = int(b, 16)
    return g, x


def test_hand_tile_inputs_are_the_stated_values():
    g, x = hand_tile()
    vals = synth.bf16_bits_to_f32(x[0])
    for k, v in g["tile_real_values"].items():
        assert float(vals[int(k)]) == v


def test_hand_tile_1x128():
    g, x = hand_tile()
    q, s, st = oracle.quant_1x128(x, oracle.E4M3)
    assert st == oracle.OK
    assert s.shape == (1, 1) and float(s[0, 0]) == g["expected_scale"]
    for k, c in g["expected_codes"].items():
        assert int(q[0, int(k)]) == int(c, 16)
    assert np.all(q[0, 4:] == int(g["expected_rest_code"], 16))
    stats = oracle.quant_stats(x, q, s, oracle.GRAN_1x128, oracle.E4M3)
    e = g["expected_stats"]
    assert list(map(int, stats)) == [e["nonzero"], e["underflow"], e["saturated"],
                                     e["distinct_in"], e["distinct_out"]]


def test_hand_block_128x128():
    g = load("hand_128x128_block.json")
    w = np.full((128, 128), 0.5, np.float32)
    w[37, 101] = 7.0
    q, s, st = oracle.quant_128x128(bits_of(w), oracle.E4M3)
    assert st == oracle.OK
    assert float(s[0, 0]) == g["expected_scale"]
    assert q[37, 101] == int(g["expected_code_of_7"], 16)
    mask = np.ones_like(q, bool)
    mask[37, 101] = False
    assert np.all(q[mask] == int(g["expected_code_of_0.5"], 16))


# ---------------------------------------------------------------- invariants

def random_bits(shape, seed, std=1.0, outliers=True):
    return synth.bf16_normal(shape, seed, std, 1e-3 if outliers else 0.0, 50.0)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_scaling_invariance_1x128(fmt):
    x = random_bits((64, 512), 3)
    x2 = bits_of(synth.bf16_bits_to_f32(x) * 2.0)   # exact in BF16
    q, s, _ = oracle.quant_1x128(x, fmt)
    q2, s2, _ = oracle.quant_1x128(x2, fmt)
    assert np.array_equal(q, q2)
    assert np.array_equal(s * 2.0, s2)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_roundtrip_error_bound(fmt):
    """|dec(q)*s - x| <= half a code spacing at x/s (round to nearest), in units of s."""
    x = random_bits((256, 1024), 5)
    q, s, _ = oracle.quant_1x128(x, fmt)
    xv = synth.bf16_bits_to_f32(x).astype(np.float64)
    sv = np.repeat(s.T, 128, axis=1).astype(np.float64)          # [R, C]
    dec = oracle.fp8_decode_table(fmt)[q]
    t = np.abs(xv / sv)
    mbits, emin = (3, -6) if fmt == oracle.E4M3 else (2, -14)
    e = np.floor(np.log2(np.maximum(t, 2.0 ** emin)))
    half_spacing = 2.0 ** (e - mbits - 1)
    # the binary32 quotient adds at most one binary32 ulp of t
    err = np.abs(dec - xv / sv)
    assert np.all(err <= half_spacing * (1 + 2 ** -20) + t * 2 ** -23)
    # the tile maximum lands exactly on fmax (|x| = amax -> fmax up to binary32 rounding)
    amax_code = np.max(np.abs(dec.reshape(256, 8, 128)), axis=2)
    assert np.all(amax_code == oracle.fmax(fmt))


def test_layout_markers_1x128_and_128x128():
    # every 1x128 tile / 128x128 block carries a distinct power-of-two marker,
    # so a mixed-up scale layout changes the scale read back at that position
    R, C = 256, 512
    x = np.ones((R, C), np.float32)
    ex = lambda r, cb: (r * 4 + cb) % 24
    for r in range(R):
        for cb in range(C // 128):
            x[r, cb * 128 + 5] = 448.0 * 2.0 ** ex(r, cb)
    q, s, _ = oracle.quant_1x128(bits_of(x), oracle.E4M3)
    assert s.shape == (C // 128, R)
    for r in range(R):
        for cb in range(C // 128):
            assert s[cb, r] == 2.0 ** ex(r, cb)
            assert q[r, cb * 128 + 5] == 0x7E
    w = np.ones((R, C), np.float32)
    for rb in range(R // 128):
        for cb in range(C // 128):
            w[rb * 128 + 3, cb * 128 + 7] = 448.0 * 2.0 ** (rb * 4 + cb)
    q2, s2, _ = oracle.quant_128x128(bits_of(w), oracle.E4M3)
    assert s2.shape == (2, 4)
    for rb in range(2):
        for cb in range(4):
            assert s2[rb, cb] == 2.0 ** (rb * 4 + cb)


def test_transposed_copy_is_row_quant_of_transpose():
    x = random_bits((384, 256), 9)
    qT, sT, st = oracle.quant_128x1_transposed(x, oracle.E4M3)
    assert st == oracle.OK
    q_ref, s_ref, _ = oracle.quant_1x128(np.ascontiguousarray(x.T), oracle.E4M3)
    assert np.array_equal(qT, q_ref)
    assert np.array_equal(sT, s_ref)


def test_transposed_equals_transpose_on_blockwise_constant_magnitude():
    # |x| constant within each 128x128 block: row and column groups share amax,
    # so the 128x1 copy is exactly the byte transpose of the 1x128 quantization.
    R, C = 256, 384
    rng = np.random.default_rng(0)
    mags = 2.0 ** rng.integers(-8, 8, size=(R // 128, C // 128))
    x = np.repeat(np.repeat(mags, 128, 0), 128, 1) * rng.choice([-1.0, 1.0], size=(R, C))
    xb = bits_of(x)
    q, s, _ = oracle.quant_1x128(xb, oracle.E4M3)
    qT, sT, _ = oracle.quant_128x1_transposed(xb, oracle.E4M3)
    assert np.array_equal(qT, q.T)
    assert np.array_equal(oracle.fp8_transpose(q), q.T)


def test_fp8_transpose_and_scale_grid():
    w = random_bits((256, 384), 11, 0.02, False)
    q, s, _ = oracle.quant_128x128(w, oracle.E4M3)
    qT = oracle.fp8_transpose(q)
    sT = oracle.scale_grid_transpose(s)
    assert np.array_equal(qT, q.T) and np.array_equal(sT, s.T)
    # 128x128 quantization commutes with transposition
    q2, s2, _ = oracle.quant_128x128(np.ascontiguousarray(w.T), oracle.E4M3)
    assert np.array_equal(q2, qT) and np.array_equal(s2, sT)


def test_zero_tile_and_nonfinite():
    x = np.zeros((2, 256), np.uint16)
    x[1, 0] = 0x8000   # -0
    q, s, st = oracle.quant_1x128(x, oracle.E4M3)
    assert st == oracle.OK and np.all(s == 1.0)
    assert q[1, 0] == 0x80 and np.all(q[0] == 0)
    x[1, 200] = 0x7F80  # +inf
    _, _, st = oracle.quant_1x128(x, oracle.E4M3)
    assert st == oracle.NONFINITE


def test_subnormal_scale_kept():
    # amax = smallest BF16 subnormal: s = amax / 448 is a binary32 subnormal (no FTZ)
    x = np.zeros((1, 128), np.uint16)
    x[0, 0] = 0x0001
    q, s, st = oracle.quant_1x128(x, oracle.E4M3)
    tiny = np.float32(synth.bf16_bits_to_f32(np.uint16(1)))
    assert st == oracle.OK
    assert s[0, 0] == np.float32(tiny / np.float32(448.0)) and 0 < s[0, 0] < np.finfo(np.float32).tiny
    # the quotient amax / s is >= 448 here because s was rounded down
    assert q[0, 0] == 0x7E


# ------------------------------------------- the scale and the quotient, exactly
#
# R2 and R3 fix s = fp32(amax / fmax) and q = enc(fp32(x / s)): two IEEE
# binary32 divisions.  The references below take each quotient of two binary32
# numbers in binary64 and round it once to binary32.  That is the correctly
# rounded binary32 quotient: the binary64 result carries 53 >= 2 * 24 + 2 bits,
# so the second rounding cannot move it (S. A. Figueroa, "When is double
# rounding innocuous?", SIGNUM Newsletter 30(3), 1995).  The FP8 step is torch's
# float8 cast, itself pinned against the oracle's encoder in
# test_oracle_formats.py.  Multiplying by a rounded reciprocal instead of
# dividing changes the scale of some BF16 amax values and, for about a fifth of
# the amax values below, the code of some x.

_FMAX = {oracle.E4M3: 448.0, oracle.E5M2: 57344.0}
_POS_BF16 = np.arange(1, 0x7F80, dtype=np.uint32)            # every positive finite BF16


def _bf16_values(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_scale_of_every_bf16_amax_is_the_rounded_quotient(fmt):
    x = np.zeros((len(_POS_BF16), 128), np.uint16)
    x[:, 0] = _POS_BF16
    x[:, 77] = _POS_BF16 ^ 0x8000           # the same magnitude with the other sign
    _, s, st = oracle.quant_1x128(x, fmt)
    assert st == oracle.OK
    want = (_bf16_values(_POS_BF16).astype(np.float64) / _FMAX[fmt]).astype(np.float32)
    assert np.array_equal(s[0], want)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_codes_are_the_cast_of_the_rounded_quotient(fmt):
    torch = pytest.importorskip("torch")
    tdt = torch.float8_e4m3fn if fmt == oracle.E4M3 else torch.float8_e5m2
    vals = _bf16_values(_POS_BF16)
    rng = np.random.default_rng(29)
    amax_bits = _POS_BF16[rng.integers(0x0800, len(_POS_BF16), 64)]   # scales in the normal range
    rows = []
    for a in amax_bits:
        xs = _POS_BF16[vals <= _bf16_values(a)]
        xs = np.where(rng.integers(0, 2, len(xs)) == 1, xs | 0x8000, xs)   # both signs
        n_t = (len(xs) + 126) // 127
        body = np.resize(xs, n_t * 127).reshape(n_t, 127)
        rows.append(np.concatenate([np.full((n_t, 1), a, np.uint32), body], axis=1))
    x = np.concatenate(rows).astype(np.uint16)
    q, s, st = oracle.quant_1x128(x, fmt)
    assert st == oracle.OK
    quot = (synth.bf16_bits_to_f32(x).astype(np.float64) / s[0].astype(np.float64)[:, None]).astype(np.float32)
    want = torch.from_numpy(quot).to(tdt).view(torch.uint8).numpy()
    assert np.array_equal(q, want)


# ---------------------------------------------------------------- monitors

def numpy_counts(xg, qg, sg, fm):
    """xg: [G, n] bf16 bits, qg: [G, n] codes, sg: [G] scales."""
    xv = synth.bf16_bits_to_f32(xg)
    nz = int(np.count_nonzero(xv != 0))
    uf = int(np.count_nonzero((xv != 0) & ((qg & 0x7F) == 0)))
    quot = xv / sg[:, None].astype(np.float32)
    sat = int(np.count_nonzero(np.abs(quot) > np.float32(fm)))
    kx = np.where((xg & 0x7FFF) == 0, 0, xg)
    kq = np.where((qg & 0x7F) == 0, 0, qg)
    din = sum(len(np.unique(r)) for r in kx)
    dout = sum(len(np.unique(r)) for r in kq)
    return [nz, uf, sat, din, dout]


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_stats_match_numpy_recount_all_granularities(fmt):
    R, C = 256, 384
    # coarse values so that repeats and underflow both occur
    x = synth.bf16_signed_lognormal((R, C), 4, -2.0, 3.0)
    x[0, :64] = 0
    x[1, :7] = 0x8000
    fm = oracle.fmax(fmt)

    q, s, _ = oracle.quant_1x128(x, fmt)
    got = oracle.quant_stats(x, q, s, oracle.GRAN_1x128, fmt)
    xg = x.reshape(R, C // 128, 128).reshape(-1, 128)
    qg = q.reshape(R, C // 128, 128).reshape(-1, 128)
    sg = s.T.reshape(-1)
    assert list(map(int, got)) == numpy_counts(xg, qg, sg, fm)

    qb, sb, _ = oracle.quant_128x128(x, fmt)
    got = oracle.quant_stats(x, qb, sb, oracle.GRAN_128x128, fmt)
    blk = lambda a: a.reshape(R // 128, 128, C // 128, 128).transpose(0, 2, 1, 3).reshape(-1, 128 * 128)
    assert list(map(int, got)) == numpy_counts(blk(x), blk(qb), sb.reshape(-1), fm)

    qT, sT, _ = oracle.quant_128x1_transposed(x, fmt)
    got = oracle.quant_stats(x, qT, sT, oracle.GRAN_128x1, fmt)
    colg = lambda a: a.reshape(R // 128, 128, C).transpose(0, 2, 1).reshape(-1, 128)
    assert list(map(int, got)) == numpy_counts(colg(x), colg(np.ascontiguousarray(qT.T)),
                                               sT.reshape(-1), fm)

    st = oracle.DelayedState()
    st.scale[0] = 0.01
    qt, used, stats, code = oracle.delayed_step(x, st, fmt)
    assert code == oracle.OK and used == np.float32(0.01)
    assert list(map(int, stats)) == numpy_counts(x.reshape(1, -1), qt.reshape(1, -1),
                                                 np.float32([used]), fm)


def test_pertensor_current_reduces_to_the_tile_and_block_quantizers():
    """Per-tensor current scaling of a tensor that is one 1x128 tile (or one 128x128
    block) is that tile's (block's) quantization; scaling x by 2 doubles s and keeps
    the codes; an all-zero tensor gets s = 1 and zero codes."""
    for fmt in (oracle.E4M3, oracle.E5M2):
        t = synth.bf16_normal((1, 128), 51, 1.0, 0.01, 30.0)
        q, s, st = oracle.quant_pertensor_current(t, fmt)
        q1, s1, _ = oracle.quant_1x128(t, fmt)
        assert st == oracle.OK and np.array_equal(q, q1) and np.float32(s) == s1.ravel()[0]
        b = synth.bf16_normal((128, 128), 52, 1.0, 0.01, 30.0)
        q, s, _ = oracle.quant_pertensor_current(b, fmt)
        q2, s2, _ = oracle.quant_128x128(b, fmt)
        assert np.array_equal(q, q2) and np.float32(s) == s2.ravel()[0]
        x = synth.bf16_normal((300, 256), 53, 1e-2, 0.001, 100.0)
        x2 = (x.astype(np.uint32) + (1 << 7)).astype(np.uint16)        # exponent + 1: x * 2 (no overflow here)
        qa, sa, _ = oracle.quant_pertensor_current(x, fmt)
        qb, sb, _ = oracle.quant_pertensor_current(x2, fmt)
        assert np.array_equal(qa, qb) and np.float32(sb) == np.float32(2 * sa)
        qz, sz, _ = oracle.quant_pertensor_current(np.zeros((3, 128), np.uint16), fmt)
        assert sz == 1.0 and not qz.any()
