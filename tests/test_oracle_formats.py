"""Pins for the oracle's number formats (BF16 decode, FP8 E4M3/E5M2 decode and
encode, FP64 -> BF16 rounding), checked against things other than the oracle:

* PyTorch's own float8_e4m3fn / float8_e5m2 / bfloat16 conversions (an
  independent library implementation of the same IEEE-style formats);
* values the pages print: E4M3 has 4 exponent and 3 mantissa bits and spans
  [-448, 448] ("FP8-LM: Training FP8 Large Language Models", "FP8 data
  formats"; FP8-RL article, "dynamic weight sync"; "FP8 training
  infrastructure" guide, "numeric precision landscape"); E5M2 has 5 exponent
  and 2 mantissa bits;
* hand-worked rounding midpoints.
"""
import numpy as np
import pytest
import torch

import oracle

TORCH_FP8 = {oracle.E4M3: torch.float8_e4m3fn, oracle.E5M2: torch.float8_e5m2}


def torch_decode(fmt):
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    return codes.view(TORCH_FP8[fmt]).to(torch.float64).numpy()


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_decode_all_codes_match_torch(fmt):
    ours = oracle.fp8_decode_table(fmt)
    ref = torch_decode(fmt)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    assert np.all((ours == ref) | both_nan)


def test_decode_page_values():
    # E4M3 range [-448, 448]; 4-bit exponent, 3-bit mantissa.
    t = oracle.fp8_decode_table(oracle.E4M3)
    finite = t[np.isfinite(t)]
    assert finite.max() == 448.0 and finite.min() == -448.0
    assert t[0x7E] == 448.0 and t[0xFE] == -448.0
    assert t[0x38] == 1.0            # exponent field 7 = bias, mantissa 0
    assert t[0x01] == 2.0 ** -9      # smallest subnormal: 2^(1-7-3)
    assert np.isnan(t[0x7F]) and np.isnan(t[0xFF])
    # 3 mantissa bits: 8 codes per binade between 1 and 2
    assert np.count_nonzero((finite >= 1.0) & (finite < 2.0)) == 8
    # E5M2: 5-bit exponent, 2-bit mantissa; max finite 57344, inf codes
    u = oracle.fp8_decode_table(oracle.E5M2)
    assert u[0x7B] == 57344.0 and u[0x3C] == 1.0 and u[0x01] == 2.0 ** -16
    assert np.isinf(u[0x7C]) and np.isnan(u[0x7D])
    fin = u[np.isfinite(u)]
    assert np.count_nonzero((fin >= 1.0) & (fin < 2.0)) == 4
    assert oracle.fmax(oracle.E4M3) == 448.0 and oracle.fmax(oracle.E5M2) == 57344.0


def test_encode_midpoints_by_hand():
    e = lambda v: int(oracle.fp8_encode(np.array([v], np.float32), oracle.E4M3)[0])
    assert e(2.0 ** -10) == 0x00          # half the smallest subnormal: tie -> even (0)
    assert e(3 * 2.0 ** -10) == 0x02      # 1.5 subnormal steps: tie -> even (2)
    assert e(2.0 ** -10 * 1.0000001) == 0x01
    assert e(464.0) == 0x7E               # beyond max: saturates
    assert e(1e30) == 0x7E and e(-1e30) == 0xFE
    assert e(float("inf")) == 0x7E
    assert e(0.150390625) == 0x22         # 1.203125 * 2^-3 -> 1.25 * 2^-3
    assert e(-0.0) == 0x80 and e(0.0) == 0x00
    assert e(-0.5) == 0xB0
    f = lambda v: int(oracle.fp8_encode(np.array([v], np.float32), oracle.E5M2)[0])
    assert f(57344.0) == 0x7B and f(60000.0) == 0x7B and f(1e9) == 0x7B
    assert f(2.0 ** -17) == 0x00 and f(3 * 2.0 ** -17) == 0x02
    assert f(1.125) == 0x3C               # tie between 1.0 and 1.25 -> even mantissa (1.0)
    assert f(1.375) == 0x3E               # tie between 1.25 and 1.5 -> even (1.5)


@pytest.mark.slow
@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_exhaustive_in_range_matches_torch(fmt):
    """Every non-negative binary32 below fmax: oracle == torch's RNE conversion;
    the negative patterns mirror them with the sign bit."""
    top = np.frombuffer(np.float32(oracle.fmax(fmt)).tobytes(), np.uint32)[0]
    chunk = 1 << 25
    first = 0
    bad = 0
    while first < top:
        n = int(min(chunk, top - first))
        ours = oracle.fp8_encode_bits_range(int(first), n, fmt)
        vals = torch.from_numpy(np.arange(first, first + n, dtype=np.uint32).view(np.float32))
        ref = vals.to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
        bad += int(np.count_nonzero(ours != ref))
        if first == 0 or (first // chunk) % 7 == 3:
            neg = oracle.fp8_encode_bits_range(int(first) | 0x80000000, n, fmt)
            assert np.array_equal(neg, ours | 0x80)
        first += n
    assert bad == 0


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_encode_saturates_at_and_beyond_max(fmt):
    fm = oracle.fmax(fmt)
    maxcode = {oracle.E4M3: 0x7E, oracle.E5M2: 0x7B}[fmt]
    start = int(np.frombuffer(np.float32(fm).tobytes(), np.uint32)[0])
    n = 0x7F800000 - start + 1            # fmax .. +inf inclusive
    step = 97
    bits = np.arange(start, start + n, step, dtype=np.int64).astype(np.uint32)
    codes = oracle.fp8_encode(bits.view(np.float32), fmt)
    assert np.all(codes == maxcode)
    assert np.all(oracle.fp8_encode(-bits.view(np.float32), fmt) == (maxcode | 0x80))


def test_bf16_decode_all_patterns_match_torch():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ours = oracle.bf16_to_f32(bits)
    ref = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).to(torch.float32).numpy()
    # NaN payloads are quieted by the float return through ctypes; compare NaN-ness there.
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(ours), nan) and nan.sum() == 2 * 127
    assert np.array_equal(ours.view(np.uint32)[~nan], ref.view(np.uint32)[~nan])


def test_f64_to_bf16_matches_torch_on_binary32_values_and_single_rounding():
    rng = np.random.default_rng(1)
    v = (rng.standard_normal(4096) * np.exp(rng.uniform(-60, 60, 4096))).astype(np.float32)
    v = np.concatenate([v, np.float32([0.0, -0.0, 1.0, 3e38, 1e-40, -2.5e-39])])
    ours = oracle.f64_to_bf16(v.astype(np.float64))
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    # A double just above a BF16 midpoint whose binary32 rounding lands on the
    # midpoint: a single rounding goes up (1 + 2^-7), a double rounding would tie to 1.0.
    x = 1.0 + 2.0 ** -8 + 2.0 ** -40
    assert int(oracle.f64_to_bf16([x])[0]) == 0x3F81
    assert int(oracle.f64_to_bf16([1.0 + 2.0 ** -8])[0]) == 0x3F80
    assert int(oracle.f64_to_bf16([1.0 + 3 * 2.0 ** -8])[0]) == 0x3F82   # tie above an odd mantissa


def test_f64_to_bf16_every_exact_tie_matches_torch():
    """Every value exactly halfway between two neighbouring BF16 numbers (the
    binary32 pattern of the lower one with 0x8000 in its low half), both
    signs, subnormal and normal, up to the tie between the largest finite
    BF16 and infinity: ties go to the even mantissa."""
    u = np.arange(0, 0x7F80, dtype=np.uint32)
    ties = ((u << 16) | 0x8000).view(np.float32)
    ties = np.concatenate([ties, -ties])
    ours = oracle.f64_to_bf16(ties.astype(np.float64))
    ref = torch.from_numpy(ties).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
