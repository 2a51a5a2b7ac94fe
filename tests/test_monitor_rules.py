"""Exhaustive CPU checks of two rules the monitor kernels rely on, against the
oracle's definitions (binary32 IEEE quotients, the oracle's FP8 encoder):

- saturation without a division: |x / s| rounded to binary32 exceeds fmax
  exactly when the BF16 magnitude bits of x reach T = bits(RZ32(|s| (fmax +
  ulp(fmax) / 2))) >> 16, plus one (and x is not a NaN);
- distinct codes by code intervals: for a scale in (0, Inf) the code of |x| is
  a non-decreasing function of the BF16 magnitude over 0 .. 0x7F80, so the set
  of codes of any set of keys follows from the interval starts of the codes.

Also pins the reading that every NaN encodes as 0x7F, whatever its sign."""
import numpy as np
import pytest

import oracle

FMTS = [oracle.E4M3, oracle.E5M2]


def f32_of_bf16(bits):
    return (np.asarray(bits, np.uint32) << 16).view(np.float32)


def rz32(p: float) -> np.float32:
    """binary64 -> binary32, rounded toward zero."""
    f = np.float32(p)
    if np.isnan(f):
        return f
    if np.isinf(f) and not np.isinf(p):
        return np.float32(np.copysign(np.finfo(np.float32).max, p))
    if abs(float(f)) > abs(p):
        f = np.nextafter(f, np.float32(0.0), dtype=np.float32)
    return f


def sat_threshold(s: float, fmt: int) -> int:
    fm = oracle.fmax(fmt)
    half_ulp = float(np.spacing(np.float32(fm))) / 2.0   # binary64 from here on
    p = abs(float(s)) * (fm + half_ulp)            # at most 24 + 25 significant bits: exact in binary64
    hi = int(np.array([rz32(p)], np.float32).view(np.uint32)[0]) >> 16
    return min(hi + 1, 0x8000)


def scales(fmt, rng, n=40):
    fm = np.float32(oracle.fmax(fmt))
    out = [np.float32(v) for v in (0.0, -0.0, 1e-45, 1e-40, 2.0 ** -125, 2.0 ** -124, 1.0, 3e37,
                                   np.finfo(np.float32).max, np.inf, np.nan, -2.5)]
    for m in rng.integers(1, 0x7F80, n):             # scales that put one BF16 value at |x/s| ~ fmax
        v = f32_of_bf16([m])[0]
        s = np.float32(v / fm)
        out += [s, np.nextafter(s, np.float32(np.inf)), np.nextafter(s, np.float32(-np.inf))]
    return out


@pytest.mark.parametrize("fmt", FMTS)
def test_saturation_threshold_rule(fmt):
    rng = np.random.default_rng(11 + fmt)
    mags = np.arange(0x8000, dtype=np.uint32)
    x = f32_of_bf16(mags)
    fm = np.float32(oracle.fmax(fmt))
    with np.errstate(all="ignore"):
        for s in scales(fmt, rng):
            sat = np.abs(x / np.float32(s)) > fm
            T = sat_threshold(s, fmt)
            rule = (mags >= T) & (mags <= 0x7F80)
            assert np.array_equal(sat, rule), (s, T)


def key_fp8(c):
    c = np.asarray(c, np.uint32)
    return np.where((c & 0x7F) == 0, 0, c)


@pytest.mark.parametrize("fmt", FMTS)
def test_distinct_codes_by_intervals(fmt):
    rng = np.random.default_rng(21 + fmt)
    mags = np.arange(0x7F81, dtype=np.uint32)                        # finite magnitudes and Inf
    with np.errstate(all="ignore"):
        for s in [np.float32(v) for v in (1e-3, 0.37, 2.0 ** -120, 1e-40, 1e30, 3.4e38)] + \
                 [np.float32(oracle.fmax(fmt)) ** -1 * np.float32(v) for v in rng.uniform(0.01, 100, 6)]:
            code = oracle.fp8_encode(f32_of_bf16(mags) / s, fmt).astype(np.int64)
            assert np.all(np.diff(code) >= 0), s                      # the premise: non-decreasing
            L = np.searchsorted(code, np.arange(129), side="left")    # interval start of each code
            for density in (0.001, 0.05, 0.5):
                present = rng.random(1 << 16) < density
                present[[0x7FC1, 0xFF81]] = rng.random(2) < 0.5       # NaN keys of either sign
                keys = np.nonzero(present)[0].astype(np.uint32)
                direct = set(key_fp8(oracle.fp8_encode(f32_of_bf16(keys) / s, fmt)).tolist())
                cum = np.concatenate([[0], np.cumsum(present)])
                by_int = set()
                for sg in (0, 1):
                    base = sg << 15
                    for c in range(128):
                        if L[c] < L[c + 1] and cum[base + L[c + 1]] > cum[base + L[c]]:
                            by_int.add(int(key_fp8((sg << 7) | c)))
                    if cum[base + 0x8000] > cum[base + 0x7F81]:
                        by_int.add(0x7F)                              # NaN keys: the NaN code
                assert by_int == direct, (s, density)


@pytest.mark.parametrize("fmt", FMTS)
def test_nan_encodes_as_0x7f_either_sign(fmt):
    nan = np.array([0x7FC00000, 0xFFC00000, 0x7F800001, 0xFFFFFFFF], np.uint32).view(np.float32)
    assert np.all(oracle.fp8_encode(nan, fmt) == 0x7F)
