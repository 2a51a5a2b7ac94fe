"""The MXFP8 quantizer kernel (csrc/mx.cu) does not divide or take a
logarithm: it reads each block's scale exponent off the bits of the block's
BF16 amax.  With amax = m * 2^p (m in [1, 2)) and fmax = 1.75 * 2^emax, the
smallest e with fmax * 2^e >= amax is p - emax, plus one when m > 1.75, i.e.
when the 7 fraction bits exceed 0x60.  This checks that rule, written out
here, against the oracle's definition for every positive finite BF16 amax
(normal and subnormal) in both formats.  It checks the derivation; the
kernel itself is compared with the oracle on the GPU."""
import numpy as np
import pytest

import oracle
from oracle import mx


def exponent_from_bits(a: int, emax: int) -> int:
    ex, man = a >> 7, a & 0x7F
    if ex:
        p, frac = ex - 127, man
    else:
        msb = man.bit_length() - 1
        p, frac = msb - 133, (man << (7 - msb)) & 0x7F
    return max(-127, min(127, p - emax + (1 if frac > 0x60 else 0)))


@pytest.mark.parametrize("fmt,emax", [(oracle.E4M3, 8), (oracle.E5M2, 15)])
def test_bit_rule_equals_the_definition_for_every_bf16_amax(fmt, emax):
    bits = np.arange(1, 0x7F80, dtype=np.uint16)          # every positive finite BF16
    amax = mx._bf16_table()[bits]
    want = mx.mx_scale_exponents(amax, fmt)
    got = np.array([exponent_from_bits(int(a), emax) for a in bits], np.int64)
    assert np.array_equal(got, want)


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_definition_at_powers_of_two_and_at_the_clamps(fmt):
    """The exponent rule itself, from its definition: amax = fmax * 2^j gives
    e = j exactly, a hair above it gives j + 1, and both ends clamp to the
    UE8M0 range [-127, 127] (code 254 at the top, 0 at the bottom)."""
    fm = float(oracle.fmax(fmt))
    j = np.arange(-140, 141)
    on = np.ldexp(fm, j)
    above = on * (1.0 + 2.0 ** -40)
    assert np.array_equal(mx.mx_scale_exponents(on, fmt), np.clip(j, -127, 127))
    assert np.array_equal(mx.mx_scale_exponents(above, fmt), np.clip(j + 1, -127, 127))
    assert int(mx.mx_scale_exponents(np.float64(0.0), fmt)) == 0
