"""The split of a Q row into two e4m3 rows used by the verify tiles on e4m3
caches: with the row scaled by a power of two so that its largest magnitude
lies in [2^7, 2^8), hi = e4m3(x) and lo = e4m3(x - hi) (round to nearest
even) give hi + lo == x exactly for every bf16 value x of magnitude 2^-2 or
more, and within half of e4m3's smallest step (2^-10) below that.

This checks the arithmetic claim the kernel rests on, with torch's own e4m3
rounding: every bf16 magnitude in the scaled range, both signs."""

import numpy as np
import pytest
import torch

pytestmark = pytest.mark.skipif(not hasattr(torch, "float8_e4m3fn"), reason="no e4m3 dtype")


def _bf16_values(lo_exp, hi_exp):
    # every bf16 value with exponent in [lo_exp, hi_exp), both signs
    bits = []
    for e in range(lo_exp, hi_exp):
        for m in range(128):
            bits.append(((e + 127) << 7) | m)
    b = np.array(bits, np.uint32) << 16
    pos = b.view(np.float32)
    return torch.from_numpy(np.concatenate([pos, -pos]))


def _split(x):
    hi = x.to(torch.float8_e4m3fn).to(torch.float32)
    rest = x - hi
    lo = rest.to(torch.float8_e4m3fn).to(torch.float32)
    return hi, rest, lo


def test_remainder_is_exact_in_float32():
    x = _bf16_values(-12, 8)
    hi, rest, _ = _split(x)
    # float64 difference equals the float32 one: no rounding in x - hi
    assert torch.equal(rest.double(), x.double() - hi.double())
    assert float(hi.abs().max()) <= 256.0


def test_hi_plus_lo_exact_within_2_pow_9_of_the_largest():
    x = _bf16_values(-2, 8)
    hi, _, lo = _split(x)
    assert torch.equal(hi + lo, x)


def test_small_elements_within_half_the_smallest_e4m3_step():
    x = _bf16_values(-12, -2)
    hi, _, lo = _split(x)
    err = (hi + lo - x).abs()
    assert float(err.max()) <= 2.0 ** -10
    # and some of them do lose bits: the bound above is not vacuous
    assert float(err.max()) > 0.0
