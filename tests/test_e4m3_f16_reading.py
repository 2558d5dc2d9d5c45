"""The e4m3 -> f16 operand conversion of the prompt and verify tiles: the
e4m3 bit pattern placed at f16's bit positions (sign at bit 15, the 4-bit
exponent and 3-bit mantissa at bits 13..7) reads, in f16, as the e4m3 value
times 2^-8 exactly, for every code except the two NaN codes; the kernels
take the factor 2^8 back in the score and output scales, where a power of
two changes no rounding.

The byte placement restated here is the kernel's (two bytes per 32-bit
word, lower byte in the lower half); the values it must give come from the
oracle's e4m3 decoder and numpy's float16, neither of which it uses."""

import numpy as np

from oracle import e4m3


def _placed_f16(codes: np.ndarray) -> np.ndarray:
    """f16 bit patterns: byte b at bits 8..15 of a 16-bit lane, then
    (t & 0x8000) | ((t >> 1) & 0x3F80), as the kernel does on 32-bit words."""
    words = codes.astype(np.uint32).reshape(-1, 2)
    t = (words[:, 0] << 8) | (words[:, 1] << 24)          # bytes (0, b0, 0, b1)
    f = (t & 0x80008000) | ((t >> 1) & 0x3F803F80)
    lanes = np.stack([f & 0xFFFF, f >> 16], axis=1).reshape(-1)
    return lanes.astype(np.uint16).view(np.float16)


def test_every_finite_code_reads_as_its_value_times_2_to_minus_8():
    codes = np.arange(256, dtype=np.uint8)
    got = _placed_f16(codes).astype(np.float64)
    want = e4m3.decode(codes).astype(np.float64) * 2.0 ** -8
    finite = np.isfinite(want)
    assert finite.sum() == 254                              # S.1111.111 are the NaNs
    np.testing.assert_array_equal(got[finite], want[finite])
    assert np.array_equal(np.signbit(got[finite]), np.signbit(want[finite]))   # -0 stays -0


def test_pairs_keep_their_order_in_a_word():
    codes = np.array([0x38, 0xB8, 0x01, 0x7E], np.uint8)     # 1, -1, 2^-9, 448
    got = _placed_f16(codes).astype(np.float64)
    np.testing.assert_array_equal(got, np.array([1.0, -1.0, 2.0 ** -9, 448.0]) * 2.0 ** -8)
