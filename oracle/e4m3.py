"""OCP FP8 E4M3 ("fn" variant) codec, written from the format's definition.

Test infrastructure only (see the package docstring).

The pages say the caches may be fp8 (TensorFold PR #1373, "What changes":
"fp8 caches"; PR #2011 "Receipt": "bf16 and fp8 KV cache") but never name the
format.  The reading taken: E4M3 with
  * 1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
  * exponent field 0 is subnormal: value = (-1)^s * 2^-6 * m/8;
  * exponent field 1..15 is normal: value = (-1)^s * 2^(e-7) * (1 + m/8);
  * no infinities; S.1111.111 is NaN; the largest finite magnitude is 448.
Encoding (the KV write) rounds to nearest, ties to even, and saturates: any
magnitude above 448 (infinity included) becomes 448, NaN becomes 0x7F, and
the sign of a zero result is kept.
"""

import numpy as np

MAX_FINITE = 448.0
NAN_CODE = 0x7F


def decode_code(code: int) -> float:
    """Value of one e4m3 byte, as a Python float (exact)."""
    code = int(code) & 0xFF
    sign = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 0x7
    if e == 0xF and m == 0x7:
        return float("nan")
    if e == 0:
        return sign * (2.0 ** -6) * (m / 8.0)
    return sign * (2.0 ** (e - 7)) * (1.0 + m / 8.0)


# Table of all 256 codes, float64.
DECODE_TABLE = np.array([decode_code(c) for c in range(256)], dtype=np.float64)

# The 127 finite non-negative codes 0x00..0x7E in increasing value order.
_POS_CODES = np.arange(0x7F, dtype=np.int64)
_POS_VALUES = DECODE_TABLE[:0x7F]
assert np.all(np.diff(_POS_VALUES) > 0)


def decode(codes: np.ndarray) -> np.ndarray:
    """Decode an array of e4m3 bytes to float64 (exact)."""
    return DECODE_TABLE[np.asarray(codes, dtype=np.uint8).astype(np.int64)]


def encode_f32(x: np.ndarray) -> np.ndarray:
    """Encode float32 values to e4m3 bytes: nearest, ties to even, saturating.

    ``x`` is taken as float32 (the precision the division ``value / scale``
    is done in on both sides); the rounding decision is then exact in
    float64, which holds every float32 and every e4m3 value.
    """
    x = np.asarray(x, dtype=np.float32)
    xf = x.astype(np.float64).ravel()
    out = np.empty(xf.shape, dtype=np.uint8)
    nan = np.isnan(xf)
    neg = np.signbit(xf)
    a = np.abs(xf)
    a = np.where(nan, 0.0, a)
    a = np.minimum(a, MAX_FINITE)  # saturation (infinity included)
    # Neighbours in the value table: lo <= a <= hi.
    hi_idx = np.searchsorted(_POS_VALUES, a, side="left")
    hi_idx = np.minimum(hi_idx, len(_POS_VALUES) - 1)
    lo_idx = np.maximum(hi_idx - 1, 0)
    exact = _POS_VALUES[hi_idx] == a
    lo_v = _POS_VALUES[lo_idx]
    hi_v = _POS_VALUES[hi_idx]
    d_lo = a - lo_v
    d_hi = hi_v - a
    pick_hi = d_hi < d_lo
    tie = d_hi == d_lo
    # Ties go to the code whose last mantissa bit is 0.
    hi_even = (_POS_CODES[hi_idx] & 1) == 0
    pick_hi = np.where(tie, hi_even, pick_hi)
    idx = np.where(exact, hi_idx, np.where(pick_hi, hi_idx, lo_idx))
    code = _POS_CODES[idx].astype(np.uint8)
    code = np.where(neg, code | 0x80, code).astype(np.uint8)
    code = np.where(nan, NAN_CODE, code).astype(np.uint8)
    out[:] = code
    return out.reshape(x.shape)


def quantise(values_f32: np.ndarray, scale_f32) -> np.ndarray:
    """KV-write quantisation: byte = encode(float32(value) / float32(scale)).

    The quotient is rounded to float32 (IEEE division), then to e4m3.
    """
    v = np.asarray(values_f32, dtype=np.float32)
    s = np.asarray(scale_f32, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        q = (v / s).astype(np.float32)
    return encode_f32(q)
