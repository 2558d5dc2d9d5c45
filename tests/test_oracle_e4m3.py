"""Pins of the oracle's e4m3 codec against the format definition and torch.

The decode table is checked against torch's own float8_e4m3fn (an independent
implementation) and against hand-derived values; the encoder against torch's
round-to-nearest-even cast in range, and against the saturating rule outside.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import e4m3


def _golden_codes(golden_dir):
    out = []
    with open(os.path.join(golden_dir, "e4m3_codes.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            c, v = line.split()
            out.append((int(c, 16), float(v)))
    return out


def test_decode_matches_torch_all_codes():
    codes = torch.arange(256, dtype=torch.int32).to(torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = e4m3.decode(np.arange(256, dtype=np.uint8))
    nan_ref = np.isnan(ref)
    assert np.array_equal(nan_ref, np.isnan(got))
    assert np.array_equal(ref[~nan_ref], got[~nan_ref])
    assert np.array_equal(np.signbit(ref[~nan_ref]), np.signbit(got[~nan_ref]))
    assert sorted(np.flatnonzero(nan_ref).tolist()) == [0x7F, 0xFF]


def test_decode_golden(golden_dir):
    for c, v in _golden_codes(golden_dir):
        got = e4m3.decode_code(c)
        if math.isnan(v):
            assert math.isnan(got), hex(c)
        else:
            assert got == v and math.copysign(1, got) == math.copysign(1, v), hex(c)


def test_encode_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    vals = e4m3.decode(codes).astype(np.float32)
    assert np.array_equal(e4m3.encode_f32(vals), codes)


def test_encode_matches_torch_rne_in_range():
    g = torch.Generator().manual_seed(5)
    x = torch.cat([
        torch.randn(20000, generator=g) * 40,
        torch.randn(20000, generator=g) * 0.02,
        (torch.rand(5000, generator=g) - 0.5) * 900,
    ]).to(torch.float32)
    x = x[x.abs() < 448]
    ref = x.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.encode_f32(x.numpy()), ref)


def test_encode_ties_go_to_even():
    pos = e4m3.decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((pos[:-1] + pos[1:]) / 2).astype(np.float32)
    assert np.array_equal(mids.astype(np.float64), (pos[:-1] + pos[1:]) / 2)  # exact in f32
    got = e4m3.encode_f32(mids)
    lo = np.arange(0x7E)
    want = np.where(lo % 2 == 0, lo, lo + 1).astype(np.uint8)
    assert np.array_equal(got, want)
    ref = torch.from_numpy(mids).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(got, ref)
    assert np.array_equal(e4m3.encode_f32(-mids), want | 0x80)


def test_encode_saturates_and_nan():
    x = np.array([448.0, 460.0, 464.0, 470.0, 500.0, 1e30, np.inf, -np.inf, -1e9, np.nan],
                 dtype=np.float32)
    got = e4m3.encode_f32(x).tolist()
    assert got == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]


def test_encode_underflow_keeps_sign():
    x = np.array([1e-10, -1e-10, 2.0 ** -10, -(2.0 ** -10), 3 * 2.0 ** -11, 0.0, -0.0],
                 dtype=np.float32)
    assert e4m3.encode_f32(x).tolist() == [0x00, 0x80, 0x00, 0x80, 0x01, 0x00, 0x80]


def test_quantise_divides_in_float32():
    g = torch.Generator().manual_seed(9)
    v = (torch.randn(5000, generator=g)).to(torch.bfloat16).to(torch.float32).numpy()
    s = np.float32(5.3 / 448)
    want = e4m3.encode_f32((v / s).astype(np.float32))
    assert np.array_equal(e4m3.quantise(v, s), want)
    ref = torch.from_numpy((v / s).astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(e4m3.quantise(v, s), ref)


@pytest.mark.parametrize("bug", ["bias8", "no_tie_even"])
def test_planted_codec_mistakes_are_caught(monkeypatch, bug):
    """A plausible mistake planted in the oracle's codec fails a pin above."""
    if bug == "bias8":
        table = np.array([e4m3.decode_code(c) / 2 for c in range(256)])
        monkeypatch.setattr(e4m3, "DECODE_TABLE", table)
        with pytest.raises(AssertionError):
            test_decode_matches_torch_all_codes()
    else:
        orig = e4m3.encode_f32

        def rounds_half_up(x):
            x = np.asarray(x, dtype=np.float32)
            pos = e4m3.decode(np.arange(0x7F, dtype=np.uint8))
            a = np.abs(x.astype(np.float64))
            idx = np.abs(a[..., None] - pos[None, :])
            best = np.argmin(idx[..., ::-1], axis=-1)
            code = (0x7E - best).astype(np.uint8)
            return np.where(np.signbit(x), code | 0x80, code).astype(np.uint8)

        monkeypatch.setattr(e4m3, "encode_f32", rounds_half_up)
        with pytest.raises(AssertionError):
            test_encode_ties_go_to_even()
        monkeypatch.setattr(e4m3, "encode_f32", orig)
