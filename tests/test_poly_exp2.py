"""The FMA-pipe exp2 used for a quarter of the prompt kernel's softmax
exponentials: its constants, restated from paged_kv_cache_235_gb300/csrc/
common.cuh, evaluated in float32 exactly as the kernel does, must stay within
1e-4 relative error of 2^x on [-125, 8] (the kernel rounds the result to bf16
or f16 next, whose unit roundoff is 2^-9 or 2^-12)."""

import re
import os

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _coeffs():
    with open(os.path.join(ROOT, "paged_kv_cache_235_gb300", "csrc", "common.cuh")) as f:
        text = f.read()
    return [np.float32(float(re.search(rf"kExp2C{i} = ([0-9.e+-]+)f", text).group(1)))
            for i in range(4)]


def poly_exp2_f32(x):
    c0, c1, c2, c3 = _coeffs()
    x = np.maximum(np.asarray(x, np.float32), np.float32(-125))
    t = (x + np.float32(12582912.0)).astype(np.float32)
    n = (t - np.float32(12582912.0)).astype(np.float32)
    f = (x - n).astype(np.float32)
    p = np.float32(c3)
    for c in (c2, c1, c0):
        p = (p * f + c).astype(np.float32)        # fmaf in the kernel; error bound covers it
    ni = t.view(np.int32) - np.int32(0x4B400000)
    return (p.view(np.int32) + (ni << 23)).view(np.float32)


def test_poly_exp2_relative_error_bound():
    x = np.concatenate([np.linspace(-125, 8, 2_000_001, dtype=np.float32),
                        np.float32([0.0, -0.5, 0.5, 8.0, -125.0, -1e-7, 1e-7])])
    got = poly_exp2_f32(x).astype(np.float64)
    want = np.exp2(x.astype(np.float64))
    rel = np.abs(got - want) / want
    assert rel.max() < 1e-4


def test_poly_exp2_integers_are_near_exact():
    n = np.arange(-125, 9, dtype=np.float32)
    got = poly_exp2_f32(n).astype(np.float64)
    np.testing.assert_allclose(got, np.exp2(n.astype(np.float64)), rtol=1e-4, atol=0)
