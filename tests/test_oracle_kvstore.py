"""Pins of the oracle's RoPE store and keep copy.

Pinned against what fixes them independently: torch's bf16 cast for the
rounding; basis vectors, whose rotation is a single product per output (so
exact), for the pairing (i, i + 64) and the signs; an explicit float64 2 x 2
rotation for random rows, within float32 rounding; math.cos/math.sin for the
table; and byte comparisons for keep, including a chain of moves.
"""

import math

import numpy as np
import pytest
import torch

from oracle import e4m3, kvcache, kvstore
from paged_kv_cache_235_gb300 import workloads as wl


def test_f32_to_bf16_matches_torch():
    g = torch.Generator().manual_seed(3)
    x = torch.cat([torch.randn(50000, generator=g) * 3,
                   torch.randn(5000, generator=g) * 1e-39,          # subnormals
                   torch.tensor([0.0, -0.0, 1e38, -3e38, float("inf"), -float("inf")])])
    # ties: values exactly halfway between two bf16 numbers
    base = (torch.randint(0, 1 << 15, (2000,), generator=g).to(torch.int32) << 16)
    ties = (base | 0x8000).view(torch.float32)
    x = torch.cat([x, ties, -ties]).to(torch.float32)
    ref = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = kvstore.f32_to_bf16(x.numpy())
    nan = np.isnan(x.numpy())               # NaN payloads are not part of the contract
    assert nan.any() and np.array_equal(got[~nan], ref[~nan])
    assert np.isnan(kvcache.bf16_to_f32(got[nan])).all()


def _bits(x):
    return kvstore.f32_to_bf16(np.asarray(x, np.float32))


def test_rotation_pairing_and_signs_on_basis_vectors():
    c, s = wl.rope_table(10000.0, 50)
    t = 37
    for i in (0, 5, 63):
        e = np.zeros(128, np.float32)
        e[i] = 1.0
        out = kvstore.rope_f32(_bits(e), c[t], s[t])
        want = np.zeros(128, np.float32)
        want[i], want[i + 64] = c[t, i], s[t, i]
        assert np.array_equal(out, want)
        e = np.zeros(128, np.float32)
        e[i + 64] = 1.0
        out = kvstore.rope_f32(_bits(e), c[t], s[t])
        want = np.zeros(128, np.float32)
        want[i], want[i + 64] = -s[t, i], c[t, i]
        assert np.array_equal(out, want)


def test_rotation_matches_float64_rotation_matrix():
    c, s = wl.rope_table(1e6, 3000)
    rng = np.random.default_rng(4)
    for t in (0, 1, 999, 2999):
        k = _bits(rng.standard_normal(128).astype(np.float32))
        kf = kvcache.bf16_to_f64(k)
        want = np.empty(128)
        for i in range(64):
            R = np.array([[float(c[t, i]), -float(s[t, i])], [float(s[t, i]), float(c[t, i])]])
            want[i], want[i + 64] = R @ np.array([kf[i], kf[i + 64]])
        got = kvstore.rope_f32(k, c[t], s[t]).astype(np.float64)
        assert np.max(np.abs(got - want)) <= 4 * np.finfo(np.float32).eps * (1 + np.abs(want)).max()
    # rotary position 0 is the identity, bit for bit
    k = _bits(rng.standard_normal(128).astype(np.float32))
    assert np.array_equal(kvstore.f32_to_bf16(kvstore.rope_f32(k, c[0], s[0])), k)


def test_rope_table_entries():
    c, s = wl.rope_table(10000.0, 4096)
    for t, i in ((1, 0), (17, 3), (4095, 63), (300, 40)):
        ang = t * 10000.0 ** (-2.0 * i / 128)
        assert c[t, i] == np.float32(math.cos(ang)) and s[t, i] == np.float32(math.sin(ang))


def _cache(dtype, L=600, hkv=2, paged=True, seed=5):
    n_pages = (L + 255) // 256 + 2
    if dtype == "bf16":
        kp = wl.randn_bf16_bits((n_pages, hkv, 256, 128), seed)
        vp = wl.randn_bf16_bits((n_pages, hkv, 256, 128), seed + 1)
        ks = vs = None
    else:
        kp = wl.random_fp8_codes((n_pages, hkv, 256, 128), seed)
        vp = wl.random_fp8_codes((n_pages, hkv, 256, 128), seed + 1)
        ks = np.array([0.011, 0.02], np.float32)[:hkv]
        vs = np.array([0.013, 0.017], np.float32)[:hkv]
    cache = kvcache.Cache(dtype, hkv, 128, kp, vp, ks, vs)
    table = np.random.default_rng(seed).permutation(n_pages)[: (L + 255) // 256].astype(np.int32)
    return cache, [kvcache.Segment(L, page_table=table)]


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_rope_store_rotates_k_only(dtype):
    cache, segs = _cache(dtype)
    c, s = wl.rope_table(1e6, 1024)
    k = wl.randn_bf16_bits((3, 2, 128), 8)
    v = wl.randn_bf16_bits((3, 2, 128), 9)
    rs, rp, rpos = [0, 0, 0], [10, 300, 599], [10, 2, 700]
    kvstore.write_rows_rope(cache, segs, k, v, rs, rp, rpos, c, s)
    for r in range(3):
        for g in range(2):
            ka, ki = kvcache._store(cache, segs[0], "k", g, rp[r])
            va, vi = kvcache._store(cache, segs[0], "v", g, rp[r])
            kf = kvstore.rope_f32(k[r, g], c[rpos[r]], s[rpos[r]])
            if dtype == "bf16":
                assert np.array_equal(ka[ki], kvstore.f32_to_bf16(kf))
                assert np.array_equal(va[vi], v[r, g])
            else:
                assert np.array_equal(ka[ki], e4m3.quantise(kf, cache.k_scale[g]))
                assert np.array_equal(va[vi], e4m3.quantise(kvcache.bf16_to_f32(v[r, g]),
                                                            cache.v_scale[g]))


def test_keep_chain_and_untouched_rows():
    cache, segs = _cache("bf16")
    before = (cache.k_pool.copy(), cache.v_pool.copy())
    snap = {}
    for pos in range(590, 600):
        for g in range(2):
            snap[(pos, g)] = (kvcache._store(cache, segs[0], "k", g, pos)[0][
                kvcache._store(cache, segs[0], "k", g, pos)[1]].copy(),
                kvcache._store(cache, segs[0], "v", g, pos)[0][
                kvcache._store(cache, segs[0], "v", g, pos)[1]].copy())
    # accepted path at tree indices 0, 2, 5 -> committed positions 590, 591, 592
    kvstore.keep_rows(cache, segs, [0, 0, 0], [590, 592, 595], [590, 591, 592])
    for src, dst in ((590, 590), (592, 591), (595, 592)):
        for g in range(2):
            ka, ki = kvcache._store(cache, segs[0], "k", g, dst)
            va, vi = kvcache._store(cache, segs[0], "v", g, dst)
            assert np.array_equal(ka[ki], snap[(src, g)][0])
            assert np.array_equal(va[vi], snap[(src, g)][1])
    changed = np.argwhere((cache.k_pool != before[0]).any(axis=-1))
    touched = {(int(p), int(g), int(r)) for p, g, r in changed}
    allowed = set()
    for dst in (591, 592):
        for g in range(2):
            _, (page, gg, row) = kvcache._store(cache, segs[0], "k", g, dst)
            allowed.add((page, gg, row))
    assert touched <= allowed


def test_planted_sign_mistake_is_caught(monkeypatch):
    def wrong(k_bits, cos, sin):
        k = kvcache.bf16_to_f32(k_bits)
        a, b = k[:64], k[64:]
        return np.concatenate([a * cos + b * sin, b * cos - a * sin]).astype(np.float32)
    monkeypatch.setattr(kvstore, "rope_f32", wrong)
    with pytest.raises(AssertionError):
        test_rotation_pairing_and_signs_on_basis_vectors()


def test_keep_reads_every_source_before_writing():
    """The chain 3 -> 2, 2 -> 1: row 1 must get the old row 2, row 2 the old row 3."""
    cache, segs = _cache("bf16")
    old = {}
    for pos in (1, 2, 3):
        a, i = kvcache._store(cache, segs[0], "k", 1, pos)
        old[pos] = a[i].copy()
    kvstore.keep_rows(cache, segs, [0, 0], [3, 2], [2, 1])
    for dst, src in ((1, 2), (2, 3)):
        a, i = kvcache._store(cache, segs[0], "k", 1, dst)
        assert np.array_equal(a[i], old[src])


def test_planted_keep_without_staging_is_caught(monkeypatch):
    """A keep that writes each destination as it goes fails the pin above."""
    def in_order(cache, segs, keep_seg, keep_src, keep_dst):
        for s, src, dst in zip(keep_seg, keep_src, keep_dst):
            for g in range(cache.hkv):
                for which in ("k", "v"):
                    a, i = kvcache._store(cache, segs[int(s)], which, g, int(src))
                    b, j = kvcache._store(cache, segs[int(s)], which, g, int(dst))
                    b[j] = a[i]
    monkeypatch.setattr(kvstore, "keep_rows", in_order)
    with pytest.raises(AssertionError):
        test_keep_reads_every_source_before_writing()
