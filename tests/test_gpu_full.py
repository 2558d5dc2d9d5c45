"""Full-size workloads, in the launch configuration the bench times, checked
on sampled streams against the oracle (each sampled stream is rebuilt on the
oracle side as a slab from the same generated values)."""

import numpy as np
import pytest
import torch

from oracle import attention, kvcache
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, WKey, assert_close, bits, fp8_scales, stream_kv, to_f64

pytestmark = [pytest.mark.gpu, pytest.mark.slow]


def oracle_stream(w, s, rows, scales):
    """Oracle output for the given rows (all of stream s)."""
    k, v = stream_kv(WKey(w), s)
    L = w.streams[s].seq_len
    cap = ((L + 255) // 256) * 256
    if w.kv_dtype == "fp8":
        from oracle import e4m3
        ks, vs = scales
        kq = np.zeros((w.hkv, cap, w.d), np.uint8)
        vq = np.zeros((w.hkv, cap, w.d), np.uint8)
        for g in range(w.hkv):
            kq[g, :L] = e4m3.quantise(kvcache.bf16_to_f32(k[g]), ks[g])
            vq[g, :L] = e4m3.quantise(kvcache.bf16_to_f32(v[g]), vs[g])
        cache = kvcache.Cache("fp8", w.hkv, w.d, None, None, ks, vs)
        seg = kvcache.Segment(L, k_slab=kq, v_slab=vq)
    else:
        kb = np.zeros((w.hkv, cap, w.d), np.uint16)
        vb = np.zeros((w.hkv, cap, w.d), np.uint16)
        kb[:, :L], vb[:, :L] = k, v
        cache = kvcache.Cache("bf16", w.hkv, w.d, None, None)
        seg = kvcache.Segment(L, k_slab=kb, v_slab=vb)
    q = w.q_bits()[rows]
    return attention.attend(cache, [seg], q, np.zeros(len(rows), np.int32), w.row_pos[rows],
                            w.softmax_scale)


def _check_streams(w, g, out, lse, streams, scales, tol):
    for s in streams:
        rows = np.flatnonzero(w.row_seg == s)
        ref, ref_lse = oracle_stream(w, s, rows, scales)
        assert_close(to_f64(out[rows]), ref, tol, f"{w.name} stream {s}")
        assert_close(to_f64(lse[rows]), ref_lse, 1e-3, f"{w.name} stream {s} lse")


def test_batched_decode_full():
    w = wl.batched_decode()
    g = GpuCase(w)
    q = g.q()
    out, lse = g.decode(q, w.row_seg, w.row_pos)
    _check_streams(w, g, out, lse, range(8), None, 1e-2)
    for s in (0, 5):                            # batched == alone, bitwise
        sel = np.flatnonzero(w.row_seg == s)
        alone, _ = g.decode(q[sel], np.zeros(len(sel), np.int32), w.row_pos[sel], segs=[g.segs[s]])
        assert np.array_equal(bits(alone), bits(out[sel]))


def test_fp8_verify_full():
    w = wl.fp8_verify()
    scales = fp8_scales(w)
    g = GpuCase(w, scales)
    out, lse = g.decode(g.q(), w.row_seg, w.row_pos)
    _check_streams(w, g, out, lse, (0, 7), scales, 3e-2)
    assert int(g.err.item()) == 0


def test_overcommitted_pool_full():
    w = wl.overcommitted_pool()
    assert len(w.streams) >= 8
    scales = fp8_scales(w)
    g = GpuCase(w, scales)
    out, lse = g.decode(g.q(), w.row_seg, w.row_pos)
    longest = int(np.argmax([st.seq_len for st in w.streams]))
    _check_streams(w, g, out, lse, (0, longest), scales, 3e-2)
