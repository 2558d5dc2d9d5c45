"""Small oracle-side cache builders shared by the oracle pin tests.

Builds an ``oracle.kvcache.Cache`` and its segments from a workload, writing
every stream's K/V rows through the oracle's own KV write.  Unused pool pages
and slab tails hold random data (never zeros), so a wrong address shows.
"""

import numpy as np

from oracle import kvcache
from paged_kv_cache_235_gb300 import workloads as wl


def build_oracle_cache(w: wl.Workload, k_scale=None, v_scale=None):
    hkv, d = w.hkv, w.d
    if w.kv_dtype == "bf16":
        kp = wl.randn_bf16_bits((w.num_pages, hkv, wl.PAGE, d), w.filler_seed("k"))
        vp = wl.randn_bf16_bits((w.num_pages, hkv, wl.PAGE, d), w.filler_seed("v"))
    else:
        kp = wl.random_fp8_codes((w.num_pages, hkv, wl.PAGE, d), w.filler_seed("k"))
        vp = wl.random_fp8_codes((w.num_pages, hkv, wl.PAGE, d), w.filler_seed("v"))
        if k_scale is None:
            k_scale, v_scale = w.fp8_scales()
    cache = kvcache.Cache(w.kv_dtype, hkv, d, kp, vp, k_scale, v_scale)
    segs = []
    for s, st in enumerate(w.streams):
        if st.paged:
            segs.append(kvcache.Segment(st.seq_len, page_table=st.page_table))
        else:
            if w.kv_dtype == "bf16":
                ks = wl.randn_bf16_bits((hkv, st.slab_cap, d), w.filler_seed("k") + 7 * s + 3)
                vs = wl.randn_bf16_bits((hkv, st.slab_cap, d), w.filler_seed("v") + 7 * s + 3)
            else:
                ks = wl.random_fp8_codes((hkv, st.slab_cap, d), w.filler_seed("k") + 7 * s + 3)
                vs = wl.random_fp8_codes((hkv, st.slab_cap, d), w.filler_seed("v") + 7 * s + 3)
            segs.append(kvcache.Segment(st.seq_len, k_slab=ks, v_slab=vs))
    for s, st in enumerate(w.streams):
        k, v = w.stream_kv_bits(s)
        L = st.seq_len
        rows_k = np.ascontiguousarray(k.transpose(1, 0, 2))   # [L][hkv][d]
        rows_v = np.ascontiguousarray(v.transpose(1, 0, 2))
        write_stream(cache, segs, s, rows_k, rows_v, L)
    return cache, segs


def write_stream(cache, segs, s, rows_k, rows_v, L):
    """All L positions of stream s (vectorised form of kvcache.write_rows)."""
    # Use the oracle's row write on a few rows, and its vector form on the rest,
    # checked equal in test_oracle_attention.test_kv_write_vector_form.
    seg = segs[s]
    for g in range(cache.hkv):
        for which, src in (("k", rows_k), ("v", rows_v)):
            if cache.dtype == "bf16":
                vals = src[:, g]
            else:
                from oracle import e4m3
                sc = cache.k_scale if which == "k" else cache.v_scale
                vals = e4m3.quantise(kvcache.bf16_to_f32(src[:, g]), sc[g])
            if seg.page_table is not None:
                pool = cache.k_pool if which == "k" else cache.v_pool
                for pi in range((L + 255) // 256):
                    lo, hi = pi * 256, min(L, pi * 256 + 256)
                    pool[int(seg.page_table[pi]), g, : hi - lo] = vals[lo:hi]
            else:
                slab = seg.k_slab if which == "k" else seg.v_slab
                slab[g, :L] = vals
