"""Device-side set-up of a workload through the library's own entry points.

Pools and slabs are first filled with the workload's random filler (the same
bytes the oracle side uses), then every stream's K/V rows are written with
``tfpa_write_kv``.  Nothing here imports the oracle.
"""

import functools

import numpy as np
import torch

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl


@functools.lru_cache(maxsize=24)
def stream_kv(w_key, s):
    w = w_key.w
    return w.stream_kv_bits(s)


class WKey:
    """Hashable handle so lru_cache keeps one workload's generated values."""

    def __init__(self, w):
        self.w = w

    def _key(self):
        w = self.w
        return (w.name, w.seed, w.hq, w.hkv, w.d, w.kv_dtype,
                tuple(st.seq_len for st in w.streams))

    def __hash__(self):
        return hash(self._key())

    def __eq__(self, o):
        return self._key() == o._key()


def fp8_scales(w):
    key = WKey(w)
    ka = np.zeros(w.hkv, np.float32)
    va = np.zeros(w.hkv, np.float32)
    for s in range(len(w.streams)):
        k, v = stream_kv(key, s)
        ka = np.maximum(ka, np.abs((k.astype(np.uint32) << 16).view(np.float32)).max(axis=(1, 2)))
        va = np.maximum(va, np.abs((v.astype(np.uint32) << 16).view(np.float32)).max(axis=(1, 2)))
    return (ka / np.float32(448)).astype(np.float32), (va / np.float32(448)).astype(np.float32)


def _dev(a, dtype=None):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype is not None:
        t = t.view(dtype)
    return t.cuda()


class GpuCase:
    """A workload's cache on the GPU, filled through tfpa_write_kv."""

    def __init__(self, w: wl.Workload, scales=None, all_paged=None, tables=None):
        self.w = w
        key = WKey(w)
        hkv, d = w.hkv, w.d
        fp8 = w.kv_dtype == "fp8"
        if fp8:
            kp = wl.random_fp8_codes((w.num_pages, hkv, wl.PAGE, d), w.filler_seed("k"))
            vp = wl.random_fp8_codes((w.num_pages, hkv, wl.PAGE, d), w.filler_seed("v"))
            self.k_pool, self.v_pool = _dev(kp), _dev(vp)
            ks, vs = scales if scales is not None else fp8_scales(w)
            self.k_scale, self.v_scale = _dev(ks), _dev(vs)
        else:
            kp = wl.randn_bf16_bits((w.num_pages, hkv, wl.PAGE, d), w.filler_seed("k"))
            vp = wl.randn_bf16_bits((w.num_pages, hkv, wl.PAGE, d), w.filler_seed("v"))
            self.k_pool = _dev(kp.view(np.int16), torch.bfloat16)
            self.v_pool = _dev(vp.view(np.int16), torch.bfloat16)
            self.k_scale = self.v_scale = None
        self.err = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.cache = B.Cache(w.kv_dtype, w.hq, hkv, self.k_pool, self.v_pool, self.k_scale,
                             self.v_scale, self.err, w.num_pages)
        self.segs = []
        for s, st in enumerate(w.streams):
            paged = st.paged if all_paged is None else all_paged
            if paged:
                table = st.page_table if tables is None else tables[s]
                self.segs.append(B.Seg(st.seq_len, page_table=_dev(table),
                                       page_table_host=np.asarray(table, np.int32)))
            else:
                cap = ((st.seq_len + 255) // 256) * 256
                if fp8:
                    ksl = wl.random_fp8_codes((hkv, cap, d), w.filler_seed("k") + 7 * s + 3)
                    vsl = wl.random_fp8_codes((hkv, cap, d), w.filler_seed("v") + 7 * s + 3)
                    ksl, vsl = _dev(ksl), _dev(vsl)
                else:
                    ksl = _dev(wl.randn_bf16_bits((hkv, cap, d), w.filler_seed("k") + 7 * s + 3)
                               .view(np.int16), torch.bfloat16)
                    vsl = _dev(wl.randn_bf16_bits((hkv, cap, d), w.filler_seed("v") + 7 * s + 3)
                               .view(np.int16), torch.bfloat16)
                self.segs.append(B.Seg(st.seq_len, k_slab=ksl, v_slab=vsl, slab_cap=cap))
        for s, st in enumerate(w.streams):
            k, v = stream_kv(key, s)
            kr = _dev(np.ascontiguousarray(k.transpose(1, 0, 2)).view(np.int16), torch.bfloat16)
            vr = _dev(np.ascontiguousarray(v.transpose(1, 0, 2)).view(np.int16), torch.bfloat16)
            L = st.seq_len
            B.tfpa_write_kv(self.cache, self.segs, kr, vr, np.full(L, s, np.int32),
                            np.arange(L, dtype=np.int32))
        torch.cuda.synchronize()

    def q(self, rows=None):
        qb = self.w.q_bits()
        if rows is not None:
            qb = qb[rows]
        return _dev(qb.view(np.int16), torch.bfloat16)

    def decode(self, q, row_seg, row_pos, cap_rows=128, segs=None, lse=True, fused=False):
        rows = len(row_seg)
        out = torch.empty(rows, self.w.hq, self.w.d, dtype=torch.bfloat16, device="cuda")
        l = torch.empty(rows, self.w.hq, dtype=torch.float32, device="cuda") if lse else None
        sc = B.make_scratch(cap_rows, self.w.hq, fused_merge=fused)
        B.tfpa_decode(self.cache, segs or self.segs, q, row_seg, row_pos, self.w.softmax_scale,
                      sc, out, l)
        torch.cuda.synchronize()
        return out, l

    def decode_tree(self, q, row_seg, row_pos, row_anc, cap_rows=128, lse=True, fused=False):
        rows = len(row_seg)
        anc = torch.from_numpy(np.ascontiguousarray(np.asarray(row_anc, np.uint64))
                               .view(np.int64)).cuda()
        out = torch.empty(rows, self.w.hq, self.w.d, dtype=torch.bfloat16, device="cuda")
        l = torch.empty(rows, self.w.hq, dtype=torch.float32, device="cuda") if lse else None
        sc = B.make_scratch(cap_rows, self.w.hq, fused_merge=fused)
        B.tfpa_decode_tree(self.cache, self.segs, q, row_seg, row_pos, anc,
                           self.w.softmax_scale, sc, out, l)
        torch.cuda.synchronize()
        return out, l

    def prefill(self, q, row_seg, row_pos, max_rows=0, segs=None):
        rows = len(row_seg)
        out = torch.empty(rows, self.w.hq, self.w.d, dtype=torch.bfloat16, device="cuda")
        l = torch.empty(rows, self.w.hq, dtype=torch.float32, device="cuda")
        B.tfpa_prefill(self.cache, segs or self.segs, q, row_seg, row_pos, self.w.softmax_scale,
                       out, l, max_rows_per_launch=max_rows)
        torch.cuda.synchronize()
        return out, l


def bits(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().astype(np.float64)


def assert_close(got: np.ndarray, ref: np.ndarray, tol: float, what: str = ""):
    """|got - ref| <= tol + tol * |ref| element-wise (the stated tolerance)."""
    err = np.abs(got - ref)
    bound = tol + tol * np.abs(ref)
    bad = err > bound
    if bad.any():
        i = np.unravel_index(np.argmax(err - bound), err.shape)
        raise AssertionError(f"{what}: {bad.sum()} of {bad.size} outside {tol}; worst at {i}: "
                             f"got {got[i]} ref {ref[i]} (max abs err {err.max():.3e})")


def append_rows(w, rows_per_stream, seed):
    """The last rows_per_stream positions of every stream, with new K / V
    and q (device bf16): row_seg, row_pos, k, v, q."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    rs, rp = [], []
    for s, st in enumerate(w.streams):
        for i in range(rows_per_stream):
            rs.append(s)
            rp.append(st.seq_len - rows_per_stream + i)
    n = len(rs)
    k = torch.randn(n, w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    v = torch.randn(n, w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
    q = torch.randn(n, w.hq, 128, generator=g, device="cuda").to(torch.bfloat16)
    return np.array(rs, np.int32), np.array(rp, np.int32), k, v, q


def same_cache(ga, gb):
    """Two GpuCases' pools and slabs hold the same bytes."""
    assert torch.equal(ga.k_pool, gb.k_pool) and torch.equal(ga.v_pool, gb.v_pool)
    for sa, sb in zip(ga.segs, gb.segs):
        if sa.page_table is None:
            assert torch.equal(sa.k_slab, sb.k_slab) and torch.equal(sa.v_slab, sb.v_slab)
