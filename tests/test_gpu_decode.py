"""Decode/verify attention on the GPU against the oracle, plus the bitwise
invariants: paged == contiguous, batched == alone, slices == one launch, and a
swapped page table that must come out red."""

import numpy as np
import pytest
import torch

from oracle import attention
from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, assert_close, bits, fp8_scales, to_f64
from tests.oracle_cases import build_oracle_cache

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp8": 3e-2}


def _oracle(w, scales=None, rows=None):
    cache, segs = build_oracle_cache(w, *(scales or (None, None)))
    q = w.q_bits()
    rs, rp = w.row_seg, w.row_pos
    if rows is not None:
        q, rs, rp = q[rows], rs[rows], rp[rows]
    return attention.attend(cache, segs, q, rs, rp, w.softmax_scale)


@pytest.mark.parametrize("name", ["tiny_paged_decode", "batched_decode", "fp8_verify",
                                  "overcommitted_pool"])
def test_small_workloads_match_oracle(name):
    w = wl.small(name)
    scales = fp8_scales(w) if w.kv_dtype == "fp8" else None
    g = GpuCase(w, scales)
    out, lse = g.decode(g.q(), w.row_seg, w.row_pos)
    ref, ref_lse = _oracle(w, scales)
    assert_close(to_f64(out), ref, TOL[w.kv_dtype], name)
    assert_close(to_f64(lse), ref_lse, 1e-3, name + " lse")
    assert int(g.err.item()) == 0


def test_tiny_paged_decode_full_size_config():
    w = wl.tiny_paged_decode()
    g = GpuCase(w)
    out, _ = g.decode(g.q(), w.row_seg, w.row_pos)
    ref, _ = _oracle(w)
    assert_close(to_f64(out), ref, 1e-2, "tiny")
    # paged == contiguous copy of the same stream, bitwise
    gc = GpuCase(w, all_paged=False)
    out2, _ = gc.decode(gc.q(), w.row_seg, w.row_pos)
    assert np.array_equal(bits(out), bits(out2))


@pytest.mark.parametrize("name", ["batched_decode", "fp8_verify"])
def test_paged_equals_contiguous_bitwise(name):
    w = wl.small(name)
    scales = fp8_scales(w) if w.kv_dtype == "fp8" else None
    lengths = [st.seq_len for st in w.streams]
    tables = wl.permuted_tables(lengths, [True] * len(lengths), w.num_pages + 40, 4242)
    w2 = wl.Workload(w.name, w.hq, w.hkv, w.kv_dtype, w.num_pages + 40, w.streams, w.row_seg,
                     w.row_pos, w.seed)
    paged = GpuCase(w2, scales, all_paged=True, tables=tables)
    slab = GpuCase(w2, scales, all_paged=False)
    a, la = paged.decode(paged.q(), w.row_seg, w.row_pos)
    b, lb = slab.decode(slab.q(), w.row_seg, w.row_pos)
    assert np.array_equal(bits(a), bits(b))
    assert torch.equal(la, lb)


@pytest.mark.parametrize("name", ["batched_decode", "fp8_verify", "overcommitted_pool"])
def test_batched_equals_alone_bitwise(name):
    w = wl.small(name)
    scales = fp8_scales(w) if w.kv_dtype == "fp8" else None
    g = GpuCase(w, scales)
    q = g.q()
    full, _ = g.decode(q, w.row_seg, w.row_pos)
    for s in range(len(w.streams)):
        sel = np.flatnonzero(w.row_seg == s)
        alone, _ = g.decode(q[sel], np.zeros(len(sel), np.int32), w.row_pos[sel],
                            segs=[g.segs[s]])
        assert np.array_equal(bits(alone), bits(full[sel])), f"stream {s}"


@pytest.mark.parametrize("cap", [1, 3, 5])
def test_slices_equal_one_launch_bitwise(cap):
    w = wl.small("fp8_verify")
    scales = fp8_scales(w)
    g = GpuCase(w, scales)
    q = g.q()
    one, l1 = g.decode(q, w.row_seg, w.row_pos, cap_rows=128)
    sl, l2 = g.decode(q, w.row_seg, w.row_pos, cap_rows=cap)
    assert np.array_equal(bits(one), bits(sl))
    assert torch.equal(l1, l2)


def test_partials_match_oracle_partials():
    w = wl.small("fp8_verify")
    scales = fp8_scales(w)
    g = GpuCase(w, scales)
    sc = B.make_scratch(w.rows, w.hq)
    B.tfpa_decode_partial(g.cache, g.segs, g.q(), w.row_seg, w.row_pos, w.softmax_scale, sc)
    torch.cuda.synchronize()
    cache, segs = build_oracle_cache(w, *scales)
    pps = B.tfpa_pages_per_split
    m, l, o, nsplit = attention.attend_partials(cache, segs, w.q_bits(), w.row_seg, w.row_pos,
                                                w.softmax_scale, pps)
    S = m.shape[-1]
    ml = sc.part_ml.view(w.rows, w.hq, B.MAX_SPLITS, 2).cpu().numpy().astype(np.float64)
    po = sc.part_o.view(w.rows, w.hq, B.MAX_SPLITS, 128).cpu().numpy().astype(np.float64)
    gm = ml[:, :, :S, 0] * np.log(2.0)   # log2 units -> natural
    gl = ml[:, :, :S, 1]
    go = po[:, :, :S]
    for r in range(w.rows):
        n = nsplit[r]
        assert n == B.tfpa_num_splits(w.streams[w.row_seg[r]].seq_len)
        fin = np.isfinite(m[r, :, :n])
        assert np.array_equal(fin, gl[r, :, :n] > 0)
        # (m, l, o) is defined up to the reference max m (the kernel may keep
        # a stale one): compare each split's lse and normalised output
        lse_o = m[r, :, :n] + np.log(np.where(fin, l[r, :, :n], 1.0))
        lse_g = gm[r, :, :n] + np.log(np.where(fin, gl[r, :, :n], 1.0))
        np.testing.assert_allclose(lse_g[fin], lse_o[fin], rtol=0, atol=2e-3)
        on = o[r, :, :n] / np.where(fin, l[r, :, :n], 1.0)[..., None]
        gn = go[r, :, :n] / np.where(fin, gl[r, :, :n], 1.0)[..., None]
        assert_close(gn[fin], on[fin], 3e-2, "normalised o")


def test_swapped_table_control_is_red():
    """Swapping the partial last page with a full page must break parity."""
    w = wl.tiny_paged_decode()
    t = w.streams[0].page_table.copy()
    t[[0, 3]] = t[[3, 0]]
    g = GpuCase(w)
    bad = B.Seg(1000, page_table=torch.from_numpy(t).cuda())
    out, _ = g.decode(g.q(), w.row_seg, w.row_pos, segs=[bad])
    ref, _ = _oracle(w)
    with pytest.raises(AssertionError):
        assert_close(to_f64(out), ref, 1e-2, "swapped")


def test_bad_page_id_is_flagged_not_faulted():
    w = wl.tiny_paged_decode()
    g = GpuCase(w)
    t = w.streams[0].page_table.copy()
    t[2] = w.num_pages + 7          # out of range; no host mirror to catch it
    bad = B.Seg(1000, page_table=torch.from_numpy(t).cuda())
    out, _ = g.decode(g.q(), w.row_seg, w.row_pos, segs=[bad])
    assert int(g.err.item()) & 1
    assert torch.isfinite(out.float()).all()


def test_host_mirror_rejects_bad_page():
    w = wl.tiny_paged_decode()
    g = GpuCase(w)
    t = w.streams[0].page_table.copy()
    t[1] = -3
    bad = B.Seg(1000, page_table=torch.from_numpy(t).cuda(), page_table_host=t)
    with pytest.raises(B.TfpaError) as e:
        g.decode(g.q(), w.row_seg, w.row_pos, segs=[bad])
    assert e.value.code == B.TFPA_ERANGE
