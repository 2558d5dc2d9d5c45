"""Host-side tests of the seeded workload generators (no GPU)."""

import numpy as np
import pytest

from paged_kv_cache_235_gb300 import workloads as wl


def test_generators_are_seeded_and_repeatable():
    a = wl.randn_bf16_bits((4, 5), 7)
    b = wl.randn_bf16_bits((4, 5), 7)
    c = wl.randn_bf16_bits((4, 5), 8)
    assert np.array_equal(a, b) and not np.array_equal(a, c)
    codes = wl.random_fp8_codes((10000,), 3)
    assert codes.dtype == np.uint8
    assert not np.isin(codes, [0x7F, 0xFF]).any()          # no NaN codes
    assert len(np.unique(codes)) == 254


def test_permuted_tables_are_disjoint_and_in_range():
    lengths = [1000, 257, 8192, 3]
    tables = wl.permuted_tables(lengths, [True, False, True, True], 64, 5)
    assert tables[1] is None
    used = np.concatenate([t for t in tables if t is not None])
    assert len(np.unique(used)) == len(used)
    assert used.min() >= 0 and used.max() < 64
    assert [len(t) for t in tables if t is not None] == [4, 32, 1]
    with pytest.raises(ValueError):
        wl.permuted_tables([100000], [True], 10, 1)


def test_first_fit_claims_lowest_free_pages_whole_or_not_at_all():
    pool = wl.FirstFitPool(10)
    a = pool.claim(3)
    b = pool.claim(2)
    assert a.tolist() == [0, 1, 2] and b.tolist() == [3, 4]
    pool.release(a[1:2])
    c = pool.claim(2)
    assert c.tolist() == [1, 5]                    # lowest free first, fragmented
    assert pool.claim(6) is None                   # does not fit: nothing claimed
    assert pool.free.sum() == 4
    assert pool.claim(4).tolist() == [6, 7, 8, 9]


def test_churn_is_deterministic_and_leaves_tenants():
    p1, p2 = wl.FirstFitPool(500), wl.FirstFitPool(500)
    p1.churn(9, rounds=300, max_pages=12, keep_fraction=0.25)
    p2.churn(9, rounds=300, max_pages=12, keep_fraction=0.25)
    assert np.array_equal(p1.free, p2.free)
    assert 0 < (~p1.free).sum() < 500


def test_workload_shapes():
    w = wl.tiny_paged_decode()
    assert (w.hq, w.hkv, w.num_pages, w.rows) == (8, 2, 16, 1)
    assert w.streams[0].seq_len == 1000 and len(w.streams[0].page_table) == 4
    assert w.row_pos.tolist() == [999]
    w = wl.batched_decode()
    assert [st.paged for st in w.streams] == [False] * 4 + [True] * 4
    assert all(st.slab_cap == 8192 for st in w.streams[:4])
    w = wl.fp8_verify()
    assert w.kv_dtype == "fp8" and w.rows == 32
    assert w.row_pos[:4].tolist() == [65532, 65533, 65534, 65535]
    w = wl.prompt_chunk()
    assert w.rows == 4096 and w.row_pos[0] == 28672 and w.row_pos[-1] == 32767
    assert w.streams[0].seq_len == 32768


def test_overcommitted_pool_seats_what_fits():
    w = wl.overcommitted_pool()
    assert w.num_pages == 1_300_000 // 256
    seated = [st.seq_len for st in w.streams]
    assert len(seated) + len(w.waiting) == 17
    pages = np.concatenate([st.page_table for st in w.streams])
    assert len(np.unique(pages)) == len(pages) and pages.max() < w.num_pages
    assert all(len(st.page_table) == (st.seq_len + 255) // 256 for st in w.streams)
    assert 262_144 in seated or 16 in w.waiting


def test_small_workloads_have_ragged_tails():
    for name in ("batched_decode", "fp8_verify", "prompt_chunk", "overcommitted_pool"):
        w = wl.small(name)
        assert any(st.seq_len % 256 for st in w.streams), name
