"""The page pool ledger (host, no GPU), the staging and save/restore planners
(dry runs), and the oracle's save/restore image."""

import threading

import numpy as np
import pytest

from oracle import kvcache
from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl

FAKE = 1 << 20


def test_claims_are_up_front_lowest_first_and_all_or_nothing():
    p = B.Pool(10)
    assert p.free() == 10 and p.fits(10) and not p.fits(11)
    assert p.claim(4).tolist() == [0, 1, 2, 3]
    with pytest.raises(B.TfpaError) as e:           # the pool cannot hold 7 now: wait
        p.claim(7)
    assert e.value.code == B.TFPA_ELANEMEM and p.free() == 6
    with pytest.raises(B.TfpaError) as e:           # never fits
        p.claim(11)
    assert e.value.code == B.TFPA_ECAPACITY
    p.release([1, 3])
    assert p.free() == 8
    assert p.claim(3).tolist() == [1, 3, 4]
    for bad in ([1, 1], [9], [-1], [10]):          # listed twice, not claimed, out of range
        with pytest.raises(B.TfpaError) as e:
            p.release(bad)
        assert e.value.code == B.TFPA_EINVAL
    assert p.free() == 5                           # nothing released by a refused call
    assert p.claim(0).tolist() == []


def test_ledger_matches_a_set_model():
    """Against an independent model: a set of free ids, lowest first."""
    rng = np.random.default_rng(2)
    p = B.Pool(64)
    free = set(range(64))
    held = []
    for _ in range(2000):
        if held and rng.random() < 0.45:
            grant = held.pop(int(rng.integers(len(held))))
            k = int(rng.integers(1, len(grant) + 1))
            back, keep = grant[:k], grant[k:]
            if keep:
                held.append(keep)
            p.release(back)
            free |= set(back)
        else:
            n = int(rng.integers(0, 20))
            if n > len(free):
                with pytest.raises(B.TfpaError) as e:
                    p.claim(n)
                assert e.value.code == B.TFPA_ELANEMEM
                continue
            got = p.claim(n).tolist()
            want = sorted(free)[:n]
            assert got == want
            free -= set(got)
            if got:
                held.append(got)
        assert p.free() == len(free)


def test_concurrent_claims_never_hand_out_a_page_twice():
    p = B.Pool(4096)
    got = [[] for _ in range(8)]

    def worker(i):
        for _ in range(50):
            try:
                got[i].extend(p.claim(7).tolist())
            except B.TfpaError as e:
                assert e.value.code == B.TFPA_ELANEMEM
    ts = [threading.Thread(target=worker, args=(i,)) for i in range(8)]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    allp = [x for g in got for x in g]
    assert len(allp) == len(set(allp)) and len(allp) + p.free() == 4096


def test_staging_and_copy_planners():
    with B.record_launches() as rec:
        B.tfpa_stage_pages(FAKE, 5, np.arange(3000))
    assert [(r["kind"], r["row0"], r["rows"]) for r in rec] == [("stage", 0, 2048),
                                                                ("stage", 2048, 952)]
    c = B.Cache("bf16", 32, 8, FAKE, 2 * FAKE, None, None, None, 4096)
    seg = B.Seg(1000, page_table=3 * FAKE)
    with B.record_launches() as rec:
        B.tfpa_save_kv(c, seg, 300, 700, 4 * FAKE)
        B.tfpa_restore_kv(c, seg, 255, 257, 4 * FAKE)
    # 300..699 spans pages 1 and 2; 255..256 spans pages 0 and 1; 8 heads x K,V per page
    assert [(r["kind"], r["rows"], r["grid"]) for r in rec] == [("save", 400, 32),
                                                                ("restore", 2, 32)]
    for p0, p1, code in ((0, 1001, B.TFPA_ERANGE), (10, 5, B.TFPA_ERANGE)):
        with pytest.raises(B.TfpaError) as e:
            B.tfpa_save_kv(c, seg, p0, p1, 4 * FAKE)
        assert e.value.code == code
    with pytest.raises(B.TfpaError) as e:
        B.tfpa_save_kv(c, seg, 0, 10, 4 * FAKE + 8)     # image not 16-byte aligned
    assert e.value.code == B.TFPA_EINVAL


@pytest.mark.parametrize("dtype", ["bf16", "fp8"])
def test_oracle_image_round_trip_and_contents(dtype):
    hkv, L = 2, 700
    n_pages = 5
    if dtype == "bf16":
        kp = wl.randn_bf16_bits((n_pages, hkv, 256, 128), 3)
        vp = wl.randn_bf16_bits((n_pages, hkv, 256, 128), 4)
    else:
        kp = wl.random_fp8_codes((n_pages, hkv, 256, 128), 3)
        vp = wl.random_fp8_codes((n_pages, hkv, 256, 128), 4)
    sc = np.array([0.01, 0.02], np.float32)
    cache = kvcache.Cache(dtype, hkv, 128, kp, vp, sc, sc)
    seg = kvcache.Segment(L, page_table=np.array([3, 0, 4], np.int32))
    k = wl.randn_bf16_bits((5, hkv, 128), 5)
    v = wl.randn_bf16_bits((5, hkv, 128), 6)
    pos = [254, 255, 256, 257, 600]
    kvcache.write_rows(cache, [seg], k, v, [0] * 5, pos)
    img = kvcache.save_image(cache, seg, 250, 610)
    assert img.shape == (2, hkv, 360, 128)
    for i, p in enumerate(pos):                    # the image holds what was written
        for g in range(hkv):
            a, idx = kvcache._store(cache, seg, "k", g, p)
            assert np.array_equal(img[0, g, p - 250], a[idx])
            if dtype == "bf16":
                assert np.array_equal(img[0, g, p - 250], k[i, g])
                assert np.array_equal(img[1, g, p - 250], v[i, g])
    other = kvcache.Cache(dtype, hkv, 128, np.zeros_like(kp), np.zeros_like(vp), sc, sc)
    seg2 = kvcache.Segment(L, page_table=np.array([1, 2, 0], np.int32))
    kvcache.restore_image(other, seg2, 250, 610, img)
    assert np.array_equal(kvcache.save_image(other, seg2, 250, 610), img)
