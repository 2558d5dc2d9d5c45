"""Host-side tests of the C ABI (no GPU): exports, the split policy, the slice
loop (recorded in dry-run mode, as the pages' launch-recording host test did)
and argument checking."""

import os
import re

import numpy as np
import pytest

from paged_kv_cache_235_gb300 import binding as B

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

FAKE = 1 << 20   # a 1 MiB-aligned fake device address; dry runs never touch it


def _declared():
    with open(os.path.join(ROOT, "include", "tfpa.h")) as f:
        text = f.read()
    return sorted(set(re.findall(r"\b(tfpa_[a-z_]+)\s*\(", text)))


def test_library_exports_every_declared_symbol():
    names = _declared()
    assert "tfpa_decode" in names and "tfpa_prefill" in names
    L = B.lib()
    for n in names:
        assert hasattr(L, n), n
    assert set(names) == set(B.EXPORTS)


def test_split_policy_depends_on_length_only():
    for L, pps, ns in [(1, 1, 1), (256, 1, 1), (257, 1, 2), (513, 1, 3), (1000, 1, 4),
                       (4096, 1, 16), (4097, 2, 9), (8192, 2, 16), (8193, 2, 17),
                       (16384, 2, 32), (16385, 3, 22), (65536, 8, 32), (262144, 32, 32),
                       (109000, 14, 31)]:
        assert B.tfpa_pages_per_split(L) == pps, L
        assert B.tfpa_num_splits(L) == ns, L
    for L in range(1, 300000, 997):
        n = B.tfpa_num_splits(L)
        assert 1 <= n <= B.MAX_SPLITS
        assert (n - 1) * B.tfpa_pages_per_split(L) * 256 < L <= n * B.tfpa_pages_per_split(L) * 256


def _cache(hq=32, hkv=8, dtype="bf16"):
    return B.Cache(dtype, hq, hkv, FAKE, 2 * FAKE, FAKE if dtype == "fp8" else None,
                   FAKE if dtype == "fp8" else None, None, 4096)


# A run of 13 or more rows (49+ query vectors per kv head at 32/8 heads) is
# computed by the tensor-core verify kernel, a shorter one by the decode
# partial kernel; both leave split partials for the same merge.
PARTIALS = ("partial", "verify")


@pytest.mark.parametrize("rows", [1, 12, 13, 127, 128, 129, 255, 256, 257, 4096])
def test_decode_slices_of_at_most_cap_rows(rows):
    c = _cache()
    segs = [B.Seg(rows + 40000, page_table=3 * FAKE)]
    with B.record_launches() as rec:
        B.tfpa_decode(c, segs, 4 * FAKE, np.zeros(rows), np.arange(40000, 40000 + rows), 0.088,
                      B.Scratch(5 * FAKE, 6 * FAKE, 128), 7 * FAKE)
    parts = [r for r in rec if r["kind"] in PARTIALS]
    merges = [r for r in rec if r["kind"] == "merge"]
    n = (rows + 127) // 128
    kind = "verify" if rows >= 13 else "partial"
    assert len(parts) == len(merges) == n
    assert [r["kind"] for r in rec] == [kind, "merge"] * n           # pairs, in order
    assert [r["row0"] for r in parts] == [128 * i for i in range(n)]
    assert sum(r["rows"] for r in merges) == rows                    # every row merged once
    hd = 32 * 128
    assert [r["q_offset"] for r in parts] == [128 * i * hd for i in range(n)]
    assert [r["out_offset"] for r in merges] == [128 * i * hd for i in range(n)]


def test_257_row_chunk_issues_three_pairs():
    c = _cache()
    segs = [B.Seg(32768, page_table=3 * FAKE)]
    with B.record_launches() as rec:
        B.tfpa_decode(c, segs, 4 * FAKE, np.zeros(257), np.arange(28672, 28929), 0.088,
                      B.Scratch(5 * FAKE, 6 * FAKE, 128), 7 * FAKE)
    # the 1-row tail belongs to a 257-row run: decided on the call's run, it
    # stays on the verify kernel
    assert [(r["kind"], r["row0"], r["rows"]) for r in rec] == [
        ("verify", 0, 128), ("merge", 0, 128), ("verify", 128, 128), ("merge", 128, 128),
        ("verify", 256, 1), ("merge", 256, 1)]


def test_mixed_paged_and_slab_streams_cross_slices():
    c = _cache()
    segs = [B.Seg(700, k_slab=8 * FAKE, v_slab=9 * FAKE, slab_cap=768),
            B.Seg(300, page_table=3 * FAKE)]
    rs = np.array([0] * 100 + [1] * 100)
    rp = np.concatenate([np.arange(600, 700), np.arange(200, 300)])
    with B.record_launches() as rec:
        B.tfpa_decode(c, segs, 4 * FAKE, rs, rp, 0.088, B.Scratch(5 * FAKE, 6 * FAKE, 128),
                      7 * FAKE)
    parts = [r for r in rec if r["kind"] in PARTIALS]
    assert [(r["row0"], r["rows"], r["runs"]) for r in parts] == [(0, 128, 2), (128, 72, 1)]


def test_prefill_slices():
    c = _cache()
    segs = [B.Seg(28672 + 257, page_table=3 * FAKE)]
    with B.record_launches() as rec:
        B.tfpa_prefill(c, segs, 4 * FAKE, np.zeros(257), np.arange(28672, 28929), 0.088,
                       7 * FAKE, max_rows_per_launch=128)
    assert [(r["kind"], r["row0"], r["rows"]) for r in rec] == [
        ("prefill", 0, 128), ("prefill", 128, 128), ("prefill", 256, 1)]
    # tiles: kv heads x head pairs x 128-row tiles; a cluster of two CTAs per tile
    assert [r["items"] for r in rec] == [8 * 2 * 1] * 3
    assert [r["grid"] for r in rec] == [2 * 8 * 2 * 1] * 3
    with B.record_launches() as rec:
        B.tfpa_prefill(c, segs, 4 * FAKE, np.zeros(257), np.arange(28672, 28929), 0.088,
                       7 * FAKE)
    assert [(r["kind"], r["rows"], r["items"]) for r in rec] == [("prefill", 257, 8 * 2 * 3)]


def test_verify_tiles_and_mixed_launch_order():
    """Verify tiles: kv head x tile of 128 / G rows x split, splits of at
    least 24 pages and at most 7 a stream; a call with a short and a long
    run issues the decode partial, then the verify launch, then one merge
    over both."""
    c = _cache()
    L = 65536
    segs = [B.Seg(L, page_table=3 * FAKE), B.Seg(L, page_table=3 * FAKE)]
    rs = np.array([0] + [1] * 16)
    rp = np.concatenate([[L - 1], np.arange(L - 16, L)])
    with B.record_launches() as rec:
        B.tfpa_decode(c, segs, 4 * FAKE, rs, rp, 0.088, B.Scratch(5 * FAKE, 6 * FAKE, 128),
                      7 * FAKE)
    assert [(r["kind"], r["row0"], r["rows"], r["runs"]) for r in rec] == [
        ("partial", 0, 17, 1), ("verify", 0, 17, 1), ("merge", 0, 17, 2)]
    v = rec[1]
    splits = 7                                    # 65,536 keys = 256 pages, 37 a split
    assert v["items"] == v["grid"] == 8 * 1 * 1 * splits
    assert rec[0]["items"] == 8 * 1 * B.tfpa_num_splits(L)   # 4 vectors: one m-tile


@pytest.mark.parametrize("hq,hkv,rows,kind,count", [
    (32, 8, 12, "partial", 8 * 3 * 32),    # 48 vectors a kv head: decode items
    (32, 8, 13, "verify", 8 * 1 * 7),      # 52 vectors: 32-row tiles, 7 splits of 37 pages
    (8, 8, 49, "verify", 8 * 1 * 7),       # one head a group: 128-row tiles
    (24, 8, 20, "verify", 8 * 1 * 7),      # three heads: 42-row tiles
    (64, 8, 20, "verify", 8 * 2 * 7),      # eight heads: 16-row tiles, two of them
    (129, 1, 1, "partial", 1 * 9 * 32),    # a group wider than a tile: decode items
])
def test_kernel_choice_by_query_vectors(hq, hkv, rows, kind, count):
    """Which kernel a run takes depends on its query vectors per kv head only:
    49 or more (and at most 128 heads a group) go to the verify kernel, whose
    tiles hold 128 / G rows; the items or tiles count follows."""
    c = _cache(hq, hkv)
    L = 65536
    segs = [B.Seg(L, page_table=3 * FAKE)]
    with B.record_launches() as rec:
        B.tfpa_decode(c, segs, 4 * FAKE, np.zeros(rows), np.arange(L - rows, L), 0.088,
                      B.Scratch(5 * FAKE, 6 * FAKE, 128), 7 * FAKE)
    assert [r["kind"] for r in rec] == [kind, "merge"]
    assert rec[0]["items"] == count


def test_write_kv_one_launch_per_64_runs():
    c = _cache()
    segs = [B.Seg(1000, page_table=3 * FAKE) for _ in range(100)]
    with B.record_launches() as rec:
        B.tfpa_write_kv(c, segs, 4 * FAKE, 5 * FAKE, np.arange(100), np.full(100, 999))
    assert [(r["kind"], r["rows"]) for r in rec] == [("write_kv", 64), ("write_kv", 36)]


@pytest.mark.parametrize("bad,code", [
    (dict(hq=30, hkv=8), B.TFPA_EINVAL),
    (dict(pos=1000), B.TFPA_ERANGE),
    (dict(pos=-1), B.TFPA_ERANGE),
    (dict(seg=1), B.TFPA_ERANGE),
    (dict(max_splits=1), B.TFPA_ECAPACITY),
    (dict(page=5000), B.TFPA_ERANGE),
    (dict(q=FAKE + 2), B.TFPA_EINVAL),
    (dict(slab_cap=1000), B.TFPA_EINVAL),
])
def test_argument_errors(bad, code):
    c = _cache(hq=bad.get("hq", 32), hkv=bad.get("hkv", 8))
    table = np.arange(4, dtype=np.int32)
    if "page" in bad:
        table[2] = bad["page"]
    segs = [B.Seg(1000, page_table=3 * FAKE, page_table_host=table)]
    if "slab_cap" in bad:
        segs = [B.Seg(1000, k_slab=FAKE, v_slab=FAKE, slab_cap=bad["slab_cap"])]
    with B.record_launches() as rec:
        with pytest.raises(B.TfpaError) as e:
            B.tfpa_decode(c, segs, bad.get("q", 4 * FAKE), [bad.get("seg", 0)],
                          [bad.get("pos", 999)], 0.088,
                          B.Scratch(5 * FAKE, 6 * FAKE, 128, bad.get("max_splits", 32)), 7 * FAKE)
    assert e.value.code == code
    assert rec == []                 # nothing enqueued on error


def test_merge_rejects_rows_beyond_capacity():
    with B.record_launches():
        with pytest.raises(B.TfpaError) as e:
            B.tfpa_merge(B.Scratch(5 * FAKE, 6 * FAKE, 128), 32, np.ones(129), 7 * FAKE)
    assert e.value.code == B.TFPA_ECAPACITY


def test_decode_tree_checks_its_ancestor_table():
    c = _cache()
    segs = [B.Seg(1000, page_table=3 * FAKE)]
    sc = B.Scratch(5 * FAKE, 6 * FAKE, 128)
    for anc in (None, 8 * FAKE + 4):                  # missing, not 8-byte aligned
        with B.record_launches() as rec:
            with pytest.raises(B.TfpaError) as e:
                B.tfpa_decode_tree(c, segs, 4 * FAKE, [0], [999], anc, 0.088, sc, 7 * FAKE)
        assert e.value.code == B.TFPA_EINVAL
        assert rec == []
    with B.record_launches() as rec:
        B.tfpa_decode_tree(c, segs, 4 * FAKE, [0] * 200, list(range(800, 1000)), 8 * FAKE,
                           0.088, sc, 7 * FAKE)
    assert [(r["kind"], r["row0"], r["rows"]) for r in rec] == [
        ("verify", 0, 128), ("merge", 0, 128), ("verify", 128, 72), ("merge", 128, 72)]


def test_write_kv_rope_and_keep_argument_checks():
    c = _cache()
    segs = [B.Seg(1000, page_table=3 * FAKE), B.Seg(500, page_table=4 * FAKE)]

    class T:          # a fake device table: address and shape only
        def __init__(self, addr, n):
            self.addr, self.shape = addr, (n, 64)

        def data_ptr(self):
            return self.addr
    cos, sin = T(5 * FAKE, 900), T(6 * FAKE, 900)
    with B.record_launches() as rec:
        with pytest.raises(B.TfpaError) as e:       # storage position 950 outside a 900-row table
            B.tfpa_write_kv_rope(c, segs, FAKE, 2 * FAKE, [0], [950], cos, sin)
    assert e.value.code == B.TFPA_ERANGE and rec == []
    with B.record_launches() as rec:
        B.tfpa_write_kv_rope(c, segs, FAKE, 2 * FAKE, [0, 0, 1], [800, 801, 3], cos, sin)
    assert [(r["kind"], r["rows"]) for r in rec] == [("write_kv", 3)]
    bad_keep = [([0], [1000], [5], B.TFPA_ERANGE),          # source past the end
                ([2], [3], [5], B.TFPA_ERANGE),             # no such segment
                ([0, 0], [3, 4], [5, 5], B.TFPA_EINVAL),    # two writers for one row
                ([0] * 257, list(range(257)), list(range(300, 557)), B.TFPA_ECAPACITY)]
    for ks, src, dst, code in bad_keep:
        with B.record_launches() as rec:
            with pytest.raises(B.TfpaError) as e:
                B.tfpa_keep_kv(c, segs, ks, src, dst)
        assert e.value.code == code and rec == []
    with B.record_launches() as rec:
        B.tfpa_keep_kv(c, segs, [0, 0, 1], [3, 2, 7], [2, 1, 8])
    assert [(r["kind"], r["rows"], r["grid"]) for r in rec] == [("keep", 3, 8)]


def test_planning_from_two_host_threads_at_once():
    """Dry-run calls from two threads at once plan the same launches as one
    thread alone (each thread builds its parameters in its own buffers)."""
    import threading
    c = _cache()
    segs_a = [B.Seg(40000 + 37 * i, page_table=3 * FAKE) for i in range(6)]
    segs_b = [B.Seg(9000, page_table=3 * FAKE), B.Seg(700, k_slab=8 * FAKE, v_slab=9 * FAKE,
                                                    slab_cap=768)]
    args_a = (np.repeat(np.arange(6), 3), np.concatenate([np.arange(L - 3, L) for L in
                                                          (40000 + 37 * i for i in range(6))]))
    args_b = (np.array([0] * 20 + [1]), np.array(list(range(8980, 9000)) + [699]))

    def call(segs, rs, rp):
        B.tfpa_decode(c, segs, 4 * FAKE, rs, rp, 0.088, B.Scratch(5 * FAKE, 6 * FAKE, 16),
                      7 * FAKE, stream=0)

    with B.record_launches() as rec:
        call(segs_a, *args_a)
    alone_a = list(rec)
    with B.record_launches() as rec:
        call(segs_b, *args_b)
    alone_b = list(rec)

    def worker(segs, args, n):
        for _ in range(n):
            call(segs, *args)

    with B.record_launches() as rec:
        ts = [threading.Thread(target=worker, args=(segs_a, args_a, 200)),
              threading.Thread(target=worker, args=(segs_b, args_b, 200))]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
    # every launch of both threads was recorded; the multiset equals 200 of each alone
    key = lambda r: tuple(sorted(r.items()))
    want = sorted([key(r) for r in alone_a] * 200 + [key(r) for r in alone_b] * 200)
    assert sorted(key(r) for r in rec) == want


def test_plans_hold_the_direct_calls_launches():
    """A plan records the same launches as the direct calls (at planning
    time), holds them until cleared, and a failing planning call leaves it
    as it was."""
    c = _cache()
    segs = [B.Seg(40000, page_table=3 * FAKE), B.Seg(700, k_slab=8 * FAKE, v_slab=9 * FAKE,
                                                     slab_cap=768)]
    rs = np.array([0] * 20 + [1])
    rp = np.array(list(range(39980, 40000)) + [699])
    sc = B.Scratch(5 * FAKE, 6 * FAKE, 16)
    with B.record_launches() as direct:
        B.tfpa_write_kv(c, segs, 4 * FAKE, 5 * FAKE, rs, rp, stream=0)
        B.tfpa_decode(c, segs, 4 * FAKE, rs, rp, 0.088, sc, 7 * FAKE, stream=0)
    plan = B.Plan()
    with B.record_launches() as planned:
        plan.write_kv(c, segs, 4 * FAKE, 5 * FAKE, rs, rp)
        plan.decode(c, segs, 4 * FAKE, rs, rp, 0.088, sc, 7 * FAKE)
        plan.launch(stream=0)                       # dry run: nothing is enqueued or recorded
    assert planned == direct
    assert len(plan) == len(direct)
    with B.record_launches():
        with pytest.raises(B.TfpaError) as e:
            plan.decode(c, segs, 4 * FAKE, rs, np.full(21, 40000), 0.088, sc, 7 * FAKE)
    assert e.value.code == B.TFPA_ERANGE
    assert len(plan) == len(direct)                 # the failed call appended nothing
    plan.clear()
    assert len(plan) == 0


def test_device_mode_plans_keep_their_shape_as_lengths_grow():
    """Device mode: the launches' lengths, splits and CTA ranges go to the
    packed data, not to the launch shape, so plans of a growing decode loop
    hash alike while their packed data differ; the decode grid is one CTA per
    SM whatever the work; rows for the tensor-core verify path, a buffer too
    small and a mode switch on a non-empty plan are refused."""
    torch = pytest.importorskip("torch")
    c = _cache()
    sc = B.Scratch(5 * FAKE, 6 * FAKE, 16)
    dyn = torch.zeros(1 << 16, dtype=torch.uint8)     # never dereferenced while planning

    def plan_at(plan, n):
        segs = [B.Seg(n, page_table=3 * FAKE), B.Seg(n, k_slab=8 * FAKE, v_slab=9 * FAKE,
                                                     slab_cap=2048)]
        rs, rp = np.array([0, 1]), np.array([n - 1, n - 1])
        plan.clear()
        with B.record_launches() as rec:
            plan.write_kv(c, segs, 4 * FAKE, 5 * FAKE, rs, rp)
            plan.decode(c, segs, 4 * FAKE, rs, rp, 0.088, sc, 7 * FAKE)
        return rec

    plan = B.Plan()
    plan.set_device(dyn)
    shapes, packs = [], []
    for n in (1020, 1024, 1025, 1300):           # 1025 crosses a split boundary
        rec = plan_at(plan, n)
        assert [r["kind"] for r in rec] == ["write_kv", "partial", "merge"]
        assert rec[1]["grid"] == 152             # one CTA per SM, not min(items, SMs)
        shapes.append(plan.shape())
        h = torch.zeros(plan.dyn_bytes(), dtype=torch.uint8)
        plan.pack(h)
        packs.append(h.numpy().copy())
        # the write launch's slot comes first: its first run's pos0 (after
        # three pointers, row0 and nrows) is the row's position
        assert int(packs[-1][32:36].view(np.int32)[0]) == n - 1
    assert len(set(shapes)) == 1
    assert len({p.tobytes() for p in packs}) == 4
    assert plan.dyn_bytes() % 16 == 0 and plan.dyn_bytes() > 0

    # parameter mode: the same calls size the decode grid by their work
    p2 = B.Plan()
    assert plan_at(p2, 1020)[1]["grid"] < 152
    with pytest.raises(B.TfpaError) as e:
        p2.pack(torch.zeros(64, dtype=torch.uint8))
    assert e.value.code == B.TFPA_EINVAL
    with pytest.raises(B.TfpaError) as e:         # not on a plan that holds launches
        p2.set_device(dyn)
    assert e.value.code == B.TFPA_EINVAL

    # a buffer too small: the call fails and the plan stays as it was
    p3 = B.Plan()
    p3.set_device(dyn[:4096])
    segs = [B.Seg(1000, page_table=3 * FAKE)]
    with B.record_launches():
        p3.write_kv(c, segs, 4 * FAKE, 5 * FAKE, np.array([0]), np.array([999]))
        used = p3.dyn_bytes()
        with pytest.raises(B.TfpaError) as e:
            p3.decode(c, segs, 4 * FAKE, np.array([0]), np.array([999]), 0.088, sc, 7 * FAKE)
    assert e.value.code == B.TFPA_ECAPACITY
    assert len(p3) == 1 and p3.dyn_bytes() == used
    with pytest.raises(B.TfpaError) as e:
        p3.pack(torch.zeros(used - 16, dtype=torch.uint8))
    assert e.value.code == B.TFPA_ECAPACITY

    # sixteen rows of one stream (four m-tiles with four heads per kv head)
    # take the tensor-core verify path, whose grid follows the lengths
    p4 = B.Plan()
    p4.set_device(dyn)
    with B.record_launches():
        with pytest.raises(B.TfpaError) as e:
            p4.decode(c, segs, 4 * FAKE, np.zeros(16), np.arange(984, 1000), 0.088, sc,
                      7 * FAKE)
    assert e.value.code == B.TFPA_EINVAL and len(p4) == 0 and p4.dyn_bytes() == 0


def test_arrival_counters_fold_the_merge_into_the_partial_launch():
    """With arrival counters a slice of plain decode-path rows over streams
    of at most 4 splits runs one partial launch and no merge; longer
    streams, tree rows, device-mode plans and slices with tensor-core verify
    rows keep the separate merge."""
    c = _cache()
    short = [B.Seg(1024, page_table=3 * FAKE), B.Seg(700, k_slab=8 * FAKE, v_slab=9 * FAKE,
                                                     slab_cap=768)]
    long = [B.Seg(1025, page_table=3 * FAKE)] + short[1:]
    plain = B.Scratch(5 * FAKE, 6 * FAKE, 16)
    counted = B.Scratch(5 * FAKE, 6 * FAKE, 16, 32, 10 * FAKE)

    def kinds(sc, segs, rs, rp, anc=None):
        with B.record_launches() as rec:
            if anc is None:
                B.tfpa_decode(c, segs, 4 * FAKE, rs, rp, 0.088, sc, 7 * FAKE, stream=0)
            else:
                B.tfpa_decode_tree(c, segs, 4 * FAKE, rs, rp, anc, 0.088, sc, 7 * FAKE, stream=0)
        return [r["kind"] for r in rec]

    rs = np.array([0, 1])
    assert kinds(plain, short, rs, np.array([1023, 699])) == ["partial", "merge"]
    assert kinds(counted, short, rs, np.array([1023, 699])) == ["partial"]
    assert kinds(counted, long, rs, np.array([1024, 699])) == ["partial", "merge"]
    assert kinds(counted, short, rs, np.array([1023, 699]), anc=11 * FAKE) == ["partial", "merge"]
    # 20 rows of stream 0 (verify path) + 1 of stream 1, 16-row slices
    rs = np.array([0] * 20 + [1])
    rp = np.array(list(range(1004, 1024)) + [699])
    assert kinds(counted, short, rs, rp) == ["verify", "merge", "partial", "verify", "merge"]
    rs, rp = np.array([0] * 3 + [1]), np.array([1021, 1022, 1023, 699])
    assert kinds(counted, short, rs, rp) == ["partial"]
    # a plan in device mode keeps the merge launch
    torch = pytest.importorskip("torch")
    plan = B.Plan()
    plan.set_device(torch.zeros(1 << 16, dtype=torch.uint8))
    with B.record_launches() as rec:
        plan.decode(c, short, 4 * FAKE, np.array([0, 1]), np.array([1023, 699]), 0.088, counted,
                    7 * FAKE)
    assert [r["kind"] for r in rec] == ["partial", "merge"]


def test_plan_capture_and_replay_follow_the_shape():
    """tfpa_plan_capture keeps the plan's shape; tfpa_plan_replay refuses a
    plan that was never captured or whose shape has changed since, and
    accepts a re-planned step of the same shape (dry run: no CUDA calls)."""
    torch = pytest.importorskip("torch")
    c = _cache()
    sc = B.Scratch(5 * FAKE, 6 * FAKE, 16)
    dyn = torch.zeros(1 << 16, dtype=torch.uint8)

    def plan_at(plan, n, rows=1):
        segs = [B.Seg(n, page_table=3 * FAKE)]
        rs, rp = np.zeros(rows), np.arange(n - rows, n)
        plan.clear()
        plan.write_kv(c, segs, 4 * FAKE, 5 * FAKE, rs, rp)
        plan.decode(c, segs, 4 * FAKE, rs, rp, 0.088, sc, 7 * FAKE)

    plan = B.Plan()
    plan.set_device(dyn)
    with B.record_launches():
        plan_at(plan, 3000)
        with pytest.raises(B.TfpaError) as e:
            plan.replay(stream=0)
        assert e.value.code == B.TFPA_EINVAL
        plan.capture(before=[(8 * FAKE, 9 * FAKE, 4096)], after=[(10 * FAKE, 7 * FAKE, 8192)],
                     stream=0)
        plan.replay(stream=0)
        plan_at(plan, 3001)                       # one position longer: same shape
        plan.replay(stream=0)
        plan_at(plan, 3001, rows=2)               # another row: the graph no longer fits
        with pytest.raises(B.TfpaError) as e:
            plan.replay(stream=0)
        assert e.value.code == B.TFPA_EINVAL
        plan.clear()
        with pytest.raises(B.TfpaError) as e:     # nothing to capture
            plan.capture(stream=0)
        assert e.value.code == B.TFPA_EINVAL


def test_append_stores_in_the_partial_kernel_where_it_can():
    """tfpa_decode_append: narrow runs, one per segment, run the partial and
    merge launches only (the partial kernel stores the rows); a wide run or
    a segment with two runs adds one KV write launch ahead of the decode."""
    c = _cache()
    segs = [B.Seg(4000, page_table=3 * FAKE), B.Seg(700, k_slab=8 * FAKE, v_slab=9 * FAKE,
                                                    slab_cap=768)]
    sc = B.Scratch(5 * FAKE, 6 * FAKE, 64, 32)

    def kinds(rs, rp):
        with B.record_launches() as rec:
            B.tfpa_decode_append(c, segs, 10 * FAKE, 11 * FAKE, 4 * FAKE, rs, rp, 0.088, sc,
                                 7 * FAKE, stream=0)
        return [r["kind"] for r in rec]

    assert kinds(np.array([0, 1]), np.array([3999, 699])) == ["partial", "merge"]
    assert kinds(np.array([0] * 4 + [1]), np.array([3996, 3997, 3998, 3999, 699])) == [
        "partial", "merge"]
    # 20 rows of stream 0: the tensor-core verify path
    assert kinds(np.array([0] * 20 + [1]), np.array(list(range(3980, 4000)) + [699])) == [
        "write_kv", "partial", "verify", "merge"]
    # stream 0 in two runs (positions not consecutive)
    assert kinds(np.array([0, 0, 1]), np.array([3990, 3999, 699])) == [
        "write_kv", "partial", "merge"]
    plan = B.Plan()
    with B.record_launches() as rec:
        plan.decode_append(c, segs, 10 * FAKE, 11 * FAKE, 4 * FAKE, np.array([0, 1]),
                           np.array([3999, 699]), 0.088, sc, 7 * FAKE)
    assert [r["kind"] for r in rec] == ["partial", "merge"]
    with B.record_launches() as rec:
        with pytest.raises(B.TfpaError) as e:
            B.tfpa_decode_append(c, segs, 10 * FAKE + 8, 11 * FAKE, 4 * FAKE, np.array([0]),
                                 np.array([3999]), 0.088, sc, 7 * FAKE, stream=0)
    assert e.value.code == B.TFPA_EINVAL and rec == []


@pytest.mark.parametrize("pages,splits", [(1, 1), (24, 1), (25, 2), (59, 3), (168, 7),
                                          (169, 7), (200, 7), (256, 7), (1024, 7)])
def test_verify_splits_follow_the_stream_length(pages, splits):
    """Verify tiles split a stream into pieces of at least 24 pages and at
    most 7 pieces; the count (kv heads x row tiles x splits in the launch
    record) depends on the stream's length only."""
    c = _cache()
    L = pages * 256
    rows = 16                                       # 64 vectors a kv head: one row tile
    segs = [B.Seg(L, page_table=3 * FAKE)]
    with B.record_launches() as rec:
        B.tfpa_decode(c, segs, 4 * FAKE, np.zeros(rows), np.arange(L - rows, L), 0.088,
                      B.Scratch(5 * FAKE, 6 * FAKE, 128), 7 * FAKE)
    v = [r for r in rec if r["kind"] == "verify"]
    assert len(v) == 1
    assert v[0]["items"] == 8 * splits
    pps = max(24, -(-pages // 7))
    assert splits == -(-pages // pps)
    ns = B.tfpa_row_splits(c, segs, np.zeros(rows), np.arange(L - rows, L))
    assert ns.tolist() == [splits] * rows


def test_row_splits_give_each_row_its_kernels_split_count():
    """tfpa_row_splits: a narrow run keeps tfpa_num_splits, a run of 49 or
    more query vectors per kv head the verify path's count, whatever the
    order of the rows in the call."""
    c = _cache()
    segs = [B.Seg(65536, page_table=3 * FAKE), B.Seg(8192, page_table=3 * FAKE)]
    rs = np.array([1] + [0] * 13 + [1], np.int32)             # 13 rows: 52 vectors
    rp = np.concatenate([[100], np.arange(65536 - 13, 65536), [8191]]).astype(np.int32)
    ns = B.tfpa_row_splits(c, segs, rs, rp)
    assert ns.tolist() == [B.tfpa_num_splits(8192)] + [7] * 13 + [B.tfpa_num_splits(8192)]
    # twelve rows (48 vectors) stay on the decode kernel
    ns = B.tfpa_row_splits(c, segs, np.zeros(12), np.arange(65536 - 12, 65536))
    assert ns.tolist() == [B.tfpa_num_splits(65536)] * 12
    with pytest.raises(B.TfpaError):
        B.tfpa_row_splits(c, segs, [2], [0])
