"""The tensor-core verify path on the GPU: decode runs of 49 or more query
vectors per kv head (13+ rows at four query heads per kv head) run on the
prefill kernel in verify mode and leave split partials for the merge.

Against the oracle: several key splits per stream next to a narrow run in the
same call, and group sizes that leave a slot empty (three heads per kv head),
need two pair groups (eight) or fall back to the decode kernel (one).
Bitwise: a wide run batched with others equals it alone, paged equals slab,
slices of any size equal one launch, and the partials plus a separate merge
(with tfpa_row_splits' counts) equal tfpa_decode."""

import numpy as np
import pytest
import torch

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, bits, fp8_scales
from tests.test_gpu_edges import _check, _make

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("paged", [(True, False), (False, True)])
def test_several_splits_next_to_a_narrow_run(kv, paged):
    # 15,000 keys: 59 pages, three verify splits (24, 24, 11 pages); the
    # 1-row run of stream 1 stays on the decode kernel in the same call
    lengths = [15000, 5000]
    rs = [0] * 20 + [1]
    rp = list(range(14980, 15000)) + [4999]
    _check(_make(lengths, list(paged), rs, rp, kv=kv, seed=611), f"{kv} splits {paged}")


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("hq,hkv", [(6, 2), (16, 2), (8, 8), (4, 1)])
def test_wide_runs_at_other_group_sizes(hq, hkv, kv):
    # 60 rows: wide at every group size (60 query vectors per kv head at one)
    L = 4700
    rs = [0] * 60
    rp = list(range(L - 60, L))
    _check(_make([L], [True], rs, rp, hq, hkv, kv, seed=612), f"G={hq // hkv} {kv}")


def _wide_case(kv, seed=613):
    lengths = [6100, 3000, 800]
    rs = np.array([0] * 17 + [1] * 30 + [2], np.int32)
    rp = np.array(list(range(6083, 6100)) + list(range(2970, 3000)) + [799], np.int32)
    return _make(lengths, [True, True, False], rs, rp, kv=kv, seed=seed, slack=9)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_wide_batched_equals_alone_bitwise(kv):
    w = _wide_case(kv)
    scales = fp8_scales(w) if kv == "fp8" else None
    g = GpuCase(w, scales)
    q = g.q()
    full, lfull = g.decode(q, w.row_seg, w.row_pos)
    for s in range(len(w.streams)):
        sel = np.flatnonzero(w.row_seg == s)
        alone, lalone = g.decode(q[sel], np.zeros(len(sel), np.int32), w.row_pos[sel],
                                 segs=[g.segs[s]])
        assert np.array_equal(bits(alone), bits(full[sel])), f"stream {s}"
        assert torch.equal(lalone, lfull[sel])


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_wide_paged_equals_slab_and_slices_bitwise(kv):
    w = _wide_case(kv, seed=614)
    scales = fp8_scales(w) if kv == "fp8" else None
    lengths = [st.seq_len for st in w.streams]
    tables = wl.permuted_tables(lengths, [True] * len(lengths), w.num_pages + 40, 4243)
    w2 = wl.Workload(w.name, w.hq, w.hkv, w.kv_dtype, w.num_pages + 40, w.streams, w.row_seg,
                     w.row_pos, w.seed)
    paged = GpuCase(w2, scales, all_paged=True, tables=tables)
    slab = GpuCase(w2, scales, all_paged=False)
    a, la = paged.decode(paged.q(), w.row_seg, w.row_pos)
    b, lb = slab.decode(slab.q(), w.row_seg, w.row_pos)
    assert np.array_equal(bits(a), bits(b))
    assert torch.equal(la, lb)
    for cap in (5, 16, 33):
        c, lc = slab.decode(slab.q(), w.row_seg, w.row_pos, cap_rows=cap)
        assert np.array_equal(bits(b), bits(c)), f"slices of {cap}"
        assert torch.equal(lb, lc)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_partial_and_merge_with_row_splits_equal_decode(kv):
    """tfpa_decode_partial then tfpa_merge, given each row's split count from
    tfpa_row_splits, give tfpa_decode's bytes for a call whose wide run (20
    rows, three verify splits) sits beside a narrow one (decode splits)."""
    lengths = [15000, 5000]
    rs = [0] * 20 + [1]
    rp = list(range(14980, 15000)) + [4999]
    w = _make(lengths, [True, False], rs, rp, kv=kv, seed=612)
    g = GpuCase(w, fp8_scales(w) if kv == "fp8" else None)
    q = g.q()
    ref, ref_lse = g.decode(q, w.row_seg, w.row_pos)
    ns = B.tfpa_row_splits(g.cache, g.segs, w.row_seg, w.row_pos)
    assert ns.tolist() == [3] * 20 + [B.tfpa_num_splits(5000)]
    sc = B.make_scratch(w.rows, w.hq, fused_merge=False)
    out = torch.empty_like(ref)
    lse = torch.empty_like(ref_lse)
    B.tfpa_decode_partial(g.cache, g.segs, q, w.row_seg, w.row_pos, w.softmax_scale, sc)
    B.tfpa_merge(sc, w.hq, ns, out, lse)
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), bits(ref))
    assert torch.equal(lse, ref_lse)
    assert int(g.err.item()) == 0
