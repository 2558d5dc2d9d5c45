"""Edge cases on the GPU against the oracle: GQA group sizes, one-key and
exact-page streams, many rows per stream, non-consecutive rows, and calls that
need more than one launch (more slab streams or runs than a launch holds)."""

import numpy as np
import pytest

from oracle import attention
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, assert_close, fp8_scales, to_f64
from tests.oracle_cases import build_oracle_cache

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp8": 3e-2}


def _make(lengths, paged, rows_seg, rows_pos, hq=32, hkv=8, kv="bf16", seed=500, slack=4):
    npages = sum((L + 255) // 256 for L, p in zip(lengths, paged) if p) + slack
    tables = wl.permuted_tables(lengths, paged, npages, seed)
    streams = [wl.Stream(L, p, t, 0 if p else ((L + 255) // 256) * 256)
               for L, p, t in zip(lengths, paged, tables)]
    return wl.Workload("edge", hq, hkv, kv, npages, streams,
                       np.asarray(rows_seg, np.int32), np.asarray(rows_pos, np.int32), seed)


def _check(w, what, prefill=False, cap_rows=128):
    scales = fp8_scales(w) if w.kv_dtype == "fp8" else None
    g = GpuCase(w, scales)
    q = g.q()
    if prefill:
        out, lse = g.prefill(q, w.row_seg, w.row_pos)
    else:
        out, lse = g.decode(q, w.row_seg, w.row_pos, cap_rows=cap_rows)
    cache, segs = build_oracle_cache(w, *(scales or (None, None)))
    ref, ref_lse = attention.attend(cache, segs, w.q_bits(), w.row_seg, w.row_pos,
                                    w.softmax_scale)
    assert_close(to_f64(out), ref, TOL[w.kv_dtype], what)
    assert_close(to_f64(lse), ref_lse, 1e-3, what + " lse")
    assert int(g.err.item()) == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (6, 2), (16, 2), (4, 1)])
def test_gqa_group_sizes(hq, hkv, kv):
    lengths = [700, 300]
    rs = [0, 0, 1]
    rp = [698, 699, 299]
    _check(_make(lengths, [True, False], rs, rp, hq, hkv, kv), f"decode G={hq // hkv}")
    rs = [0] * 140
    rp = list(range(560, 700))
    _check(_make([700], [True], rs, rp, hq, hkv, kv), f"prefill G={hq // hkv}", prefill=True)


@pytest.mark.parametrize("L", [1, 2, 255, 256, 257, 511, 512, 513])
def test_stream_lengths_around_page_edges(L):
    w = _make([L, L], [True, False], [0, 1], [L - 1, L - 1])
    _check(w, f"decode L={L}")
    _check(_make([L], [True], [0] * L, list(range(L))), f"prefill L={L}", prefill=True)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_many_rows_per_stream_span_m_tiles(kv):
    # 40 verify rows x 4 heads = 160 query vectors: 10 m-tiles per kv head
    L = 900
    w = _make([L], [True], [0] * 40, list(range(L - 40, L)), kv=kv)
    _check(w, "40 rows")
    _check(w, "40 rows in slices of 7", cap_rows=7)


def test_non_consecutive_rows_of_one_stream():
    w = _make([1200, 600], [True, True], [0, 1, 0, 0, 1], [100, 599, 1199, 640, 5])
    _check(w, "scattered rows")


def test_more_slab_streams_than_one_launch_holds():
    n = 20                                            # more than 15 slab sources
    lengths = [300 + 37 * i for i in range(n)]
    w = _make(lengths, [False] * n, list(range(n)), [L - 1 for L in lengths], hq=8, hkv=2)
    _check(w, "20 slab streams")


def test_more_runs_than_one_launch_holds():
    n = 70                                            # more than 64 runs
    lengths = [200 + 11 * i for i in range(n)]
    w = _make(lengths, [True] * n, list(range(n)), [L - 1 for L in lengths], hq=8, hkv=2)
    _check(w, "70 paged streams")
