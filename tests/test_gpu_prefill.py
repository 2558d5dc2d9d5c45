"""Prompt-chunk attention (tcgen05) on the GPU against the oracle, and the
bitwise invariants: 128-row slices == one launch == the contiguous path."""

import numpy as np
import pytest
import torch

from oracle import attention
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, assert_close, bits, fp8_scales, to_f64
from tests.oracle_cases import build_oracle_cache

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp8": 3e-2}


def _case(w, **kw):
    scales = fp8_scales(w) if w.kv_dtype == "fp8" else None
    return GpuCase(w, scales, **kw), scales


def _oracle(w, rows=None, scales=None):
    cache, segs = build_oracle_cache(w, *(scales or (None, None)))
    q = w.q_bits()
    rs, rp = w.row_seg, w.row_pos
    if rows is not None:
        q, rs, rp = q[rows], rs[rows], rp[rows]
    return attention.attend(cache, segs, q, rs, rp, w.softmax_scale)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("prefix,chunk", [(300, 257), (0, 300), (256, 128), (1000, 1), (77, 130)])
def test_prompt_chunk_matches_oracle(prefix, chunk, kv):
    w = wl.prompt_chunk(seed=300 + prefix + chunk, prefix=prefix, chunk=chunk, slack_pages=3,
                        kv_dtype=kv)
    g, scales = _case(w)
    out, lse = g.prefill(g.q(), w.row_seg, w.row_pos)
    ref, ref_lse = _oracle(w, scales=scales)
    assert_close(to_f64(out), ref, TOL[kv], f"prefill {kv} {prefix}+{chunk}")
    assert_close(to_f64(lse), ref_lse, 1e-3, "lse")
    assert int(g.err.item()) == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_prompt_chunk_slices_equal_one_launch_and_contiguous(kv):
    w = wl.prompt_chunk(seed=1235, prefix=300, chunk=257, slack_pages=3, kv_dtype=kv)
    g, scales = _case(w)
    q = g.q()
    one, l1 = g.prefill(q, w.row_seg, w.row_pos)
    sl, l2 = g.prefill(q, w.row_seg, w.row_pos, max_rows=128)
    assert np.array_equal(bits(one), bits(sl))
    assert torch.equal(l1, l2)
    gc = GpuCase(w, scales, all_paged=False)
    cont, l3 = gc.prefill(gc.q(), w.row_seg, w.row_pos)
    assert np.array_equal(bits(one), bits(cont))
    assert torch.equal(l1, l3)


def test_two_prompt_chunks_in_one_call():
    lengths = [700, 450]
    tables = wl.permuted_tables(lengths, [True, False], 8, 91)
    streams = [wl.Stream(700, True, tables[0]), wl.Stream(450, False, None, 512)]
    rs = np.array([0] * 200 + [1] * 150, np.int32)
    rp = np.concatenate([np.arange(500, 700), np.arange(300, 450)]).astype(np.int32)
    w = wl.Workload("two_chunks", 32, 8, "bf16", 8, streams, rs, rp, 92)
    g = GpuCase(w)
    q = g.q()
    out, _ = g.prefill(q, rs, rp)
    ref, _ = _oracle(w)
    assert_close(to_f64(out), ref, 1e-2, "two chunks")
    # each chunk alone gives the same bytes
    for s in range(2):
        sel = np.flatnonzero(rs == s)
        alone, _ = g.prefill(q[sel], np.zeros(len(sel), np.int32), rp[sel], segs=[g.segs[s]])
        assert np.array_equal(bits(alone), bits(out[sel]))


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_prefill_equals_decode_within_tolerance(kv):
    """The prompt tiles and the decode partials compute the same attention."""
    w = wl.prompt_chunk(seed=1235, prefix=300, chunk=257, slack_pages=3, kv_dtype=kv)
    g, _ = _case(w)
    q = g.q()
    a, _ = g.prefill(q, w.row_seg, w.row_pos)
    b, _ = g.decode(q, w.row_seg, w.row_pos, cap_rows=64)
    assert_close(to_f64(a), to_f64(b), TOL[kv], "prefill vs decode")


def test_swapped_table_control_is_red_for_prompt_rows():
    w = wl.small("prompt_chunk")              # pages 0, 1 hold the prefix; 2 the chunk
    g = GpuCase(w)
    t = w.streams[0].page_table.copy()
    t[[0, 2]] = t[[2, 0]]
    from paged_kv_cache_235_gb300 import binding as B
    bad = B.Seg(w.streams[0].seq_len, page_table=torch.from_numpy(t).cuda())
    out, _ = g.prefill(g.q(), w.row_seg, w.row_pos, segs=[bad])
    ref, _ = _oracle(w)
    with pytest.raises(AssertionError):
        assert_close(to_f64(out), ref, 1e-2, "swapped")


@pytest.mark.slow
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_prompt_chunk_full_size_sampled(kv):
    """28,672-position paged prefix + 4,096 causal rows, as the bench runs it;
    a sample of rows (first, last, and across tiles) against the oracle."""
    from tests.test_gpu_full import oracle_stream
    w = wl.prompt_chunk(kv_dtype=kv)
    g, scales = _case(w)
    q = g.q()
    out, lse = g.prefill(q, w.row_seg, w.row_pos)
    rows = np.array([0, 1, 127, 128, 1000, 2047, 2048, 4000, 4094, 4095])
    ref, ref_lse = oracle_stream(w, 0, rows, scales)
    assert_close(to_f64(out[rows]), ref, TOL[kv], "full prefill")
    assert_close(to_f64(lse[rows]), ref_lse, 1e-3, "full prefill lse")
    assert int(g.err.item()) == 0


@pytest.mark.slow
@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_257_row_chunk_on_the_full_prefix_slices_bitwise(kv):
    """A 257-row chunk on the 28,672-position paged prefix (PR #1355, "Follow-up
    checks": the 257-row chunk run as 128-row partial slices): 128 + 128 + 1
    slices equal one launch, and both equal the contiguous path, bit for bit;
    at this length every tile splits its key range over the cluster's two
    CTAs and crosses many page edges.  Sampled rows against the oracle."""
    from tests.test_gpu_full import oracle_stream
    w = wl.prompt_chunk(prefix=28672, chunk=257, kv_dtype=kv)
    g, scales = _case(w)
    q = g.q()
    one, l1 = g.prefill(q, w.row_seg, w.row_pos)
    sl, l2 = g.prefill(q, w.row_seg, w.row_pos, max_rows=128)
    assert np.array_equal(bits(one), bits(sl))
    assert torch.equal(l1, l2)
    gc = GpuCase(w, scales, all_paged=False)
    cont, l3 = gc.prefill(gc.q(), w.row_seg, w.row_pos)
    assert np.array_equal(bits(one), bits(cont))
    assert torch.equal(l1, l3)
    rows = np.array([0, 1, 127, 128, 200, 255, 256])
    ref, ref_lse = oracle_stream(w, 0, rows, scales)
    assert_close(to_f64(one[rows]), ref, TOL[kv], "257-row chunk, full prefix")
    assert_close(to_f64(l1[rows]), ref_lse, 1e-3, "257-row chunk, full prefix, lse")
    assert int(g.err.item()) == 0 and int(gc.err.item()) == 0
