"""Draft-tree verify rows on the GPU (tfpa_decode_tree) against the oracle.

Also the bitwise properties: 7-row slices equal one launch (so the ancestor
table is shifted with the other row tables), all-ones masks equal
tfpa_decode, and a planted control (the table handed over one row off, as an
unshifted slice would see it) comes out red.
"""

import numpy as np
import pytest

from oracle import attention
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, assert_close, bits, fp8_scales, to_f64
from tests.oracle_cases import build_oracle_cache

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp8": 3e-2}


def _small(kv, nodes=20, seq_len=1300, n_streams=3, seed=1235):
    return wl.tree_verify(seed, seq_len=seq_len, n_streams=n_streams, nodes=nodes,
                          kv_dtype=kv, slack_pages=5)


def _oracle(w, scales, rows=None):
    cache, segs = build_oracle_cache(w, *(scales or (None, None)))
    sel = slice(None) if rows is None else rows
    return attention.attend(cache, segs, w.q_bits()[sel], w.row_seg[sel], w.row_pos[sel],
                            w.softmax_scale, row_anc=w.row_anc[sel])


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("nodes,seq_len", [(20, 1300), (64, 900), (33, 40)])
def test_tree_verify_matches_oracle(kv, nodes, seq_len):
    w = _small(kv, nodes, seq_len)
    scales = fp8_scales(w) if kv == "fp8" else None
    g = GpuCase(w, scales)
    out, lse = g.decode_tree(g.q(), w.row_seg, w.row_pos, w.row_anc)
    ref, ref_lse = _oracle(w, scales)
    assert_close(to_f64(out), ref, TOL[kv], f"tree {nodes} nodes")
    assert_close(to_f64(lse), ref_lse, 1e-3, "tree lse")
    assert int(g.err.item()) == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_slices_equal_one_launch_and_unshifted_table_is_red(kv):
    w = _small(kv)
    scales = fp8_scales(w) if kv == "fp8" else None
    g = GpuCase(w, scales)
    q = g.q()
    one, _ = g.decode_tree(q, w.row_seg, w.row_pos, w.row_anc)
    sliced, _ = g.decode_tree(q, w.row_seg, w.row_pos, w.row_anc, cap_rows=7)
    assert np.array_equal(bits(one), bits(sliced))
    # planted control: each row handed the mask of the row before it
    wrong, _ = g.decode_tree(q, w.row_seg, w.row_pos, np.roll(w.row_anc, 1))
    assert not np.array_equal(bits(one), bits(wrong))


def test_all_ones_masks_equal_tfpa_decode():
    w = _small("bf16")
    g = GpuCase(w)
    q = g.q()
    a, la = g.decode_tree(q, w.row_seg, w.row_pos, np.full(w.rows, (1 << 64) - 1, np.uint64))
    b, lb = g.decode(q, w.row_seg, w.row_pos)
    assert np.array_equal(bits(a), bits(b))
    assert np.array_equal(la.cpu().numpy(), lb.cpu().numpy())


@pytest.mark.slow
def test_full_size_tree_verify_sampled_rows():
    w = wl.tree_verify()
    scales = fp8_scales(w)
    g = GpuCase(w, scales)
    out, lse = g.decode_tree(g.q(), w.row_seg, w.row_pos, w.row_anc)
    rows = np.array([0, 5, 15, 16, 47, 100, 127])
    ref, ref_lse = _oracle(w, scales, rows)
    assert_close(to_f64(out)[rows], ref, TOL["fp8"], "full-size tree rows")
    assert_close(to_f64(lse)[rows], ref_lse, 1e-3, "full-size tree lse")
    assert int(g.err.item()) == 0
