"""Pins of the oracle's draft-tree verify rows (ancestor masks).

The visibility each test expects is built here from the tree itself, by
walking parent links, and never from the mask bits; so these tests pin the
oracle's reading of a mask and the workload module's encoding of a tree
together.  Reading (the pages name the per-row ancestor table but not its
format): bit d of a row's mask says whether the key d positions back is
visible; keys more than 63 back always are, later keys never are.
"""

import numpy as np
import pytest
import torch

from oracle import attention
from paged_kv_cache_235_gb300 import workloads as wl
from tests.oracle_cases import build_oracle_cache


def _tree_case(L, nodes, parents, kv="bf16", seed=31, hq=8, hkv=2):
    """One paged stream of length L whose last ``nodes`` positions hold the tree."""
    num_pages = (L + 255) // 256 + 2
    tables = wl.permuted_tables([L], [True], num_pages, seed)
    rs, rp = wl.decode_rows([L], nodes)
    w = wl.Workload("tree", hq, hkv, kv, num_pages, [wl.Stream(L, True, tables[0])], rs, rp, seed)
    w.row_anc = np.array(wl.tree_masks(parents), dtype=np.uint64)
    return w


def _visible_by_walking(L, nodes, parents):
    """[nodes][L] boolean: node i sees the prefix, its ancestors and itself."""
    base = L - nodes
    vis = np.zeros((nodes, L), dtype=bool)
    for i in range(nodes):
        vis[i, :base] = True
        a = i
        while a >= 0:
            vis[i, base + a] = True
            a = parents[a]
    return vis


def _sdpa_with_mask(w, cache, segs, vis):
    """float64 torch SDPA with an explicit boolean mask, per kv head group."""
    from oracle.kvcache import bf16_to_f64, gather
    q = torch.from_numpy(bf16_to_f64(w.q_bits()))          # [rows][hq][d]
    G = w.hq // w.hkv
    L = w.streams[0].seq_len
    out = torch.zeros(w.rows, w.hq, w.d, dtype=torch.float64)
    for g in range(w.hkv):
        K, V = gather(cache, segs[0], g, L)
        K, V = torch.from_numpy(K), torch.from_numpy(V)
        for h in range(g * G, (g + 1) * G):
            o = torch.nn.functional.scaled_dot_product_attention(
                q[:, h][None], K[None], V[None], attn_mask=torch.from_numpy(vis)[None],
                scale=w.softmax_scale)
            out[:, h] = o[0]
    return out.numpy()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("nodes,L", [(20, 700), (64, 900), (9, 12)])
def test_tree_matches_sdpa_with_walked_mask(kv, nodes, L):
    parents = wl.random_tree(nodes, seed=5 + nodes)
    w = _tree_case(L, nodes, parents, kv)
    cache, segs = build_oracle_cache(w)
    got, _ = attention.attend(cache, segs, w.q_bits(), w.row_seg, w.row_pos,
                              w.softmax_scale, row_anc=w.row_anc)
    ref = _sdpa_with_mask(w, cache, segs, _visible_by_walking(L, nodes, parents))
    assert np.max(np.abs(got - ref)) < 1e-12


def test_all_ones_mask_is_the_causal_row():
    w = _tree_case(600, 8, [-1, 0, 1, 2, 3, 4, 5, 6])     # a chain
    cache, segs = build_oracle_cache(w)
    assert all(int(m) == attention.ALL_VISIBLE for m in w.row_anc)
    a, la = attention.attend(cache, segs, w.q_bits(), w.row_seg, w.row_pos, w.softmax_scale,
                             row_anc=w.row_anc)
    b, lb = attention.attend(cache, segs, w.q_bits(), w.row_seg, w.row_pos, w.softmax_scale)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_star_tree_closed_form():
    """Leaf i of a star sees the prefix, the root and itself: plain softmax
    over exactly those keys, written out here."""
    L, nodes = 400, 6
    w = _tree_case(L, nodes, [-1] + [0] * (nodes - 1))
    cache, segs = build_oracle_cache(w)
    got, lse = attention.attend(cache, segs, w.q_bits(), w.row_seg, w.row_pos,
                                w.softmax_scale, row_anc=w.row_anc)
    from oracle.kvcache import bf16_to_f64, gather
    q = bf16_to_f64(w.q_bits())
    base = L - nodes
    G = w.hq // w.hkv
    for i in range(1, nodes):
        keys = list(range(base + 1)) + [base + i]
        for g in range(w.hkv):
            K, V = gather(cache, segs[0], g, L)
            for h in range(g * G, (g + 1) * G):
                s = w.softmax_scale * (K[keys] @ q[i, h])
                e = np.exp(s - s.max())
                assert np.max(np.abs(got[i, h] - (e @ V[keys]) / e.sum())) < 1e-12
                assert abs(lse[i, h] - (s.max() + np.log(e.sum()))) < 1e-12


@pytest.mark.parametrize("pps", [1, 2, 3])
def test_tree_partials_merge_equal_one_pass(pps):
    nodes, L = 40, 1100
    w = _tree_case(L, nodes, wl.random_tree(nodes, seed=8), "fp8")
    cache, segs = build_oracle_cache(w)
    one, lse1 = attention.attend(cache, segs, w.q_bits(), w.row_seg, w.row_pos,
                                 w.softmax_scale, row_anc=w.row_anc)
    m, l, o, _ = attention.attend_partials(cache, segs, w.q_bits(), w.row_seg, w.row_pos,
                                           w.softmax_scale, pps, row_anc=w.row_anc)
    two, lse2 = attention.merge(m, l, o)
    assert np.max(np.abs(one - two)) < 1e-12 and np.max(np.abs(lse1 - lse2)) < 1e-12


def test_tree_masks_encoding_by_hand():
    # root, two children of the root, one grandchild under node 1
    m = wl.tree_masks([-1, 0, 0, 1])
    full = (1 << 64) - 1
    assert m[0] == full and m[1] == full
    assert m[2] == full & ~(1 << 1)          # node 2 does not see its sibling node 1
    assert m[3] == full & ~(1 << 1)          # node 3 does not see node 2 (one back)


def test_mask_must_show_the_rows_own_key():
    with pytest.raises(ValueError):
        attention.visible_keys(100, attention.ALL_VISIBLE & ~1)


def test_planted_off_by_one_mask_is_caught(monkeypatch):
    """A plausible mistake (bit d read as the key d + 1 back) fails the pin."""
    def shifted(p, anc=attention.ALL_VISIBLE):
        anc = int(anc)
        keys = [j for j in range(max(0, p - 63), p + 1)
                if j == p or (anc >> (p - j - 1)) & 1]
        return np.concatenate([np.arange(0, max(0, p - 63)), np.asarray(keys)]).astype(np.int64)
    monkeypatch.setattr(attention, "visible_keys", shifted)
    with pytest.raises(AssertionError):
        test_tree_matches_sdpa_with_walked_mask("bf16", 20, 700)
