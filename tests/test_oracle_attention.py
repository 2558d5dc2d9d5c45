"""Pins of the oracle's attention against mathematics and a library routine.

Each pin is chosen so a plausible mistake in the oracle (a dropped causal
mask, a wrong GQA head mapping, an unused page table, a mis-weighted merge,
a wrong KV address) fails at least one of them; the planted-mistake tests at
the end check exactly that.
"""

import math
import os

import numpy as np
import pytest
import torch

from oracle import attention, e4m3, kvcache
from paged_kv_cache_235_gb300 import workloads as wl
from tests.oracle_cases import build_oracle_cache


def bits(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def tiny_cache(k_rows, v_rows, page_table=None, num_pages=None):
    """A bf16 cache of one stream, one kv head, from exact float rows [n][d]."""
    n, d = np.asarray(k_rows).shape
    kb, vb = bits(k_rows), bits(v_rows)
    if page_table is None:
        ks = np.zeros((1, max(256, n), d), np.uint16)
        vs = np.zeros((1, max(256, n), d), np.uint16)
        ks[0, :n], vs[0, :n] = kb, vb
        return kvcache.Cache("bf16", 1, d, None, None), [kvcache.Segment(n, k_slab=ks, v_slab=vs)]
    kp = np.zeros((num_pages, 1, 256, d), np.uint16)
    vp = np.zeros((num_pages, 1, 256, d), np.uint16)
    for i in range(n):
        kp[page_table[i // 256], 0, i % 256] = kb[i]
        vp[page_table[i // 256], 0, i % 256] = vb[i]
    return (kvcache.Cache("bf16", 1, d, kp, vp),
            [kvcache.Segment(n, page_table=np.array(page_table, np.int32))])


def _worked(golden_dir):
    cases, cur = {}, None
    with open(os.path.join(golden_dir, "attention_worked.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            tok = line.split()
            if tok[0] == "case":
                cur = cases.setdefault(tok[1], {})
            else:
                cur[tok[0]] = [float(t) for t in tok[1:]]
    return cases


def test_worked_example(golden_dir):
    cases = _worked(golden_dir)
    cache, segs = tiny_cache([[1, 0], [0, 1]], [[1, 0], [0, 1]])
    for name, q, pos in (("two_keys", [1, 0], 1), ("causal_first_row", [1, 0], 0),
                         ("two_keys_q2", [2, 0], 1)):
        out, lse = attention.attend(cache, segs, bits([[q]]), [0], [pos], 1.0)
        np.testing.assert_allclose(out[0, 0], cases[name]["out"], rtol=0, atol=1e-15)
        np.testing.assert_allclose(lse[0, 0], cases[name]["lse"][0], rtol=0, atol=1e-15)


def _sdpa_reference(cache, segs, q_bits, row_seg, row_pos, scale):
    """torch scaled_dot_product_attention in float64 with an explicit mask."""
    rows, hq, d = q_bits.shape
    q = torch.from_numpy(kvcache.bf16_to_f64(q_bits))
    out = torch.zeros(rows, hq, d, dtype=torch.float64)
    for r in range(rows):
        s, p = int(row_seg[r]), int(row_pos[r])
        L = segs[s].seq_len
        K = torch.stack([torch.from_numpy(kvcache.gather(cache, segs[s], g, L)[0]) for g in range(cache.hkv)])
        V = torch.stack([torch.from_numpy(kvcache.gather(cache, segs[s], g, L)[1]) for g in range(cache.hkv)])
        mask = torch.zeros(1, L, dtype=torch.bool)
        mask[0, : p + 1] = True
        o = torch.nn.functional.scaled_dot_product_attention(
            q[r][:, None, :], K, V, attn_mask=mask, scale=scale, enable_gqa=True)
        out[r] = o[:, 0, :]
    return out.numpy()


def _small_mixed_workload(seed=11, kv="bf16"):
    lengths = [300, 513, 77, 256]
    paged = [True, False, True, False]
    tables = wl.permuted_tables(lengths, paged, 12, seed)
    streams = [wl.Stream(L, p, t, 0 if p else ((L + 255) // 256) * 256)
               for L, p, t in zip(lengths, paged, tables)]
    rs, rp = wl.decode_rows(lengths, [3, 1, 2, 4])
    # add a prompt-style row at position 0 and a mid-stream row
    rs = np.concatenate([rs, [0, 1]]).astype(np.int32)
    rp = np.concatenate([rp, [0, 200]]).astype(np.int32)
    w = wl.Workload("mixed", 8, 2, kv, 12, streams, rs, rp, seed, d=16)
    return w


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_matches_torch_sdpa(kv):
    w = _small_mixed_workload(kv=kv)
    cache, segs = build_oracle_cache(w)
    q = w.q_bits()
    out, _ = attention.attend(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale)
    ref = _sdpa_reference(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale)
    np.testing.assert_allclose(out, ref, rtol=0, atol=1e-12)


def test_closed_forms():
    rng = np.random.default_rng(3)
    n, d = 40, 8
    k = rng.standard_normal((n, d))
    # V constant c -> out = c exactly (weights sum to one within rounding)
    cache, segs = tiny_cache(k, np.full((n, d), 0.75))
    q = bits(rng.standard_normal((1, 1, d)))
    out, _ = attention.attend(cache, segs, q, [0], [n - 1], 0.3)
    np.testing.assert_allclose(out[0, 0], 0.75, rtol=0, atol=1e-15)
    # q = 0 -> uniform weights -> mean of the visible V; lse = ln(visible)
    v = np.round(rng.standard_normal((n, d)) * 8) / 8
    cache, segs = tiny_cache(k, v)
    out, lse = attention.attend(cache, segs, bits(np.zeros((1, 1, d))), [0], [24], 0.3)
    np.testing.assert_allclose(out[0, 0], v[:25].mean(axis=0), rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse[0, 0], math.log(25), rtol=0, atol=1e-14)
    # one visible key -> that V
    out, lse = attention.attend(cache, segs, q, [0], [0], 0.3)
    np.testing.assert_array_equal(out[0, 0], kvcache.bf16_to_f64(bits(v[0])))
    # duplicate keys -> their weights split evenly
    kd = np.vstack([k[:1], k[:1]])
    vd = np.array([[1.0] * d, [3.0] * d])
    cache, segs = tiny_cache(kd, vd)
    out, _ = attention.attend(cache, segs, q, [0], [1], 0.3)
    np.testing.assert_allclose(out[0, 0], 2.0, rtol=0, atol=1e-15)


def test_gqa_mapping_consecutive_heads_share_kv():
    """With V constant per kv head, query head h reads kv head h // G."""
    hq, hkv, d, L = 8, 2, 4, 10
    kp = np.zeros((1, hkv, 256, d), np.uint16)
    vp = np.zeros((1, hkv, 256, d), np.uint16)
    for g in range(hkv):
        vp[0, g, :L] = bits(np.full((L, d), float(g + 1)))
        kp[0, g, :L] = bits(np.random.default_rng(g).standard_normal((L, d)))
    cache = kvcache.Cache("bf16", hkv, d, kp, vp)
    segs = [kvcache.Segment(L, page_table=np.array([0], np.int32))]
    q = bits(np.random.default_rng(7).standard_normal((1, hq, d)))
    out, _ = attention.attend(cache, segs, q, [0], [L - 1], 0.5)
    want = np.array([1, 1, 1, 1, 2, 2, 2, 2], dtype=np.float64)
    np.testing.assert_allclose(out[0, :, 0], want, rtol=0, atol=1e-15)


def _permute_pool(cache, segs, seed):
    """Move every pool page to a new index and rewrite the tables to match."""
    n = cache.k_pool.shape[0]
    perm = np.random.default_rng(seed).permutation(n)   # new index of page i
    kp = np.empty_like(cache.k_pool)
    vp = np.empty_like(cache.v_pool)
    kp[perm] = cache.k_pool
    vp[perm] = cache.v_pool
    c2 = kvcache.Cache(cache.dtype, cache.hkv, cache.d, kp, vp, cache.k_scale, cache.v_scale)
    s2 = [kvcache.Segment(s.seq_len, page_table=perm[s.page_table].astype(np.int32))
          if s.page_table is not None else s for s in segs]
    return c2, s2


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_pool_permutation_leaves_output_unchanged(kv):
    w = _small_mixed_workload(kv=kv)
    cache, segs = build_oracle_cache(w)
    q = w.q_bits()
    a, la = attention.attend(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale)
    c2, s2 = _permute_pool(cache, segs, 99)
    b, lb = attention.attend(c2, s2, q, w.row_seg, w.row_pos, w.softmax_scale)
    assert np.array_equal(a, b) and np.array_equal(la, lb)


def test_paged_equals_slab():
    w = wl.batched_decode(seed=5, seq_len=700, n_streams=4, num_pages=12)
    wp = wl.batched_decode(seed=5, seq_len=700, n_streams=4, num_pages=12)
    for st in wp.streams:          # same values, every stream on pages now
        st.paged = True
    tables = wl.permuted_tables([700] * 4, [True] * 4, 12, 77)
    for st, t in zip(wp.streams, tables):
        st.page_table, st.slab_cap = t, 0
    c1, s1 = build_oracle_cache(w)
    c2, s2 = build_oracle_cache(wp)
    q = w.q_bits()
    a, _ = attention.attend(c1, s1, q, w.row_seg, w.row_pos, w.softmax_scale)
    b, _ = attention.attend(c2, s2, q, wp.row_seg, wp.row_pos, wp.softmax_scale)
    assert np.array_equal(a, b)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("pps", [1, 2, 3])
def test_split_merge_equals_one_pass(kv, pps):
    w = _small_mixed_workload(kv=kv)
    cache, segs = build_oracle_cache(w)
    q = w.q_bits()
    a, la = attention.attend(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale)
    m, l, o, nsplit = attention.attend_partials(cache, segs, q, w.row_seg, w.row_pos,
                                                w.softmax_scale, pps)
    b, lb = attention.merge(m, l, o)
    np.testing.assert_allclose(b, a, rtol=0, atol=1e-12)
    np.testing.assert_allclose(lb, la, rtol=0, atol=1e-12)
    for r in range(w.rows):
        L = w.streams[int(w.row_seg[r])].seq_len
        assert nsplit[r] == -(-((L + 255) // 256) // pps)


def test_stream_output_independent_of_batch():
    w = _small_mixed_workload()
    cache, segs = build_oracle_cache(w)
    q = w.q_bits()
    full, _ = attention.attend(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale)
    for s in range(len(segs)):
        sel = np.flatnonzero(w.row_seg == s)
        alone, _ = attention.attend(cache, [segs[s]], q[sel], np.zeros(len(sel), np.int32),
                                    w.row_pos[sel], w.softmax_scale)
        assert np.array_equal(alone, full[sel])


def test_causal_rows_of_a_prompt_chunk():
    w = wl.small("prompt_chunk")
    cache, segs = build_oracle_cache(w)
    q = w.q_bits()
    # the chunk's first and last rows, plus a row at position 0
    rs = np.array([0, 0, 0], np.int32)
    rp = np.array([0, int(w.row_pos[0]), int(w.row_pos[-1])], np.int32)
    out, _ = attention.attend(cache, segs, q[[0, 0, -1]], rs, rp, w.softmax_scale)
    V0 = kvcache.gather(cache, segs[0], 0, 1)[1][0]
    np.testing.assert_array_equal(out[0, 0], V0)             # sees only key 0
    L = segs[0].seq_len
    assert rp[2] == L - 1                                    # last row sees every key
    qf = torch.from_numpy(kvcache.bf16_to_f64(q[-1]))[:, None, :]
    K = torch.stack([torch.from_numpy(kvcache.gather(cache, segs[0], g, L)[0]) for g in range(8)])
    V = torch.stack([torch.from_numpy(kvcache.gather(cache, segs[0], g, L)[1]) for g in range(8)])
    full = torch.nn.functional.scaled_dot_product_attention(qf, K, V, scale=w.softmax_scale,
                                                            enable_gqa=True)[:, 0].numpy()
    np.testing.assert_allclose(out[2], full, rtol=0, atol=1e-12)


def test_swapped_table_control():
    """Swapping the partial last page with a full page changes the output
    (the control is red); swapping two full pages of a row that sees every
    key keeps the same key set, so that control would stay green."""
    w = wl.tiny_paged_decode(seed=236)
    cache, segs = build_oracle_cache(w)
    q = w.q_bits()
    a, _ = attention.attend(cache, segs, q, w.row_seg, w.row_pos, w.softmax_scale)
    t = segs[0].page_table.copy()
    t_bad = t.copy()
    t_bad[[0, 3]] = t_bad[[3, 0]]                    # partial last page <-> full page
    b, _ = attention.attend(cache, [kvcache.Segment(1000, page_table=t_bad)], q,
                            w.row_seg, w.row_pos, w.softmax_scale)
    assert np.abs(a - b).max() > 1e-3
    t_same = t.copy()
    t_same[[0, 1]] = t_same[[1, 0]]                  # two full pages
    c, _ = attention.attend(cache, [kvcache.Segment(1000, page_table=t_same)], q,
                            w.row_seg, w.row_pos, w.softmax_scale)
    np.testing.assert_allclose(c, a, rtol=0, atol=1e-12)


def test_kv_write_addresses_and_codes():
    """write_rows puts row (seg, pos, g) at pool[PT[pos//256]][g][pos%256] or
    slab[g][pos]; bf16 bits unchanged, fp8 = encode(float32(x)/scale)."""
    hkv, d = 2, 8
    rng = np.random.default_rng(4)
    for dtype in ("bf16", "fp8"):
        store = np.uint16 if dtype == "bf16" else np.uint8
        kp = np.zeros((6, hkv, 256, d), store)
        vp = np.zeros((6, hkv, 256, d), store)
        ks = np.array([0.5, 0.01], np.float32)
        vs = np.array([0.25, 0.02], np.float32)
        cache = kvcache.Cache(dtype, hkv, d, kp, vp, ks, vs)
        slab_k = np.zeros((hkv, 512, d), store)
        slab_v = np.zeros((hkv, 512, d), store)
        segs = [kvcache.Segment(600, page_table=np.array([4, 1, 5], np.int32)),
                kvcache.Segment(300, k_slab=slab_k, v_slab=slab_v)]
        kr = bits(rng.standard_normal((3, hkv, d)))
        vr = bits(rng.standard_normal((3, hkv, d)))
        kvcache.write_rows(cache, segs, kr, vr, [0, 0, 1], [3, 513, 299])
        for g in range(hkv):
            for (arr, idx, r) in ((kp, (4, g, 3), 0), (kp, (5, g, 1), 1), (slab_k, (g, 299), 2)):
                if dtype == "bf16":
                    assert np.array_equal(arr[idx], kr[r, g])
                else:
                    x = (kr[r, g].astype(np.uint32) << 16).view(np.float32)
                    want = torch.from_numpy((x / ks[g]).astype(np.float32)).to(
                        torch.float8_e4m3fn).view(torch.uint8).numpy()
                    assert np.array_equal(arr[idx], want)
        assert np.count_nonzero(kp) == np.count_nonzero(kp[[4, 5]])   # nothing else written


def test_kv_write_vector_form():
    """The vectorised stream writer used by the tests equals write_rows."""
    from tests.oracle_cases import write_stream
    w = wl.small("fp8_verify")
    c1, s1 = build_oracle_cache(w)
    c2 = kvcache.Cache("fp8", w.hkv, w.d, np.zeros_like(c1.k_pool), np.zeros_like(c1.v_pool),
                       c1.k_scale, c1.v_scale)
    c3 = kvcache.Cache("fp8", w.hkv, w.d, np.zeros_like(c1.k_pool), np.zeros_like(c1.v_pool),
                       c1.k_scale, c1.v_scale)
    k, v = w.stream_kv_bits(1)
    L = w.streams[1].seq_len
    rk, rv = np.ascontiguousarray(k.transpose(1, 0, 2)), np.ascontiguousarray(v.transpose(1, 0, 2))
    write_stream(c2, s1, 1, rk, rv, L)
    kvcache.write_rows(c3, s1, rk, rv, np.ones(L, np.int32), np.arange(L, dtype=np.int32))
    assert np.array_equal(c2.k_pool, c3.k_pool) and np.array_equal(c2.v_pool, c3.v_pool)


# ---------------------------------------------------------------------------
# Planted mistakes: each is a plausible bug put into the oracle on the CPU;
# at least one pin above must go red for it.
# ---------------------------------------------------------------------------

def test_planted_dropped_causal_mask(monkeypatch):
    orig = attention.attend

    def no_mask(cache, segs, q, row_seg, row_pos, scale):
        return orig(cache, segs, q, row_seg, [segs[int(s)].seq_len - 1 for s in row_seg], scale)

    monkeypatch.setattr(attention, "attend", no_mask)
    with pytest.raises(AssertionError):
        test_matches_torch_sdpa("bf16")


def test_planted_wrong_kv_head(monkeypatch):
    orig = kvcache.gather

    def wrong_head(cache, seg, g, n):
        return orig(cache, seg, (g + 1) % cache.hkv, n)

    monkeypatch.setattr(kvcache, "gather", wrong_head)
    monkeypatch.setattr(attention, "gather", wrong_head)
    with pytest.raises(AssertionError):
        test_gqa_mapping_consecutive_heads_share_kv()


def test_planted_page_table_ignored(monkeypatch):
    orig = kvcache.gather

    def identity_table(cache, seg, g, n):
        if seg.page_table is not None:
            seg = kvcache.Segment(seg.seq_len, page_table=np.arange(len(seg.page_table), dtype=np.int32))
        return orig(cache, seg, g, n)

    monkeypatch.setattr(attention, "gather", identity_table)
    with pytest.raises(AssertionError):
        test_pool_permutation_leaves_output_unchanged("bf16")


def test_planted_merge_without_rescale(monkeypatch):
    def bad_merge(m, l, o):
        M = m.max(axis=-1, keepdims=True)
        w = np.where(np.isfinite(m), np.exp(m - M), 0.0)
        L = l.sum(axis=-1)                       # l not rescaled
        O = (w[..., None] * o).sum(axis=-2) / L[..., None]
        return O, M[..., 0] + np.log(L)

    monkeypatch.setattr(attention, "merge", bad_merge)
    with pytest.raises(AssertionError):
        test_split_merge_equals_one_pass("bf16", 1)


def test_planted_slot_in_page(monkeypatch):
    orig = kvcache._store

    def wrong_slot(cache, seg, which, g, pos):
        arr, idx = orig(cache, seg, which, g, pos)
        if seg.page_table is not None:
            idx = (idx[0], g, (pos + 1) % 256)
        return arr, idx

    monkeypatch.setattr(kvcache, "_store", wrong_slot)
    with pytest.raises(AssertionError):
        test_kv_write_addresses_and_codes()
