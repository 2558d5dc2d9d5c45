"""RoPE KV store and keep on the GPU against the oracle, byte for byte, and
the drafted == plain gate (a draft tree stored, verified and its accepted
path kept gives the bytes and the next decode row of a plain decode), with a
planted wrong keep as the red control."""

import numpy as np
import pytest
import torch

from oracle import kvstore
from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, bits, fp8_scales
from tests.oracle_cases import build_oracle_cache

pytestmark = pytest.mark.gpu


def _mixed(kv, lengths=(700, 300, 520), paged=(True, False, True), seed=71):
    npages = sum((L + 255) // 256 for L, p in zip(lengths, paged) if p) + 3
    tables = wl.permuted_tables(list(lengths), list(paged), npages, seed)
    streams = [wl.Stream(L, p, t, 0 if p else ((L + 255) // 256) * 256)
               for L, p, t in zip(lengths, paged, tables)]
    return wl.Workload("store", 8, 2, kv, npages, streams, np.zeros(1, np.int32),
                       np.zeros(1, np.int32), seed)


def _host(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy().view(np.uint8)


def _assert_same_bytes(g, cache_o, segs_o):
    assert np.array_equal(_host(g.k_pool), cache_o.k_pool)
    assert np.array_equal(_host(g.v_pool), cache_o.v_pool)
    for sg, so in zip(g.segs, segs_o):
        if so.k_slab is not None:
            assert np.array_equal(_host(sg.k_slab), so.k_slab)
            assert np.array_equal(_host(sg.v_slab), so.v_slab)


def _dev_rows(bits16):
    t = torch.from_numpy(np.ascontiguousarray(bits16).view(np.int16))
    return t.cuda().view(torch.bfloat16)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("device_pos", [True, False])
def test_rope_store_bytes_match_oracle(kv, device_pos):
    w = _mixed(kv)
    scales = fp8_scales(w) if kv == "fp8" else None
    g = GpuCase(w, scales)
    cache_o, segs_o = build_oracle_cache(w, *(scales or (None, None)))
    cos, sin = wl.rope_table(1e6, 2048)
    rs = np.array([0, 0, 1, 2, 2], np.int32)
    rp = np.array([5, 699, 12, 300, 301], np.int32)
    rpos = np.array([5, 3, 1000, 0, 2047], np.int32) if device_pos else rp
    k = wl.randn_bf16_bits((5, 2, 128), 81)
    v = wl.randn_bf16_bits((5, 2, 128), 82)
    B.tfpa_write_kv_rope(g.cache, g.segs, _dev_rows(k), _dev_rows(v), rs, rp,
                         torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda(),
                         torch.from_numpy(rpos).cuda() if device_pos else None)
    torch.cuda.synchronize()
    kvstore.write_rows_rope(cache_o, segs_o, k, v, rs, rp, rpos, cos, sin)
    _assert_same_bytes(g, cache_o, segs_o)
    assert int(g.err.item()) == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_keep_bytes_match_oracle(kv):
    w = _mixed(kv)
    scales = fp8_scales(w) if kv == "fp8" else None
    g = GpuCase(w, scales)
    cache_o, segs_o = build_oracle_cache(w, *(scales or (None, None)))
    # a chain (10 -> 3, 3 -> 11), a swap (7 <-> 8) on the slab stream, one across pages
    ks, src, dst = [0, 0, 1, 1, 2], [10, 3, 7, 8, 100], [3, 11, 8, 7, 400]
    B.tfpa_keep_kv(g.cache, g.segs, ks, src, dst)
    torch.cuda.synchronize()
    kvstore.keep_rows(cache_o, segs_o, ks, src, dst)
    _assert_same_bytes(g, cache_o, segs_o)
    assert int(g.err.item()) == 0


def _round(kv, path_override=None, seed=90):
    """Plain and drafted rounds on one stream; returns both next-row outputs
    and the bytes of the committed positions."""
    L0, n = 600, 12
    parents = wl.random_tree(n, seed)
    depth = wl.tree_depths(parents)
    leaf = max(range(n), key=lambda i: (depth[i], i))
    accepted = path_to(parents, leaf)        # root .. leaf, in depth order
    path = accepted if path_override is None else path_override(accepted, parents)
    acc = len(accepted)
    cap = L0 + n + 1
    w = _mixed(kv, lengths=(cap,), paged=(True,), seed=seed)
    scales = fp8_scales(w) if kv == "fp8" else None
    cos, sin = wl.rope_table(1e6, 4096)
    cos_d, sin_d = torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda()
    node_k = wl.randn_bf16_bits((n, 2, 128), seed + 1)
    node_v = wl.randn_bf16_bits((n, 2, 128), seed + 2)
    nxt_k = wl.randn_bf16_bits((1, 2, 128), seed + 3)
    nxt_v = wl.randn_bf16_bits((1, 2, 128), seed + 4)
    q = wl.randn_bf16_bits((1, 8, 128), seed + 5)
    outs, stored = [], []
    for drafted in (False, True):
        g = GpuCase(w, scales)
        if not drafted:                      # the accepted tokens, stored in place
            pk, pv = node_k[accepted], node_v[accepted]
            pos = np.arange(L0, L0 + acc, dtype=np.int32)
            B.tfpa_write_kv_rope(g.cache, g.segs, _dev_rows(pk), _dev_rows(pv),
                                 np.zeros(acc, np.int32), pos, cos_d, sin_d)
        else:                                # the tree, the verify pass, then keep
            pos = np.arange(L0, L0 + n, dtype=np.int32)
            rope = torch.from_numpy(np.asarray([L0 + d for d in depth], np.int32)).cuda()
            B.tfpa_write_kv_rope(g.cache, g.segs, _dev_rows(node_k), _dev_rows(node_v),
                                 np.zeros(n, np.int32), pos, cos_d, sin_d, rope)
            anc = np.array(wl.tree_masks(parents), np.uint64)
            qt = torch.randn(n, 8, 128, device="cuda").to(torch.bfloat16)
            g.decode_tree(qt, np.zeros(n, np.int32), pos, anc)           # the verify pass
            B.tfpa_keep_kv(g.cache, g.segs, [0] * acc, [L0 + i for i in path],
                           [L0 + d for d in range(acc)])
        ln = L0 + acc
        B.tfpa_write_kv_rope(g.cache, g.segs, _dev_rows(nxt_k), _dev_rows(nxt_v), [0], [ln],
                             cos_d, sin_d)
        segs = [B.Seg(ln + 1, page_table=g.segs[0].page_table,
                      page_table_host=g.segs[0].page_table_host)]
        out, _ = g.decode(_dev_rows(q), [0], [ln], segs=segs)
        outs.append(bits(out))
        k_rows = [_host(g.k_pool)[int(w.streams[0].page_table[p // 256]), :, p % 256]
                  for p in range(L0 - 2, ln + 1)]
        stored.append(np.stack(k_rows))
        assert int(g.err.item()) == 0
    return outs, stored


def path_to(parents, node):
    path = []
    while node >= 0:
        path.append(node)
        node = parents[node]
    return path[::-1]


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_drafted_equals_plain(kv):
    (plain, drafted), (sp, sd) = _round(kv)
    assert np.array_equal(sp, sd)
    assert np.array_equal(plain, drafted)


def test_planted_wrong_keep_is_red():
    def swap_in_sibling(path, parents):
        # keep a node off the accepted path in place of the path's second node
        others = [i for i in range(len(parents)) if i not in path and parents[i] == path[0]]
        alt = others[0] if others else next(i for i in range(len(parents)) if i not in path)
        return [path[0], alt] + path[2:]
    (plain, drafted), (sp, sd) = _round("bf16", path_override=swap_in_sibling)
    assert not np.array_equal(sp, sd)
    assert not np.array_equal(plain, drafted)
