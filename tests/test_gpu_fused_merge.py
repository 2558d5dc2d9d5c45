"""The merge inside the partial kernel (a scratch with arrival counters)
against the separate merge launch: the same bytes of out and lse for plain
decode rows, draft-tree rows, sliced calls and calls that mix decode-path
and tensor-core verify rows, and the counters back at zero after each call."""

import numpy as np
import pytest
import torch

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, bits, fp8_scales

pytestmark = pytest.mark.gpu


def _lse_bits(t):
    return t.cpu().numpy().view(np.uint32)


def _pair(g, fn, *args, **kw):
    fused = fn(*args, fused=True, **kw)
    plain = fn(*args, fused=False, **kw)
    assert np.array_equal(bits(fused[0]), bits(plain[0]))
    assert np.array_equal(_lse_bits(fused[1]), _lse_bits(plain[1]))
    assert int(g.err.item()) == 0


@pytest.mark.parametrize("name", ["tiny_paged_decode", "batched_decode", "fp8_verify",
                                  "overcommitted_pool"])
@pytest.mark.parametrize("cap_rows", [128, 3])
def test_fused_merge_equals_separate_merge(name, cap_rows):
    w = wl.small(name)
    g = GpuCase(w, fp8_scales(w) if w.kv_dtype == "fp8" else None)
    _pair(g, g.decode, g.q(), w.row_seg, w.row_pos, cap_rows=cap_rows)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_tree_rows_with_counters_equal_the_separate_merge(kv):
    # 12 nodes x 4 heads per kv head = 3 m-tiles: the decode partial kernel;
    # tree rows keep the separate merge whatever the scratch
    w = wl.tree_verify(1235, seq_len=1300, n_streams=3, nodes=12, kv_dtype=kv, slack_pages=5)
    g = GpuCase(w, fp8_scales(w) if kv == "fp8" else None)
    _pair(g, g.decode_tree, g.q(), w.row_seg, w.row_pos, w.row_anc)


def test_mixed_slices_keep_the_separate_merge_where_verify_rows_run():
    # stream 0: 20 rows (tensor-core verify path), streams 1, 2: one row each
    # (decode path); 16-row slices put the verify rows in the first two slices
    w = wl.small("fp8_verify")
    g = GpuCase(w, fp8_scales(w))
    L = [st.seq_len for st in w.streams]
    rs = np.array([0] * 20 + [1, 2], np.int32)
    rp = np.array(list(range(L[0] - 20, L[0])) + [L[1] - 1, L[2] - 1], np.int32)
    q = torch.randn(len(rs), w.hq, 128, device="cuda").to(torch.bfloat16)
    _pair(g, g.decode, q, rs, rp)
    _pair(g, g.decode, q, rs, rp, cap_rows=16)


def test_counters_return_to_zero_and_repeat_calls_agree():
    w = wl.small("batched_decode")
    g = GpuCase(w)
    sc = B.make_scratch(8, w.hq, fused_merge=True)
    out = torch.empty(w.rows, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    first = None
    for _ in range(5):
        B.tfpa_decode(g.cache, g.segs, g.q(), w.row_seg, w.row_pos, w.softmax_scale, sc, out)
        torch.cuda.synchronize()
        assert int(sc.arrive.abs().sum().item()) == 0
        if first is None:
            first = bits(out)
        assert np.array_equal(bits(out), first)


def test_graph_of_layer_calls_replays_the_direct_bytes():
    """Tiny calls on caches of their own (one per layer of a decode step, as
    the bench's layer-call line runs them) captured as one CUDA graph: every
    replay gives the direct calls' bytes, and each call leaves its arrival
    counters at zero, so the next replay merges again."""
    layers = []
    for i in range(4):
        w = wl.tiny_paged_decode(seed=500 + i)
        g = GpuCase(w)
        sc = B.make_scratch(1, w.hq)
        out = torch.empty(w.rows, w.hq, 128, dtype=torch.bfloat16, device="cuda")
        layers.append((w, g, sc, out, g.q()))

    def calls():
        for w, g, sc, out, q in layers:
            B.tfpa_decode(g.cache, g.segs, q, w.row_seg, w.row_pos, w.softmax_scale, sc, out)

    calls()
    torch.cuda.synchronize()
    ref = [bits(out).copy() for _, _, _, out, _ in layers]
    graph = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        with torch.cuda.graph(graph, stream=s):
            calls()
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(3):
        for _, _, _, out, _ in layers:
            out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for (w, g, sc, out, q), r in zip(layers, ref):
            assert np.array_equal(bits(out), r)
            assert int(sc.arrive.abs().sum().item()) == 0
            assert int(g.err.item()) == 0
