"""Plans on the GPU: launches planned ahead and enqueued later give exactly
the bytes of the direct calls, for a decode loop whose lengths advance
(each step planned while the previous one runs)."""

import numpy as np
import pytest
import torch

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, bits

pytestmark = pytest.mark.gpu


def test_planned_decode_loop_equals_direct_calls():
    w = wl.small("batched_decode")
    L = [st.seq_len for st in w.streams]
    nst = len(w.streams)
    ga, gb = GpuCase(w), GpuCase(w)            # two identical caches: direct and planned
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    steps = 4
    ks = [torch.randn(nst, w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(steps)]
    vs = [torch.randn_like(k) for k in ks]
    q = ga.q()[:nst].contiguous()
    sidx = np.arange(nst, dtype=np.int32)
    tab_a, tab_b = B.SegTable(ga.segs), B.SegTable(gb.segs)
    sc_a, sc_b = B.make_scratch(16, w.hq), B.make_scratch(16, w.hq)
    out_a = torch.empty(nst, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty_like(out_a)
    plan = B.Plan()
    # lengths go back three positions and then forward one a step (the
    # positions written hold the workload's data already, so both caches
    # stay equal to each other)
    for i in range(steps):
        n = [x - 3 + i for x in L]
        for j in range(nst):
            tab_a.set_seq_len(j, n[j])
            tab_b.set_seq_len(j, n[j])
        rp = np.array([x - 1 for x in n], np.int32)
        B.tfpa_write_kv(ga.cache, tab_a, ks[i], vs[i], sidx, rp)
        B.tfpa_decode(ga.cache, tab_a, q, sidx, rp, w.softmax_scale, sc_a, out_a)
        plan.clear()
        plan.write_kv(gb.cache, tab_b, ks[i], vs[i], sidx, rp)
        plan.decode(gb.cache, tab_b, q, sidx, rp, w.softmax_scale, sc_b, out_b)
        plan.launch()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out_a), bits(out_b)), f"step {i}"
    plan.launch()                                 # a plan may be launched again
    torch.cuda.synchronize()
    assert np.array_equal(bits(out_a), bits(out_b))
    assert int(ga.err.item()) == 0 and int(gb.err.item()) == 0


@pytest.mark.parametrize("via", ["torch_graph", "plan_capture"])
@pytest.mark.parametrize("name", ["batched_decode", "fp8_verify"])
def test_device_mode_graph_replays_a_growing_decode_loop(name, via):
    """A plan in device mode captured once as a CUDA graph (the copy of its
    packed data, then its launches; by torch's graph capture, or by
    tfpa_plan_capture) and replayed step after step with the lengths growing
    by one, across a split boundary, gives the bytes of the direct calls at
    every step."""
    w = wl.small(name)
    nst = len(w.streams)
    L = min(st.seq_len for st in w.streams)
    b = (L - 8) // 512 * 512                      # n = b - 3 .. b + 4 crosses b
    assert b >= 512
    ga, gb = GpuCase(w), GpuCase(w)
    g = torch.Generator(device="cuda")
    g.manual_seed(11)
    steps = 8
    ks = [torch.randn(nst, w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(steps)]
    vs = [torch.randn_like(k) for k in ks]
    qs = [torch.randn(nst, w.hq, 128, generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(steps)]
    kbuf, vbuf, qbuf = torch.empty_like(ks[0]), torch.empty_like(vs[0]), torch.empty_like(qs[0])
    sidx = np.arange(nst, dtype=np.int32)
    tab_a, tab_b = B.SegTable(ga.segs), B.SegTable(gb.segs)
    sc_a, sc_b = B.make_scratch(16, w.hq), B.make_scratch(16, w.hq)
    out_a = torch.empty(nst, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    out_b = torch.empty_like(out_a)
    dyn = torch.zeros(1 << 16, dtype=torch.uint8, device="cuda")
    hdyn = torch.zeros(1 << 16, dtype=torch.uint8).pin_memory()
    plan = B.Plan()
    plan.set_device(dyn)

    def lengths(i):
        n = b - 3 + i
        for j in range(nst):
            tab_a.set_seq_len(j, n)
            tab_b.set_seq_len(j, n)
        return np.full(nst, n - 1, np.int32)

    graph, shape, nb = None, None, 0
    s = torch.cuda.current_stream()
    for i in range(steps):
        rp = lengths(i)
        B.tfpa_write_kv(ga.cache, tab_a, ks[i], vs[i], sidx, rp)
        B.tfpa_decode(ga.cache, tab_a, qs[i], sidx, rp, w.softmax_scale, sc_a, out_a)
        plan.clear()
        plan.write_kv(gb.cache, tab_b, kbuf, vbuf, sidx, rp)
        plan.decode(gb.cache, tab_b, qbuf, sidx, rp, w.softmax_scale, sc_b, out_b)
        plan.pack(hdyn)
        kbuf.copy_(ks[i])
        vbuf.copy_(vs[i])
        qbuf.copy_(qs[i])
        if graph is None:
            # step 0 runs the plan directly (and sets the kernels up), then
            # the graph is captured for the later steps
            nb = plan.dyn_bytes()
            shape = plan.shape()
            dyn[:nb].copy_(hdyn[:nb], non_blocking=True)
            plan.launch()
            torch.cuda.synchronize()
            cap = torch.cuda.Stream()
            if via == "plan_capture":
                plan.capture(before=[(dyn, hdyn, nb)], stream=cap)
                graph = plan
            else:
                graph = torch.cuda.CUDAGraph()
                cap.wait_stream(s)
                with torch.cuda.stream(cap):
                    with torch.cuda.graph(graph, stream=cap):
                        dyn[:nb].copy_(hdyn[:nb], non_blocking=True)
                        plan.launch(cap)
                s.wait_stream(cap)
        else:
            assert plan.shape() == shape and plan.dyn_bytes() == nb, f"step {i}"
            graph.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out_a), bits(out_b)), f"step {i}"
    assert int(ga.err.item()) == 0 and int(gb.err.item()) == 0
    # the caches took the same rows
    for sa, sb in zip(ga.segs, gb.segs):
        if sa.page_table is None:
            assert torch.equal(sa.k_slab, sb.k_slab) and torch.equal(sa.v_slab, sb.v_slab)
    assert torch.equal(ga.k_pool, gb.k_pool)
    assert torch.equal(ga.v_pool, gb.v_pool)


def test_plan_capture_refuses_the_legacy_stream_and_a_changed_shape():
    """tfpa_plan_capture needs a created stream; a replay after the plan was
    re-planned with another row count is refused (the captured launches no
    longer fit), and the plan still launches directly."""
    w = wl.small("batched_decode")
    g = GpuCase(w)
    nst = len(w.streams)
    q = g.q()[:nst].contiguous()
    sidx = np.arange(nst, dtype=np.int32)
    rp = np.array([st.seq_len - 1 for st in w.streams], np.int32)
    sc = B.make_scratch(16, w.hq)
    out = torch.empty(nst, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    plan = B.Plan()
    plan.decode(g.cache, g.segs, q, sidx, rp, w.softmax_scale, sc, out)
    plan.launch()
    torch.cuda.synchronize()
    for bad in (0, 1):                               # NULL and cudaStreamLegacy
        with pytest.raises(B.TfpaError) as e:
            plan.capture(stream=bad)
        assert e.value.code == B.TFPA_EINVAL
    plan.capture(stream=torch.cuda.Stream())
    plan.replay()
    torch.cuda.synchronize()
    ref = bits(out)
    plan.clear()
    plan.decode(g.cache, g.segs, q[:2], sidx[:2], rp[:2], w.softmax_scale, sc, out[:2])
    with pytest.raises(B.TfpaError) as e:
        plan.replay()
    assert e.value.code == B.TFPA_EINVAL
    plan.clear()
    plan.decode(g.cache, g.segs, q, sidx, rp, w.softmax_scale, sc, out)
    plan.replay()                                    # the captured shape again
    torch.cuda.synchronize()
    assert np.array_equal(bits(out), ref)
    assert int(g.err.item()) == 0
