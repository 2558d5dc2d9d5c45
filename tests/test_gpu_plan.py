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
