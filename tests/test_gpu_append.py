"""tfpa_decode_append against tfpa_write_kv followed by tfpa_decode: the same
bytes in the cache (pool pages and slabs) and in the output and lse, when
the partial kernel stores the new rows itself (narrow runs, bf16 and e4m3,
sliced calls, the merge inside the partial kernel) and when a KV write
launch goes first (a wide run); also a device-mode plan replayed as a graph
over a growing decode loop."""

import numpy as np
import pytest
import torch

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, bits, fp8_scales
from tests.gpu_cases import append_rows as _rows
from tests.gpu_cases import same_cache as _same_cache

pytestmark = pytest.mark.gpu


def _pair(w, rows_per_stream, cap_rows=128, seed=21):
    scales = fp8_scales(w) if w.kv_dtype == "fp8" else None
    ga, gb = GpuCase(w, scales), GpuCase(w, scales)
    rs, rp, k, v, q = _rows(w, rows_per_stream, seed)
    n = len(rs)
    outs = []
    for g, fused in ((ga, False), (gb, True)):
        out = torch.empty(n, w.hq, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(n, w.hq, dtype=torch.float32, device="cuda")
        sc = B.make_scratch(cap_rows, w.hq)
        if fused:
            B.tfpa_decode_append(g.cache, g.segs, k, v, q, rs, rp, w.softmax_scale, sc, out, lse)
        else:
            B.tfpa_write_kv(g.cache, g.segs, k, v, rs, rp)
            B.tfpa_decode(g.cache, g.segs, q, rs, rp, w.softmax_scale, sc, out, lse)
        torch.cuda.synchronize()
        outs.append((out, lse))
    assert np.array_equal(bits(outs[0][0]), bits(outs[1][0]))
    assert np.array_equal(outs[0][1].cpu().numpy().view(np.uint32),
                          outs[1][1].cpu().numpy().view(np.uint32))
    _same_cache(ga, gb)
    assert int(ga.err.item()) == 0 and int(gb.err.item()) == 0


@pytest.mark.parametrize("name,rows", [("batched_decode", 1), ("batched_decode", 3),
                                       ("fp8_verify", 1), ("fp8_verify", 4),
                                       ("tiny_paged_decode", 1), ("overcommitted_pool", 1)])
def test_append_equals_write_then_decode(name, rows):
    _pair(wl.small(name), rows)


def test_append_in_slices_and_with_a_wide_run():
    w = wl.small("fp8_verify")
    _pair(w, 4, cap_rows=3)          # slices of three rows: a run's rows over two launches
    _pair(w, 20)                     # 20 rows a stream: the verify path, a write launch first


def test_device_mode_plan_appends_over_a_growing_loop():
    """One captured graph of a device-mode append plan, replayed as the
    lengths grow across a split boundary, against write + decode calls."""
    w = wl.small("batched_decode")
    nst = len(w.streams)
    L = min(st.seq_len for st in w.streams)
    b = (L - 8) // 512 * 512
    ga, gb = GpuCase(w), GpuCase(w)
    g = torch.Generator(device="cuda")
    g.manual_seed(31)
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
    for i in range(steps):
        n = b - 3 + i
        for j in range(nst):
            tab_a.set_seq_len(j, n)
            tab_b.set_seq_len(j, n)
        rp = np.full(nst, n - 1, np.int32)
        B.tfpa_write_kv(ga.cache, tab_a, ks[i], vs[i], sidx, rp)
        B.tfpa_decode(ga.cache, tab_a, qs[i], sidx, rp, w.softmax_scale, sc_a, out_a)
        plan.clear()
        plan.decode_append(gb.cache, tab_b, kbuf, vbuf, qbuf, sidx, rp, w.softmax_scale, sc_b,
                           out_b)
        assert len(plan) == 2                       # partial + merge: no write launch
        plan.pack(hdyn)
        kbuf.copy_(ks[i])
        vbuf.copy_(vs[i])
        qbuf.copy_(qs[i])
        if i == 0:
            nb = plan.dyn_bytes()
            dyn[:nb].copy_(hdyn[:nb], non_blocking=True)
            plan.launch()
            torch.cuda.synchronize()
            plan.capture(before=[(dyn, hdyn, nb)], stream=torch.cuda.Stream())
        else:
            plan.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out_a), bits(out_b)), f"step {i}"
    _same_cache(ga, gb)
    assert int(ga.err.item()) == 0 and int(gb.err.item()) == 0
