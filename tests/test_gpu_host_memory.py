"""Pinned host memory on the decode path: q, the new K/V rows, out and lse
(and a device-mode plan's packed data) in page-locked host memory, which the
kernels read and write over the host link, give the bytes that device
buffers give; q in host memory is refused where TMA would load it (the
tensor-core verify path, the prompt path), with nothing enqueued."""

import numpy as np
import pytest
import torch

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, append_rows, bits, fp8_scales, same_cache

pytestmark = pytest.mark.gpu


def _pinned(t):
    return t.cpu().pin_memory()


@pytest.mark.parametrize("name,rows", [("batched_decode", 1), ("fp8_verify", 2),
                                       ("tiny_paged_decode", 1), ("overcommitted_pool", 1)])
def test_host_rows_and_output_equal_device_buffers(name, rows):
    w = wl.small(name)
    scales = fp8_scales(w) if w.kv_dtype == "fp8" else None
    ga, gb = GpuCase(w, scales), GpuCase(w, scales)
    rs, rp, k, v, q = append_rows(w, rows, 41)
    n = len(rs)
    out = torch.empty(n, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(n, w.hq, dtype=torch.float32, device="cuda")
    hk, hv, hq = _pinned(k), _pinned(v), _pinned(q)
    hout = torch.zeros(n, w.hq, 128, dtype=torch.bfloat16).pin_memory()
    hlse = torch.zeros(n, w.hq, dtype=torch.float32).pin_memory()
    for fused_merge in (True, False):
        sa = B.make_scratch(128, w.hq, fused_merge=fused_merge)
        sb = B.make_scratch(128, w.hq, fused_merge=fused_merge)
        B.tfpa_decode_append(ga.cache, ga.segs, k, v, q, rs, rp, w.softmax_scale, sa, out, lse)
        B.tfpa_decode_append(gb.cache, gb.segs, hk, hv, hq, rs, rp, w.softmax_scale, sb, hout,
                             hlse)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), bits(hout))
        assert np.array_equal(lse.cpu().numpy().view(np.uint32), hlse.numpy().view(np.uint32))
        # tfpa_decode alone, q and out in host memory
        B.tfpa_decode(ga.cache, ga.segs, q, rs, rp, w.softmax_scale, sa, out, lse)
        B.tfpa_decode(gb.cache, gb.segs, hq, rs, rp, w.softmax_scale, sb, hout, hlse)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), bits(hout))
    same_cache(ga, gb)
    assert int(ga.err.item()) == 0 and int(gb.err.item()) == 0


def test_plan_with_host_buffers_replays_a_growing_loop():
    """A device-mode append plan whose packed data, q, K/V rows and output
    all sit in pinned host memory, captured once (no copies) and replayed as
    the lengths grow across a split boundary, against direct calls on
    device buffers; the host writes each step's inputs before the replay."""
    w = wl.small("batched_decode")
    nst = len(w.streams)
    L = min(st.seq_len for st in w.streams)
    b = (L - 8) // 512 * 512
    ga, gb = GpuCase(w), GpuCase(w)
    g = torch.Generator(device="cuda")
    g.manual_seed(37)
    steps = 8
    ks = [torch.randn(nst, w.hkv, 128, generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(steps)]
    vs = [torch.randn_like(x) for x in ks]
    qs = [torch.randn(nst, w.hq, 128, generator=g, device="cuda").to(torch.bfloat16)
          for _ in range(steps)]
    hk, hv, hq = (torch.empty(x.shape, dtype=x.dtype).pin_memory() for x in (ks[0], vs[0], qs[0]))
    hout = torch.zeros(nst, w.hq, 128, dtype=torch.bfloat16).pin_memory()
    hdyn = torch.zeros(1 << 16, dtype=torch.uint8).pin_memory()
    sidx = np.arange(nst, dtype=np.int32)
    tab_a, tab_b = B.SegTable(ga.segs), B.SegTable(gb.segs)
    sc_a, sc_b = B.make_scratch(16, w.hq), B.make_scratch(16, w.hq)
    out_a = torch.empty(nst, w.hq, 128, dtype=torch.bfloat16, device="cuda")
    plan = B.Plan()
    plan.set_device(hdyn)
    for i in range(steps):
        n = b - 3 + i
        for j in range(nst):
            tab_a.set_seq_len(j, n)
            tab_b.set_seq_len(j, n)
        rp = np.full(nst, n - 1, np.int32)
        B.tfpa_decode_append(ga.cache, tab_a, ks[i], vs[i], qs[i], sidx, rp, w.softmax_scale,
                             sc_a, out_a)
        torch.cuda.synchronize()            # the previous replay is done with host memory
        plan.clear()
        plan.decode_append(gb.cache, tab_b, hk, hv, hq, sidx, rp, w.softmax_scale, sc_b, hout)
        assert len(plan) == 2
        plan.pack(hdyn)                     # straight into the buffer the kernels read
        hk.copy_(ks[i])
        hv.copy_(vs[i])
        hq.copy_(qs[i])
        if i == 0:
            plan.launch()
            torch.cuda.synchronize()
            plan.capture(stream=torch.cuda.Stream())
        else:
            plan.replay()
        torch.cuda.synchronize()
        assert np.array_equal(bits(out_a), bits(hout)), f"step {i}"
    same_cache(ga, gb)
    assert int(ga.err.item()) == 0 and int(gb.err.item()) == 0


def test_host_q_refused_where_tma_loads_it():
    w = wl.small("fp8_verify")
    gc = GpuCase(w, fp8_scales(w))
    rs, rp, k, v, q = append_rows(w, 20, 43)        # 20 rows a stream: verify tiles
    hq = _pinned(q)
    out = torch.full((len(rs), w.hq, 128), 7.0, dtype=torch.bfloat16, device="cuda")
    before = out.clone()
    k_pool = gc.k_pool.clone()
    sc = B.make_scratch(128, w.hq)
    with pytest.raises(B.TfpaError) as e:
        B.tfpa_decode(gc.cache, gc.segs, hq, rs, rp, w.softmax_scale, sc, out)
    assert e.value.code == B.TFPA_EINVAL
    with pytest.raises(B.TfpaError) as e:          # the KV write would have gone first
        B.tfpa_decode_append(gc.cache, gc.segs, k, v, hq, rs, rp, w.softmax_scale, sc, out)
    assert e.value.code == B.TFPA_EINVAL
    torch.cuda.synchronize()
    assert torch.equal(out, before) and torch.equal(gc.k_pool, k_pool)
    wp = wl.small("prompt_chunk")
    gp = GpuCase(wp)
    qp = torch.randn(wp.rows, wp.hq, 128).to(torch.bfloat16).pin_memory()
    op = torch.empty(wp.rows, wp.hq, 128, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(B.TfpaError) as e:
        B.tfpa_prefill(gp.cache, gp.segs, qp, wp.row_seg, wp.row_pos, wp.softmax_scale, op)
    assert e.value.code == B.TFPA_EINVAL


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_kv_write_from_host_rows_equals_device_rows(kv):
    """tfpa_write_kv and tfpa_write_kv_rope reading the new rows from pinned
    host memory store the bytes they store from device rows."""
    w = wl.small("fp8_verify" if kv == "fp8" else "batched_decode")
    scales = fp8_scales(w) if kv == "fp8" else None
    ga, gb = GpuCase(w, scales), GpuCase(w, scales)
    rs, rp, k, v, _ = append_rows(w, 3, 47)
    hk, hv = _pinned(k), _pinned(v)
    B.tfpa_write_kv(ga.cache, ga.segs, k, v, rs, rp)
    B.tfpa_write_kv(gb.cache, gb.segs, hk, hv, rs, rp)
    cos, sin = wl.rope_table(1e6, 4096)
    cos_d, sin_d = torch.from_numpy(cos).cuda(), torch.from_numpy(sin).cuda()
    rp2 = rp - 3                                    # the three positions before
    B.tfpa_write_kv_rope(ga.cache, ga.segs, k, v, rs, rp2, cos_d, sin_d)
    B.tfpa_write_kv_rope(gb.cache, gb.segs, hk, hv, rs, rp2, cos_d, sin_d)
    torch.cuda.synchronize()
    same_cache(ga, gb)
    assert int(ga.err.item()) == 0 and int(gb.err.item()) == 0
