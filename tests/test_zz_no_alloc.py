"""tfpa_decode_static: decode for callers that cannot allocate device memory
(a plug-in inside another framework's memory manager, a runtime that makes
all its allocations before serving).  Its split-K partials live in an array
compiled into the library; its output must match tfpa_decode's.

This file is collected last on purpose, so a run that stops at the first
failure has run every other test before it."""

import numpy as np
import pytest

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, assert_close, bits, fp8_scales, to_f64

pytestmark = pytest.mark.gpu

TOL = {"bf16": 1e-2, "fp8": 3e-2}


@pytest.mark.parametrize("name", ["fp8_verify", "batched_decode"])
def test_static_scratch_decode_matches_decode(name):
    import torch
    w = wl.small(name)
    scales = fp8_scales(w) if w.kv_dtype == "fp8" else None
    g = GpuCase(w, scales)
    q = g.q()
    ref, ref_lse = g.decode(q, w.row_seg, w.row_pos)
    for call in range(2):                      # two calls in a row share the array
        out = torch.empty_like(ref)
        lse = torch.empty_like(ref_lse)
        B.tfpa_decode_static(g.cache, g.segs, q, w.row_seg, w.row_pos, w.softmax_scale, out, lse)
        torch.cuda.synchronize()
        assert_close(to_f64(out), to_f64(ref), TOL[w.kv_dtype], f"{name} call {call}")
        assert_close(to_f64(lse), to_f64(ref_lse), 1e-3, f"{name} lse call {call}")
        # the rows run in smaller slices; slicing never changes a row's bytes
        assert np.array_equal(bits(out), bits(ref))


def test_static_scratch_wide_run_matches_decode_bitwise():
    """A 64-row run of one stream (256 query vectors per kv head at 32 / 8
    heads) takes the tensor-core verify kernel; through the library's array it
    runs in slices of 8 rows, and still gives tfpa_decode's bytes."""
    import torch
    from tests.test_gpu_edges import _make
    L = 5000
    w = _make([L], [True], [0] * 64, list(range(L - 64, L)), 32, 8, "bf16", seed=615)
    g = GpuCase(w)
    q = g.q()
    ref, ref_lse = g.decode(q, w.row_seg, w.row_pos)
    for call in range(2):
        out = torch.empty_like(ref)
        lse = torch.empty_like(ref_lse)
        B.tfpa_decode_static(g.cache, g.segs, q, w.row_seg, w.row_pos, w.softmax_scale, out, lse)
        torch.cuda.synchronize()
        assert np.array_equal(bits(out), bits(ref)), f"call {call}"
        assert torch.equal(lse, ref_lse)


def test_static_scratch_refuses_head_counts_beyond_its_size():
    import torch
    w = wl.small("batched_decode")
    g = GpuCase(w)
    big = B.Cache("bf16", 512, 8, g.k_pool, g.v_pool, None, None, None, w.num_pages)
    q = torch.zeros(1, 512, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.empty_like(q)
    with pytest.raises(B.TfpaError) as e:
        B.tfpa_decode_static(big, g.segs[:1], q, [0], [0], 0.088, out)
    assert e.value.code == B.TFPA_ECAPACITY
