"""The merge inside the decode partial kernel (scratch counters): the same
bytes as the separate merge kernel, for decode rows, draft trees, wide verify
runs next to narrow ones and sliced calls; every call leaves the counters
zero."""

import numpy as np
import pytest
import torch

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, bits, fp8_scales
from tests.test_gpu_verify import _wide_case

pytestmark = pytest.mark.gpu


def _both(g, q, rs, rp, cap, anc=None):
    outs = []
    for fused in (True, False):
        sc = B.make_scratch(cap, g.w.hq, fused_merge=fused)
        out = torch.empty(len(rs), g.w.hq, 128, dtype=torch.bfloat16, device="cuda")
        lse = torch.empty(len(rs), g.w.hq, dtype=torch.float32, device="cuda")
        for _ in range(2):                       # a second call starts from the reset counters
            if anc is None:
                B.tfpa_decode(g.cache, g.segs, q, rs, rp, g.w.softmax_scale, sc, out, lse)
            else:
                B.tfpa_decode_tree(g.cache, g.segs, q, rs, rp, anc, g.w.softmax_scale, sc, out,
                                   lse)
        torch.cuda.synchronize()
        if fused:
            assert int(sc.counters.abs().sum().item()) == 0, "counters left non-zero"
        outs.append((out, lse))
    (a, la), (b, lb) = outs
    assert np.array_equal(bits(a), bits(b))
    assert torch.equal(la, lb)
    assert int(g.err.item()) == 0


@pytest.mark.parametrize("name", ["batched_decode", "fp8_verify", "tiny_paged_decode"])
@pytest.mark.parametrize("cap", [128, 3])
def test_fused_merge_equals_merge_kernel(name, cap):
    w = wl.tiny_paged_decode() if name == "tiny_paged_decode" else wl.small(name)
    g = GpuCase(w, fp8_scales(w) if w.kv_dtype == "fp8" else None)
    _both(g, g.q(), w.row_seg, w.row_pos, cap)


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_fused_merge_next_to_verify_tiles(kv):
    w = _wide_case(kv)
    g = GpuCase(w, fp8_scales(w) if kv == "fp8" else None)
    _both(g, g.q(), w.row_seg, w.row_pos, 128)
    _both(g, g.q(), w.row_seg, w.row_pos, 7)


def test_fused_merge_draft_trees():
    w = wl.small("tree_verify")
    g = GpuCase(w, fp8_scales(w))
    anc = torch.from_numpy(np.ascontiguousarray(np.asarray(w.row_anc, np.uint64))
                           .view(np.int64)).cuda()
    _both(g, g.q(), w.row_seg, w.row_pos, 128, anc)
