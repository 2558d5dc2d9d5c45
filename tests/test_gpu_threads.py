"""Calls from several host threads at once: each thread plans its launches in
its own buffers (no lock on the call path), so concurrent calls on separate
streams give exactly the bytes of the same calls made one at a time."""

import threading

import numpy as np
import pytest
import torch

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, bits

pytestmark = pytest.mark.gpu


def test_two_host_threads_decode_concurrently_on_two_streams():
    cases = [GpuCase(wl.small("batched_decode")), GpuCase(wl.small("fp8_verify"))]
    qs = [g.q() for g in cases]
    refs = [g.decode(q, g.w.row_seg, g.w.row_pos)[0] for g, q in zip(cases, qs)]
    calls = 50
    outs = [[torch.empty_like(r) for _ in range(calls)] for r in refs]
    errors = []
    start = threading.Barrier(len(cases))

    def worker(i):
        try:
            g, q = cases[i], qs[i]
            sc = B.make_scratch(128, g.w.hq)
            st = torch.cuda.Stream()
            st.wait_stream(torch.cuda.current_stream())
            start.wait()
            for k in range(calls):
                B.tfpa_decode(g.cache, g.segs, q, g.w.row_seg, g.w.row_pos, g.w.softmax_scale,
                              sc, outs[i][k], stream=st)
            st.synchronize()
        except Exception as e:          # reported by the main thread
            errors.append(e)

    ts = [threading.Thread(target=worker, args=(i,)) for i in range(len(cases))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    assert not errors, errors
    for i, r in enumerate(refs):
        for k in range(calls):
            assert np.array_equal(bits(outs[i][k]), bits(r)), (i, k)
    assert all(int(g.err.item()) == 0 for g in cases)
