"""KV write on the GPU: pool and slab bytes equal the oracle's, bit for bit."""

import numpy as np
import pytest
import torch

from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, fp8_scales
from tests.oracle_cases import build_oracle_cache

pytestmark = pytest.mark.gpu


def _host_bytes(t):
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


@pytest.mark.parametrize("name", ["batched_decode", "fp8_verify", "prompt_chunk",
                                  "overcommitted_pool"])
def test_cache_bytes_equal_oracle(name):
    w = wl.small(name)
    scales = fp8_scales(w) if w.kv_dtype == "fp8" else (None, None)
    g = GpuCase(w, scales if w.kv_dtype == "fp8" else None)
    oc, osegs = build_oracle_cache(w, *scales)
    assert np.array_equal(_host_bytes(g.k_pool), oc.k_pool)
    assert np.array_equal(_host_bytes(g.v_pool), oc.v_pool)
    for gs, os_ in zip(g.segs, osegs):
        if os_.k_slab is not None:
            assert np.array_equal(_host_bytes(gs.k_slab), os_.k_slab)
            assert np.array_equal(_host_bytes(gs.v_slab), os_.v_slab)
    assert int(g.err.item()) == 0


def test_fp8_quantisation_edges():
    """Ties, saturation and signed zero of the e4m3 store, against the oracle."""
    from oracle import e4m3
    hkv = 1
    vals = np.concatenate([
        e4m3.decode(np.arange(0x7F, dtype=np.uint8)),                 # every code
        (e4m3.decode(np.arange(0x7E, dtype=np.uint8)) +
         e4m3.decode(np.arange(1, 0x7F, dtype=np.uint8))) / 2,       # midpoints
        [500.0, 1e4, -1e4, -0.0, 1e-30, -1e-30],
    ]).astype(np.float32)
    vals = np.concatenate([vals, -vals])
    bf = torch.from_numpy(vals).to(torch.bfloat16)          # values as bf16 rows
    n = (len(vals) + 127) // 128
    rows = torch.zeros(n * 128, dtype=torch.bfloat16)
    rows[: len(vals)] = bf
    rows = rows.view(n, hkv, 128).cuda()
    scale = torch.ones(hkv, dtype=torch.float32, device="cuda")
    pool = torch.zeros(1, hkv, 256, 128, dtype=torch.uint8, device="cuda")
    cache = B.Cache("fp8", 1, hkv, pool, pool.clone(), scale, scale, None, 1)
    seg = B.Seg(n, page_table=torch.zeros(1, dtype=torch.int32, device="cuda"))
    B.tfpa_write_kv(cache, [seg], rows, rows, np.zeros(n, np.int32), np.arange(n))
    torch.cuda.synchronize()
    got = pool[0, 0, :n].cpu().numpy().ravel()
    x = rows.view(torch.int16).cpu().numpy().view(np.uint16).ravel()
    want = e4m3.quantise((x.astype(np.uint32) << 16).view(np.float32), np.float32(1.0))
    assert np.array_equal(got, want)
