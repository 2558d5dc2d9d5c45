"""Page-table staging and save/restore on the GPU: staged ids land in the
device table; saved images (pinned host and device memory) equal the
oracle's byte for byte; a stream saved to host memory and restored into
pages claimed from the ledger and staged into a new table decodes to the same
bits as before."""

import numpy as np
import pytest
import torch

from oracle import kvcache
from paged_kv_cache_235_gb300 import binding as B
from paged_kv_cache_235_gb300 import workloads as wl
from tests.gpu_cases import GpuCase, bits, fp8_scales
from tests.oracle_cases import build_oracle_cache

pytestmark = pytest.mark.gpu


def _mixed(kv, lengths=(700, 300, 1100), paged=(True, False, True), seed=73, slack=12):
    npages = sum((L + 255) // 256 for L, p in zip(lengths, paged) if p) + slack
    tables = wl.permuted_tables(list(lengths), list(paged), npages, seed)
    streams = [wl.Stream(L, p, t, 0 if p else ((L + 255) // 256) * 256)
               for L, p, t in zip(lengths, paged, tables)]
    return wl.Workload("copy", 8, 2, kv, npages, streams, np.zeros(1, np.int32),
                       np.zeros(1, np.int32), seed)


def test_stage_pages_lands_in_the_device_table():
    table = torch.full((5000,), -7, dtype=torch.int32, device="cuda")
    ids = np.random.default_rng(1).integers(0, 10**6, size=3000).astype(np.int32)
    B.tfpa_stage_pages(table, 1000, ids)
    torch.cuda.synchronize()
    t = table.cpu().numpy()
    assert np.array_equal(t[1000:4000], ids)
    assert (t[:1000] == -7).all() and (t[4000:] == -7).all()


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
@pytest.mark.parametrize("s,p0,p1", [(0, 0, 700), (2, 300, 700), (2, 255, 257), (1, 17, 300)])
@pytest.mark.parametrize("where", ["pinned", "device"])
def test_saved_image_matches_oracle(kv, s, p0, p1, where):
    w = _mixed(kv)
    scales = fp8_scales(w) if kv == "fp8" else None
    g = GpuCase(w, scales)
    cache_o, segs_o = build_oracle_cache(w, *(scales or (None, None)))
    ref = kvcache.save_image(cache_o, segs_o[s], p0, p1)
    nbytes = ref.nbytes
    if where == "pinned":
        img = torch.empty(nbytes, dtype=torch.uint8, pin_memory=True)
    else:
        img = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    B.tfpa_save_kv(g.cache, g.segs[s], p0, p1, img)
    torch.cuda.synchronize()
    assert np.array_equal(img.cpu().numpy(), ref.reshape(-1).view(np.uint8))
    assert int(g.err.item()) == 0


@pytest.mark.parametrize("kv", ["bf16", "fp8"])
def test_save_claim_stage_restore_decodes_the_same(kv):
    w = _mixed(kv)
    scales = fp8_scales(w) if kv == "fp8" else None
    g = GpuCase(w, scales)
    L = w.streams[2].seq_len
    q = torch.randn(2, 8, 128, device="cuda").to(torch.bfloat16)
    before, lse_b = g.decode(q, [2, 2], [L - 2, L - 1])
    elem = 1 if kv == "fp8" else 2
    img = torch.empty(2 * 2 * L * 128 * elem, dtype=torch.uint8, pin_memory=True)
    B.tfpa_save_kv(g.cache, g.segs[2], 0, L, img)
    # fresh pages for the restored stream from the ledger, staged into a new table
    pool = B.Pool(w.num_pages)
    npages = (L + 255) // 256
    pages = pool.claim(npages)
    table = torch.empty(npages, dtype=torch.int32, device="cuda")
    B.tfpa_stage_pages(table, 0, pages)
    seg = B.Seg(L, page_table=table, page_table_host=pages)
    B.tfpa_restore_kv(g.cache, seg, 0, L, img)
    segs = list(g.segs)
    segs[2] = seg
    after, lse_a = g.decode(q, [2, 2], [L - 2, L - 1], segs=segs)
    assert np.array_equal(bits(before), bits(after))
    assert np.array_equal(lse_b.cpu().numpy(), lse_a.cpu().numpy())
    assert int(g.err.item()) == 0
