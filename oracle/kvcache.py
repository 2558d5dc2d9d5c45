"""The physical KV cache and the KV row write, as plain NumPy.

Test infrastructure only (see the package docstring).

Layout (TensorFold PR #2011, review section "Is paged output the same as
windowed output?": a key of kv head ``hk`` at position ``k`` of a paged stream
lives at ``PT[k/256]*PS + (hk*256 + k%256)*D``; PR #1373 "What changes": the
slab is addressed by cache position as before):

* paged stream: K and V each live in a pool ``[num_pages][hkv][256][D]``; the
  key at position ``j`` of kv head ``g`` is ``pool[PT[j // 256]][g][j % 256]``;
* slab stream: K and V each live in a slab ``[hkv][cap][D]``; the key at
  position ``j`` of kv head ``g`` is ``slab[g][j]``.

One layer per cache.  Storage: bf16 caches hold the bf16 bit patterns
(uint16); fp8 caches hold e4m3 codes (uint8) plus one float32 scale per kv
head for K and one for V, so that ``value = decode(code) * scale[g]``.
"""

from dataclasses import dataclass
from typing import List, Optional

import numpy as np

from . import e4m3

PAGE = 256


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns to float64: a bf16 is the top half of a float32."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32)


@dataclass
class Cache:
    """One layer's KV storage: page pools (may be None if unused) and scales."""
    dtype: str                      # "bf16" or "fp8"
    hkv: int
    d: int
    k_pool: Optional[np.ndarray]    # [num_pages][hkv][256][d]
    v_pool: Optional[np.ndarray]
    k_scale: Optional[np.ndarray] = None   # [hkv] float32, fp8 only
    v_scale: Optional[np.ndarray] = None


@dataclass
class Segment:
    """One stream: its length and either a page table or a pair of slabs."""
    seq_len: int
    page_table: Optional[np.ndarray] = None   # int32 [>= ceil(seq_len/256)]
    k_slab: Optional[np.ndarray] = None       # [hkv][cap][d]
    v_slab: Optional[np.ndarray] = None


def _store(cache: Cache, seg: Segment, which: str, g: int, pos: int):
    """(array, index) of the storage row for (kv head g, position pos)."""
    if seg.page_table is not None:
        page = int(seg.page_table[pos // PAGE])
        arr = cache.k_pool if which == "k" else cache.v_pool
        return arr, (page, g, pos % PAGE)
    arr = seg.k_slab if which == "k" else seg.v_slab
    return arr, (g, pos)


def write_rows(cache: Cache, segs: List[Segment], k_rows: np.ndarray,
               v_rows: np.ndarray, row_seg, row_pos) -> None:
    """Write new K/V rows into their pages or slab (in place).

    ``k_rows``/``v_rows`` are bf16 bit patterns ``[rows][hkv][d]``.  A bf16
    cache stores the bits unchanged; an fp8 cache stores
    ``encode(float32(x) / scale[g])`` (round to nearest even, saturating).
    """
    rows = len(row_seg)
    for r in range(rows):
        seg = segs[int(row_seg[r])]
        pos = int(row_pos[r])
        for g in range(cache.hkv):
            for which, src in (("k", k_rows), ("v", v_rows)):
                arr, idx = _store(cache, seg, which, g, pos)
                if cache.dtype == "bf16":
                    arr[idx] = src[r, g]
                else:
                    sc = cache.k_scale if which == "k" else cache.v_scale
                    arr[idx] = e4m3.quantise(bf16_to_f32(src[r, g]), sc[g])


def _rows_of(arr, page_table, g, n):
    """Raw storage rows 0..n-1 of kv head g, gathered by logical position."""
    if page_table is None:
        return arr[g, :n]
    npages = (n + PAGE - 1) // PAGE
    blocks = [arr[int(page_table[i]), g] for i in range(npages)]
    return np.concatenate(blocks, axis=0)[:n]


def gather(cache: Cache, seg: Segment, g: int, n: int):
    """K and V of kv head ``g`` at positions 0..n-1, dequantised to float64."""
    if seg.page_table is not None:
        k_raw = _rows_of(cache.k_pool, seg.page_table, g, n)
        v_raw = _rows_of(cache.v_pool, seg.page_table, g, n)
    else:
        k_raw = _rows_of(seg.k_slab, None, g, n)
        v_raw = _rows_of(seg.v_slab, None, g, n)
    if cache.dtype == "bf16":
        return bf16_to_f64(k_raw), bf16_to_f64(v_raw)
    ks = np.float64(np.float32(cache.k_scale[g]))
    vs = np.float64(np.float32(cache.v_scale[g]))
    return e4m3.decode(k_raw) * ks, e4m3.decode(v_raw) * vs


def save_image(cache: Cache, seg: Segment, p0: int, p1: int) -> np.ndarray:
    """Stored rows [p0, p1) of a stream, every kv head, K then V, as stored
    (bf16 bits or e4m3 codes): ``[2][hkv][p1 - p0][d]``.  The layout of a
    save/restore image (TensorFold PR #2011 review: save and restore copies)."""
    out = []
    for which in ("k", "v"):
        heads = []
        for g in range(cache.hkv):
            heads.append(np.stack([_store(cache, seg, which, g, p)[0][
                _store(cache, seg, which, g, p)[1]] for p in range(p0, p1)]) if p1 > p0 else
                np.zeros((0, cache.d), dtype=(np.uint16 if cache.dtype == "bf16" else np.uint8)))
        out.append(np.stack(heads))
    return np.stack(out)


def restore_image(cache: Cache, seg: Segment, p0: int, p1: int, image: np.ndarray) -> None:
    """The inverse of ``save_image``: writes the image back into rows [p0, p1) (in place)."""
    for wi, which in enumerate(("k", "v")):
        for g in range(cache.hkv):
            for i, p in enumerate(range(p0, p1)):
                arr, idx = _store(cache, seg, which, g, p)
                arr[idx] = image[wi, g, i]
