"""KV store with rotary position embedding, and the keep copy, as plain NumPy.

Test infrastructure only (see the package docstring).

The pages list these among the checks of the paged KV store (TensorFold PR
#1373, review: "rope stores and keep", "paged == contiguous for queries, rows,
stores and keep") without spelling out either operation.  Readings taken:

* RoPE store: before a new row's K is stored, it is rotated by its rotary
  position ``t`` in the rotate-half pairing of the head dimension: for
  ``i < 64``, with ``c = cos_t[i]`` and ``s = sin_t[i]`` from the caller's
  float32 table, ``k'[i] = k[i] c - k[i+64] s`` and
  ``k'[i+64] = k[i+64] c + k[i] s``.  Every product, difference and sum is
  rounded to float32 (no fused multiply-add), so the stored code is fixed by
  the inputs.  V is stored as is.  bf16 caches store ``k'`` rounded to bf16
  (nearest, ties to even); e4m3 caches store ``e4m3(k' / scale[g])`` as the
  plain store does.  The rotary position may differ from the storage
  position (a draft-tree node is rotated by its depth, stored at its index).
* keep: stored K/V rows are copied byte for byte from one position of a
  stream to another, all kv heads; a call reads every source row before it
  writes any destination, so chains of moves (2 -> 1, 5 -> 2) are exact.
"""

from typing import List, Sequence

import numpy as np

from . import e4m3
from .kvcache import Cache, Segment, _store, bf16_to_f32

HALF = 64


def f32_to_bf16(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit patterns, round to nearest, ties to even."""
    u = np.asarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    lsb = (u >> 16) & 1
    r = ((u + 0x7FFF + lsb) >> 16) & 0xFFFF
    r = np.where(nan, (u >> 16) | 0x40, r)           # keep NaN a (quiet) NaN
    return r.astype(np.uint16)


def rope_f32(k_bits: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """One row's K (bf16 bits, [128]) rotated with float32 cos/sin [64]: float32 [128]."""
    k = bf16_to_f32(k_bits)
    a, b = k[:HALF], k[HALF:]
    c = np.asarray(cos, dtype=np.float32)
    s = np.asarray(sin, dtype=np.float32)
    out = np.empty(2 * HALF, dtype=np.float32)
    out[:HALF] = (a * c).astype(np.float32) - (b * s).astype(np.float32)
    out[HALF:] = (b * c).astype(np.float32) + (a * s).astype(np.float32)
    return out


def write_rows_rope(cache: Cache, segs: List[Segment], k_rows: np.ndarray, v_rows: np.ndarray,
                    row_seg, row_pos, rope_pos, cos_tab: np.ndarray, sin_tab: np.ndarray):
    """As ``kvcache.write_rows``, with K rotated by ``rope_pos[r]`` (in place)."""
    for r in range(len(row_seg)):
        seg = segs[int(row_seg[r])]
        pos = int(row_pos[r])
        t = int(rope_pos[r])
        for g in range(cache.hkv):
            kf = rope_f32(k_rows[r, g], cos_tab[t], sin_tab[t])
            arr, idx = _store(cache, seg, "k", g, pos)
            if cache.dtype == "bf16":
                arr[idx] = f32_to_bf16(kf)
            else:
                arr[idx] = e4m3.quantise(kf, cache.k_scale[g])
            arr, idx = _store(cache, seg, "v", g, pos)
            if cache.dtype == "bf16":
                arr[idx] = v_rows[r, g]
            else:
                arr[idx] = e4m3.quantise(bf16_to_f32(v_rows[r, g]), cache.v_scale[g])


def keep_rows(cache: Cache, segs: List[Segment], keep_seg: Sequence[int],
              keep_src: Sequence[int], keep_dst: Sequence[int]):
    """Copy stored rows (all kv heads, K and V) from src to dst positions (in place).

    Every source row is read before any destination is written.
    """
    saved = []
    for s, src in zip(keep_seg, keep_src):
        seg = segs[int(s)]
        rows = []
        for g in range(cache.hkv):
            for which in ("k", "v"):
                arr, idx = _store(cache, seg, which, g, int(src))
                rows.append(arr[idx].copy())
        saved.append(rows)
    for s, dst, rows in zip(keep_seg, keep_dst, saved):
        seg = segs[int(s)]
        i = 0
        for g in range(cache.hkv):
            for which in ("k", "v"):
                arr, idx = _store(cache, seg, which, g, int(dst))
                arr[idx] = rows[i]
                i += 1
