"""Softmax attention over the KV cache, one pass, and as split partials.

Test infrastructure only (see the package docstring).

The method (the pages never write the formula out; the plain textbook reading
is taken, as the rest of the pages support): for every row ``r`` with segment
``s = row_seg[r]`` and position ``p = row_pos[r]``, and every query head ``h``
with kv head ``g = h // G`` (``G = hq / hkv``; consecutive query heads share a
kv head, TensorFold PR #1373 "What changes": the tiles "take the key head"):

1. gather ``K[j], V[j]`` of kv head ``g`` for ``j = 0..p`` by logical position
   (through the page table or the slab), dequantised to float64;
2. ``s_j = scale * sum_d q[r,h,d] * K[j,d]``;
3. ``w_j = exp(s_j - max s) / sum_j exp(s_j - max s)``;
4. ``out[r,h] = sum_j w_j V[j]`` and ``lse[r,h] = max s + ln sum_j exp(s_j - max s)``.

The causal rule: a row at position ``p`` sees keys ``0..p`` inclusive; its own
K/V are written before it attends.  Masked keys contribute nothing (PR #2011,
review: masked keys "read offset 0 and land zeros").

Draft-tree verify rows (TensorFold PR #1355, "Follow-up checks": the partial
kernels index the queries, ``rowseg``, ``rowanc``, the partials and the output
by row, and a sliced launch shifts the ancestor table with the other row
tables).  The pages name the per-row ancestor table but do not spell out its
format; the reading taken here: ``row_anc[r]`` is a 64-bit mask relative to
the row's own position ``p``.  Bit ``d`` set means the key at position
``p - d`` is visible to the row; keys more than 63 positions back are always
visible and keys after ``p`` never are.  A causal chain is every bit set.  A
draft tree of at most 64 nodes laid out at consecutive positions sets, for
each node, the bits of its ancestors and itself plus every bit that reaches
below the tree's first position (the committed prefix).  Bit 0 (the row's own
key) must be set.

Split partials (TensorFold Issue #1344, "Mechanism": the partial kernels then
``attn_merge``): a split covers a page-aligned range of positions; for the
visible keys in it ``m = max s`` (``-inf`` if none), ``l = sum exp(s - m)``,
``o = sum exp(s - m) v`` (unnormalised).  The merge takes
``M = max m``, ``L = sum l exp(m - M)``, ``O = sum o exp(m - M) / L`` and
``lse = M + ln L``.  Any page-aligned split gives the same real result.
"""

from typing import List, Sequence

import numpy as np

from .kvcache import PAGE, Cache, Segment, bf16_to_f64, gather


def _check_rows(segs, row_seg, row_pos):
    for r in range(len(row_seg)):
        s = int(row_seg[r])
        p = int(row_pos[r])
        if not (0 <= s < len(segs)):
            raise ValueError(f"row {r}: segment {s} out of range")
        if not (0 <= p < segs[s].seq_len):
            raise ValueError(f"row {r}: position {p} outside 0..{segs[s].seq_len - 1}")


ALL_VISIBLE = (1 << 64) - 1      # the ancestor mask of a causal row


def visible_keys(p: int, anc: int = ALL_VISIBLE) -> np.ndarray:
    """Positions a row at position ``p`` with ancestor mask ``anc`` sees, ascending."""
    anc = int(anc) & ALL_VISIBLE
    if not anc & 1:
        raise ValueError("an ancestor mask must let a row see its own key (bit 0)")
    keys = [j for j in range(max(0, p - 63), p + 1) if (anc >> (p - j)) & 1]
    return np.concatenate([np.arange(0, max(0, p - 63), dtype=np.int64),
                           np.asarray(keys, dtype=np.int64)])


def attend(cache: Cache, segs: List[Segment], q_bits: np.ndarray,
           row_seg: Sequence[int], row_pos: Sequence[int], scale: float,
           row_anc: Sequence[int] = None):
    """One-pass GQA attention.  Returns (out [rows][hq][d], lse [rows][hq]).

    ``q_bits`` holds bf16 bit patterns ``[rows][hq][d]``; all arithmetic is
    float64.  Rows are causal, or see the keys their ancestor mask
    ``row_anc[r]`` allows.  Rows are grouped by segment only so each (segment,
    kv head) is gathered once; every row is computed on its own.
    """
    rows, hq, d = q_bits.shape
    hkv = cache.hkv
    if hq % hkv:
        raise ValueError("hq must be a multiple of hkv")
    G = hq // hkv
    _check_rows(segs, row_seg, row_pos)
    q = bf16_to_f64(q_bits)
    out = np.zeros((rows, hq, d), dtype=np.float64)
    lse = np.zeros((rows, hq), dtype=np.float64)
    by_seg = {}
    for r in range(rows):
        by_seg.setdefault(int(row_seg[r]), []).append(r)
    for s, rs in by_seg.items():
        n = max(int(row_pos[r]) for r in rs) + 1
        for g in range(hkv):
            K, V = gather(cache, segs[s], g, n)
            for r in rs:
                p = int(row_pos[r])
                if row_anc is None:
                    Kp, Vp = K[: p + 1], V[: p + 1]
                else:
                    idx = visible_keys(p, row_anc[r])
                    Kp, Vp = K[idx], V[idx]
                Q = q[r, g * G:(g + 1) * G]             # [G][d]
                S = scale * (Q @ Kp.T)                  # [G][p+1]
                mx = S.max(axis=1, keepdims=True)
                E = np.exp(S - mx)
                Z = E.sum(axis=1, keepdims=True)
                out[r, g * G:(g + 1) * G] = (E @ Vp) / Z
                lse[r, g * G:(g + 1) * G] = mx[:, 0] + np.log(Z[:, 0])
    return out, lse


def split_ranges(seq_len: int, pages_per_split: int):
    """Page-aligned key ranges [lo, hi) covering 0..seq_len-1."""
    step = pages_per_split * PAGE
    return [(lo, min(lo + step, seq_len)) for lo in range(0, seq_len, step)]


def attend_partials(cache: Cache, segs: List[Segment], q_bits: np.ndarray,
                    row_seg, row_pos, scale: float, pages_per_split, row_anc=None):
    """Split partials per (row, head, split).

    ``pages_per_split`` is an int or a callable ``seq_len -> int``.  Returns
    ``(m, l, o, nsplit)`` with ``m, l: [rows][hq][S]``, ``o: [rows][hq][S][d]``
    (``S`` = the largest split count; unused slots hold ``m = -inf, l = 0,
    o = 0``) and ``nsplit: [rows]``.
    """
    rows, hq, d = q_bits.shape
    hkv = cache.hkv
    G = hq // hkv
    _check_rows(segs, row_seg, row_pos)
    pps = pages_per_split if callable(pages_per_split) else (lambda L: pages_per_split)
    ranges = [split_ranges(segs[int(row_seg[r])].seq_len, pps(segs[int(row_seg[r])].seq_len))
              for r in range(rows)]
    S_max = max(len(x) for x in ranges)
    m = np.full((rows, hq, S_max), -np.inf)
    l = np.zeros((rows, hq, S_max))
    o = np.zeros((rows, hq, S_max, d))
    q = bf16_to_f64(q_bits)
    for r in range(rows):
        s = int(row_seg[r])
        p = int(row_pos[r])
        for g in range(hkv):
            K, V = gather(cache, segs[s], g, segs[s].seq_len)
            for h in range(g * G, (g + 1) * G):
                vis = visible_keys(p, ALL_VISIBLE if row_anc is None else row_anc[r])
                for si, (lo, hi) in enumerate(ranges[r]):
                    idx = vis[(vis >= lo) & (vis < hi)]
                    if idx.size == 0:
                        continue  # no visible key in this split
                    sc = scale * (K[idx] @ q[r, h])
                    mm = sc.max()
                    e = np.exp(sc - mm)
                    m[r, h, si] = mm
                    l[r, h, si] = e.sum()
                    o[r, h, si] = e @ V[idx]
    nsplit = np.array([len(x) for x in ranges], dtype=np.int64)
    return m, l, o, nsplit


def merge(m: np.ndarray, l: np.ndarray, o: np.ndarray):
    """Log-sum-exp merge of split partials over the last split axis.

    ``m, l: [..., S]``, ``o: [..., S, d]``.  Empty splits (``m = -inf``) carry
    weight 0.  Returns ``(out [..., d], lse [...])``.
    """
    M = m.max(axis=-1, keepdims=True)
    if np.any(~np.isfinite(M)):
        raise ValueError("a (row, head) has no visible key")
    w = np.where(np.isfinite(m), np.exp(m - M), 0.0)
    L = (w * l).sum(axis=-1)
    O = (w[..., None] * o).sum(axis=-2) / L[..., None]
    return O, M[..., 0] + np.log(L)
