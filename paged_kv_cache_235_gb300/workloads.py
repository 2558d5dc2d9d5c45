"""Seeded synthetic workloads shaped like the pages' attention calls.

This module generates inputs only: random values, page tables, row tables and
per-head fp8 scales.  It holds none of the attention arithmetic, so both the
CUDA path (through the binding) and the CPU oracle can be fed from it.

Shapes follow the pages' workloads (TensorFold PR #1373 checks: 8 streams at
65,536 positions on 256-position pages; PR #2011 receipt: 4,096-row prompt
chunks, a 32k prompt, 16 streams of about 109k tokens in a 1.30M-row pool).
Values are N(0, 1) float32 from ``torch.Generator`` on the CPU, rounded to
bf16; fp8 caches take per-kv-head scales ``amax / 448`` of the values written.
"""

from dataclasses import dataclass, field
from typing import List, Optional

import math
import numpy as np
import torch

PAGE = 256
HEAD_DIM = 128


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator()
    g.manual_seed(int(seed) & 0x7FFFFFFFFFFFFFFF)
    return g


def randn_bf16_bits(shape, seed: int) -> np.ndarray:
    """N(0,1) float32 rounded to bf16, returned as uint16 bit patterns."""
    x = torch.randn(*shape, generator=_gen(seed), dtype=torch.float32)
    return x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def random_fp8_codes(shape, seed: int) -> np.ndarray:
    """Random e4m3 codes with the two NaN codes (0x7F, 0xFF) avoided."""
    c = torch.randint(0, 254, tuple(shape), generator=_gen(seed), dtype=torch.uint8)
    c += (c >= 0x7F).to(torch.uint8)      # skip 0x7F; 254 values -> 0..0xFE
    return c.numpy()


@dataclass
class Stream:
    seq_len: int
    paged: bool
    page_table: Optional[np.ndarray] = None   # int32, length ceil(seq_len/256)
    slab_cap: int = 0                          # positions, multiple of 256


@dataclass
class Workload:
    """One attention call: cache geometry, streams, rows and value seeds."""
    name: str
    hq: int
    hkv: int
    kv_dtype: str                 # "bf16" or "fp8"
    num_pages: int
    streams: List[Stream]
    row_seg: np.ndarray           # int32 [rows]
    row_pos: np.ndarray           # int32 [rows]
    seed: int
    d: int = HEAD_DIM
    waiting: List[int] = field(default_factory=list)  # streams not seated
    row_anc: Optional[np.ndarray] = None   # uint64 [rows] ancestor masks; None = causal

    @property
    def rows(self) -> int:
        return int(len(self.row_seg))

    @property
    def softmax_scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    # ---- values -------------------------------------------------------
    def stream_kv_bits(self, s: int):
        """Logical K and V of stream ``s``: bf16 bits ``[hkv][seq_len][d]``."""
        L = self.streams[s].seq_len
        k = randn_bf16_bits((self.hkv, L, self.d), self.seed * 1_000_003 + 2 * s + 1)
        v = randn_bf16_bits((self.hkv, L, self.d), self.seed * 1_000_003 + 2 * s + 2)
        return k, v

    def q_bits(self) -> np.ndarray:
        """Query rows: bf16 bits ``[rows][hq][d]``."""
        return randn_bf16_bits((self.rows, self.hq, self.d), self.seed * 1_000_003 + 999_983)

    def filler_seed(self, which: str) -> int:
        return self.seed * 1_000_003 + (500_009 if which == "k" else 500_011)

    def fp8_scales(self):
        """Per-kv-head float32 scales ``amax / 448`` over every stream's values."""
        ka = np.zeros(self.hkv, dtype=np.float32)
        va = np.zeros(self.hkv, dtype=np.float32)
        for s in range(len(self.streams)):
            k, v = self.stream_kv_bits(s)
            kf = (k.astype(np.uint32) << 16).view(np.float32)
            vf = (v.astype(np.uint32) << 16).view(np.float32)
            ka = np.maximum(ka, np.abs(kf).max(axis=(1, 2)))
            va = np.maximum(va, np.abs(vf).max(axis=(1, 2)))
        return (ka / np.float32(448.0)).astype(np.float32), (va / np.float32(448.0)).astype(np.float32)


def _pages(L: int) -> int:
    return (L + PAGE - 1) // PAGE


def decode_rows(lengths, rows_per_stream):
    """Rows of a decode/verify call: each stream's last R positions, in order."""
    seg, pos = [], []
    for s, L in enumerate(lengths):
        R = rows_per_stream if isinstance(rows_per_stream, int) else rows_per_stream[s]
        for i in range(R):
            seg.append(s)
            pos.append(L - R + i)
    return np.array(seg, dtype=np.int32), np.array(pos, dtype=np.int32)


ALL_VISIBLE = (1 << 64) - 1


def tree_masks(parents) -> List[int]:
    """Ancestor masks of a draft tree laid out at consecutive positions.

    Node ``i`` sits at position ``base + i`` and ``parents[i] < i`` is its
    parent (``parents[0] = -1``: the root).  The mask of node ``i`` is relative
    to its own position: bit ``d`` set means the key ``d`` positions back is
    visible.  It holds node ``i``, its ancestors, and every position before
    the root (the committed prefix).  At most 64 nodes.
    """
    n = len(parents)
    if n > 64:
        raise ValueError("at most 64 tree nodes")
    masks = []
    for i in range(n):
        m = ALL_VISIBLE & ~((1 << (i + 1)) - 1)      # bits i+1..63: before the root
        a = i
        while a >= 0:
            m |= 1 << (i - a)
            a = parents[a]
        masks.append(m)
    return masks


def rope_table(theta: float, n_pos: int, d: int = HEAD_DIM):
    """The caller's rotary table: float32 cos and sin ``[n_pos][d / 2]`` of
    ``t * theta ** (-2 i / d)``, computed in float64 and rounded once."""
    i = np.arange(d // 2, dtype=np.float64)
    inv = theta ** (-2.0 * i / d)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


def tree_depths(parents) -> List[int]:
    """Depth of each node of a draft tree (the root has depth 0)."""
    depth = []
    for i, par in enumerate(parents):
        depth.append(0 if par < 0 else depth[par] + 1)
    return depth


def random_tree(n: int, seed: int) -> List[int]:
    """Parents of a seeded random recursive tree of ``n`` nodes (node 0 the root)."""
    rng = np.random.default_rng(seed)
    return [-1] + [int(rng.integers(0, i)) for i in range(1, n)]


def permuted_tables(lengths, paged_flags, num_pages: int, seed: int):
    """Page tables from one seeded permutation of the pool, dealt in order."""
    perm = torch.randperm(num_pages, generator=_gen(seed)).numpy().astype(np.int32)
    need = sum(_pages(L) for L, p in zip(lengths, paged_flags) if p)
    if need > num_pages:
        raise ValueError("pool too small")
    tables, at = [], 0
    for L, p in zip(lengths, paged_flags):
        if p:
            n = _pages(L)
            tables.append(perm[at:at + n].copy())
            at += n
        else:
            tables.append(None)
    return tables


class FirstFitPool:
    """A page pool with seeded churn and first-fit claims of whole requests.

    A request claims all of its pages up front or waits (TensorFold PR #2011,
    review "Memory admission": pages are claimed when a request is seated; a
    full or fragmented pool makes it wait).  Pages are handed out lowest
    free index first.
    """

    def __init__(self, num_pages: int):
        self.free = np.ones(num_pages, dtype=bool)

    def claim(self, n: int):
        idx = np.flatnonzero(self.free)
        if len(idx) < n:
            return None
        got = idx[:n]
        self.free[got] = False
        return got.astype(np.int32)

    def release(self, pages):
        self.free[np.asarray(pages)] = True

    def churn(self, seed: int, rounds: int, max_pages: int, keep_fraction: float):
        """Claim and release random-size runs so later claims are fragmented."""
        rng = np.random.default_rng(seed)
        held = []
        for _ in range(rounds):
            n = int(rng.integers(1, max_pages + 1))
            got = self.claim(n)
            if got is not None:
                held.append(got)
            if held and rng.random() < 0.5:
                self.release(held.pop(int(rng.integers(len(held)))))
        # Keep a fraction of the held runs as other tenants of the pool.
        rng.shuffle(held)
        keep = int(len(held) * keep_fraction)
        for h in held[keep:]:
            self.release(h)


# ---------------------------------------------------------------------------
# The five workloads.  ``small=True`` scales a workload down to a size the
# oracle finishes in seconds while keeping its structure (several tiles and a
# ragged tail).
# ---------------------------------------------------------------------------

def tiny_paged_decode(seed: int = 236) -> Workload:
    """1 stream, 1 row; 8/2 heads; 1,000 positions in 4 pages of a 16-page pool."""
    L = 1000
    tables = permuted_tables([L], [True], 16, seed)
    rs, rp = decode_rows([L], 1)
    return Workload("tiny_paged_decode", 8, 2, "bf16", 16,
                    [Stream(L, True, tables[0])], rs, rp, seed)


def batched_decode(seed: int = 237, seq_len: int = 8192, n_streams: int = 8,
                   num_pages: int = 512) -> Workload:
    """8 streams, 1 row each; 32/8 heads; bf16; streams 0-3 slabs, 4-7 paged."""
    lengths = [seq_len] * n_streams
    paged = [s >= n_streams // 2 for s in range(n_streams)]
    tables = permuted_tables(lengths, paged, num_pages, seed)
    streams = [Stream(L, p, t, 0 if p else _pages(L) * PAGE)
               for L, p, t in zip(lengths, paged, tables)]
    rs, rp = decode_rows(lengths, 1)
    return Workload("batched_decode", 32, 8, "bf16", num_pages, streams, rs, rp, seed)


def fp8_verify(seed: int = 238, seq_len: int = 65536, n_streams: int = 8,
               slack_pages: int = 64) -> Workload:
    """8 streams x 4 causal verify rows; 32/8 heads; fp8 e4m3 KV, all paged."""
    lengths = [seq_len] * n_streams
    num_pages = sum(_pages(L) for L in lengths) + slack_pages
    tables = permuted_tables(lengths, [True] * n_streams, num_pages, seed)
    streams = [Stream(L, True, t) for L, t in zip(lengths, tables)]
    rs, rp = decode_rows(lengths, 4)
    return Workload("fp8_verify", 32, 8, "fp8", num_pages, streams, rs, rp, seed)


def tree_verify(seed: int = 241, seq_len: int = 65536, n_streams: int = 8, nodes: int = 16,
                kv_dtype: str = "fp8", slack_pages: int = 64) -> Workload:
    """Draft-tree verify: each stream's last ``nodes`` positions hold a seeded
    random draft tree, one row per node, attending through ancestor masks."""
    lengths = [seq_len] * n_streams
    num_pages = sum(_pages(L) for L in lengths) + slack_pages
    tables = permuted_tables(lengths, [True] * n_streams, num_pages, seed)
    streams = [Stream(L, True, t) for L, t in zip(lengths, tables)]
    rs, rp = decode_rows(lengths, nodes)
    anc = []
    for s in range(n_streams):
        anc += tree_masks(random_tree(nodes, seed * 1_000_003 + 77 + s))
    w = Workload("tree_verify", 32, 8, kv_dtype, num_pages, streams, rs, rp, seed)
    w.row_anc = np.array(anc, dtype=np.uint64)
    return w


def prompt_chunk(seed: int = 239, prefix: int = 28672, chunk: int = 4096,
                 slack_pages: int = 32, paged: bool = True, kv_dtype: str = "bf16") -> Workload:
    """One stream: a paged prefix plus a causal chunk of rows; 32/8 heads."""
    L = prefix + chunk
    num_pages = _pages(L) + slack_pages
    tables = permuted_tables([L], [paged], num_pages, seed)
    st = Stream(L, paged, tables[0], 0 if paged else _pages(L) * PAGE)
    rs = np.zeros(chunk, dtype=np.int32)
    rp = np.arange(prefix, L, dtype=np.int32)
    return Workload("prompt_chunk", 32, 8, kv_dtype, num_pages, [st], rs, rp, seed)


def overcommitted_pool(seed: int = 240, n_short: int = 16, lo: int = 1000,
                       hi: int = 109_000, long_len: int = 262_144,
                       pool_rows: int = 1_300_000) -> Workload:
    """16 streams of U[1k,109k] positions plus one of 262,144; fp8; first-fit pool.

    Streams that do not fit wait and are left out of the call (recorded in
    ``waiting``).
    """
    rng = np.random.default_rng(seed)
    lengths = [int(x) for x in rng.integers(lo, hi + 1, size=n_short)] + [long_len]
    num_pages = pool_rows // PAGE
    pool = FirstFitPool(num_pages)
    pool.churn(seed + 1, rounds=400, max_pages=24, keep_fraction=0.25)
    streams, waiting = [], []
    for s, L in enumerate(lengths):
        got = pool.claim(_pages(L))
        if got is None:
            waiting.append(s)
            continue
        streams.append(Stream(L, True, got))
    seated_lengths = [st.seq_len for st in streams]
    rs, rp = decode_rows(seated_lengths, 1)
    w = Workload("overcommitted_pool", 32, 8, "fp8", num_pages, streams, rs, rp, seed)
    w.waiting = waiting
    return w


def small(w_name: str, seed: int = 1235) -> Workload:
    """Oracle-sized versions of the workloads, same structure."""
    if w_name == "tiny_paged_decode":
        return tiny_paged_decode(seed)
    if w_name == "batched_decode":
        return batched_decode(seed, seq_len=1000, n_streams=4, num_pages=24)
    if w_name == "fp8_verify":
        return fp8_verify(seed, seq_len=1300, n_streams=3, slack_pages=5)
    if w_name == "prompt_chunk":
        return prompt_chunk(seed, prefix=300, chunk=257, slack_pages=3)
    if w_name == "tree_verify":
        return tree_verify(seed, seq_len=1300, n_streams=3, nodes=20, kv_dtype="fp8",
                           slack_pages=5)
    if w_name == "overcommitted_pool":
        return overcommitted_pool(seed, n_short=5, lo=100, hi=2000, long_len=3000,
                                  pool_rows=60 * PAGE)
    raise KeyError(w_name)
