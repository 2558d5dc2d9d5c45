"""Thin ctypes binding of libtfpa.so: the same entry-point names as the C ABI.

Only argument marshalling happens here: tensors become device pointers, row
tables become host int32 arrays, the current torch stream becomes the
``cudaStream_t``.  Every step of the attention runs in the library's kernels.
Loading fails loudly if the library has not been built.
"""

import contextlib
import ctypes
import os
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import numpy as np

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libtfpa.so")

PAGE = 256
HEAD_DIM = 128
MAX_SPLITS = 32
BF16, FP8_E4M3 = 0, 1

TFPA_OK, TFPA_EINVAL, TFPA_ERANGE, TFPA_ECAPACITY, TFPA_ECUDA, TFPA_EDEVICE = 0, -1, -2, -3, -4, -5
TFPA_ELANEMEM = -6

EXPORTS = ("tfpa_pages_per_split", "tfpa_num_splits", "tfpa_write_kv", "tfpa_decode_partial",
           "tfpa_merge", "tfpa_decode", "tfpa_prefill", "tfpa_set_launch_hook",
           "tfpa_strerror", "tfpa_version", "tfpa_decode_static", "tfpa_decode_tree",
           "tfpa_write_kv_rope", "tfpa_keep_kv", "tfpa_pool_create", "tfpa_pool_destroy",
           "tfpa_pool_free", "tfpa_pool_fits", "tfpa_pool_claim", "tfpa_pool_release",
           "tfpa_stage_pages", "tfpa_save_kv", "tfpa_restore_kv", "tfpa_plan_create",
           "tfpa_plan_destroy", "tfpa_plan_clear", "tfpa_plan_launches", "tfpa_plan_write_kv",
           "tfpa_plan_decode", "tfpa_plan_launch", "tfpa_plan_set_device", "tfpa_plan_dyn_bytes",
           "tfpa_plan_dyn_pack", "tfpa_plan_shape", "tfpa_plan_capture", "tfpa_plan_replay",
           "tfpa_decode_append", "tfpa_plan_decode_append", "tfpa_row_splits")


class TfpaError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {code} ({strerror(code)})")


class tfpa_seg(ctypes.Structure):
    _fields_ = [("seq_len", ctypes.c_int32), ("page_table", ctypes.c_void_p),
                ("page_table_host", ctypes.c_void_p), ("k_slab", ctypes.c_void_p),
                ("v_slab", ctypes.c_void_p), ("slab_cap", ctypes.c_int32)]


class tfpa_cache(ctypes.Structure):
    _fields_ = [("dtype", ctypes.c_int), ("hq", ctypes.c_int32), ("hkv", ctypes.c_int32),
                ("head_dim", ctypes.c_int32), ("k_pool", ctypes.c_void_p),
                ("v_pool", ctypes.c_void_p), ("num_pages", ctypes.c_int32),
                ("k_scale", ctypes.c_void_p), ("v_scale", ctypes.c_void_p),
                ("err_flag", ctypes.c_void_p)]


class tfpa_scratch(ctypes.Structure):
    _fields_ = [("part_o", ctypes.c_void_p), ("part_ml", ctypes.c_void_p),
                ("cap_rows", ctypes.c_int32), ("max_splits", ctypes.c_int32),
                ("arrive", ctypes.c_void_p)]


class tfpa_copy(ctypes.Structure):
    _fields_ = [("dst", ctypes.c_void_p), ("src", ctypes.c_void_p), ("bytes", ctypes.c_size_t)]


class tfpa_launch_record(ctypes.Structure):
    _fields_ = [("kind", ctypes.c_int32), ("row0", ctypes.c_int32), ("rows", ctypes.c_int32),
                ("runs", ctypes.c_int32), ("items", ctypes.c_int32), ("grid", ctypes.c_int32),
                ("q_offset", ctypes.c_int64), ("out_offset", ctypes.c_int64)]


HOOK = ctypes.CFUNCTYPE(None, ctypes.POINTER(tfpa_launch_record), ctypes.c_void_p)
KINDS = {0: "write_kv", 1: "partial", 2: "merge", 3: "prefill", 4: "keep", 5: "stage",
         6: "save", 7: "restore", 8: "verify"}

_lib = None


def lib():
    """The loaded library (built by ``__graft_entry__.build()``)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"{LIB_PATH} is missing: build it first "
                               "(python -c 'import __graft_entry__ as g; g.build()')")
        L = ctypes.CDLL(LIB_PATH)
        i32, vp, P = ctypes.c_int32, ctypes.c_void_p, ctypes.POINTER
        L.tfpa_pages_per_split.argtypes = [i32]
        L.tfpa_pages_per_split.restype = i32
        L.tfpa_num_splits.argtypes = [i32]
        L.tfpa_num_splits.restype = i32
        L.tfpa_write_kv.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, vp, i32, vp]
        L.tfpa_write_kv.restype = ctypes.c_int
        L.tfpa_decode_partial.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, i32,
                                          ctypes.c_float, P(tfpa_scratch), vp]
        L.tfpa_decode_partial.restype = ctypes.c_int
        L.tfpa_merge.argtypes = [P(tfpa_scratch), i32, i32, vp, vp, vp, vp]
        L.tfpa_merge.restype = ctypes.c_int
        L.tfpa_row_splits.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, i32, vp]
        L.tfpa_row_splits.restype = ctypes.c_int
        L.tfpa_decode.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, i32,
                                  ctypes.c_float, P(tfpa_scratch), vp, vp, vp]
        L.tfpa_decode.restype = ctypes.c_int
        L.tfpa_write_kv_rope.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, vp, vp,
                                         vp, vp, i32, i32, vp]
        L.tfpa_write_kv_rope.restype = ctypes.c_int
        L.tfpa_keep_kv.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, i32, vp]
        L.tfpa_keep_kv.restype = ctypes.c_int
        L.tfpa_pool_create.argtypes = [i32]
        L.tfpa_pool_create.restype = vp
        L.tfpa_pool_destroy.argtypes = [vp]
        L.tfpa_pool_destroy.restype = None
        L.tfpa_pool_free.argtypes = [vp]
        L.tfpa_pool_free.restype = i32
        L.tfpa_pool_fits.argtypes = [vp, i32]
        L.tfpa_pool_fits.restype = ctypes.c_int
        L.tfpa_pool_claim.argtypes = [vp, i32, vp]
        L.tfpa_pool_claim.restype = ctypes.c_int
        L.tfpa_pool_release.argtypes = [vp, vp, i32]
        L.tfpa_pool_release.restype = ctypes.c_int
        L.tfpa_stage_pages.argtypes = [vp, i32, vp, i32, vp]
        L.tfpa_stage_pages.restype = ctypes.c_int
        L.tfpa_save_kv.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, i32, vp, vp]
        L.tfpa_save_kv.restype = ctypes.c_int
        L.tfpa_restore_kv.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, i32, vp, vp]
        L.tfpa_restore_kv.restype = ctypes.c_int
        L.tfpa_decode_tree.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, vp, i32,
                                       ctypes.c_float, P(tfpa_scratch), vp, vp, vp]
        L.tfpa_decode_tree.restype = ctypes.c_int
        L.tfpa_decode_static.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, i32,
                                         ctypes.c_float, vp, vp, vp]
        L.tfpa_decode_static.restype = ctypes.c_int
        L.tfpa_prefill.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, i32,
                                   ctypes.c_float, i32, vp, vp, vp]
        L.tfpa_prefill.restype = ctypes.c_int
        L.tfpa_plan_create.argtypes = []
        L.tfpa_plan_create.restype = vp
        L.tfpa_plan_destroy.argtypes = [vp]
        L.tfpa_plan_destroy.restype = None
        L.tfpa_plan_clear.argtypes = [vp]
        L.tfpa_plan_clear.restype = None
        L.tfpa_plan_launches.argtypes = [vp]
        L.tfpa_plan_launches.restype = i32
        L.tfpa_plan_write_kv.argtypes = [vp, P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, vp, i32]
        L.tfpa_plan_write_kv.restype = ctypes.c_int
        L.tfpa_plan_decode.argtypes = [vp, P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, i32,
                                       ctypes.c_float, P(tfpa_scratch), vp, vp]
        L.tfpa_plan_decode.restype = ctypes.c_int
        L.tfpa_plan_launch.argtypes = [vp, vp]
        L.tfpa_plan_launch.restype = ctypes.c_int
        L.tfpa_plan_set_device.argtypes = [vp, vp, ctypes.c_size_t]
        L.tfpa_plan_set_device.restype = ctypes.c_int
        L.tfpa_plan_dyn_bytes.argtypes = [vp]
        L.tfpa_plan_dyn_bytes.restype = ctypes.c_size_t
        L.tfpa_plan_dyn_pack.argtypes = [vp, vp, ctypes.c_size_t]
        L.tfpa_plan_dyn_pack.restype = ctypes.c_int
        L.tfpa_plan_shape.argtypes = [vp]
        L.tfpa_plan_shape.restype = ctypes.c_uint64
        L.tfpa_decode_append.argtypes = [P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, vp, vp, i32,
                                         ctypes.c_float, P(tfpa_scratch), vp, vp, vp]
        L.tfpa_decode_append.restype = ctypes.c_int
        L.tfpa_plan_decode_append.argtypes = [vp, P(tfpa_cache), P(tfpa_seg), i32, vp, vp, vp, vp,
                                              vp, i32, ctypes.c_float, P(tfpa_scratch), vp, vp]
        L.tfpa_plan_decode_append.restype = ctypes.c_int
        L.tfpa_plan_capture.argtypes = [vp, P(tfpa_copy), i32, P(tfpa_copy), i32, vp]
        L.tfpa_plan_capture.restype = ctypes.c_int
        L.tfpa_plan_replay.argtypes = [vp, vp]
        L.tfpa_plan_replay.restype = ctypes.c_int
        L.tfpa_set_launch_hook.argtypes = [HOOK, vp, ctypes.c_int]
        L.tfpa_set_launch_hook.restype = None
        L.tfpa_strerror.argtypes = [ctypes.c_int]
        L.tfpa_strerror.restype = ctypes.c_char_p
        L.tfpa_version.argtypes = []
        L.tfpa_version.restype = ctypes.c_char_p
        _lib = L
    return _lib


def strerror(code: int) -> str:
    return lib().tfpa_strerror(code).decode()


def _check(code: int, where: str):
    if code != TFPA_OK:
        raise TfpaError(code, where)


def _ptr(x) -> Optional[int]:
    """Device (or host) address of a tensor/array, or an int passed through."""
    if x is None:
        return None
    t = type(x)
    if t is int:
        return x
    if t is np.ndarray:
        return x.ctypes.data
    if isinstance(x, int):
        return int(x)
    return x.data_ptr()


def _stream(stream) -> Optional[int]:
    """A ``cudaStream_t`` handle: an int passes through (the cheapest form in a
    loop), a torch stream gives its handle, None the current torch stream."""
    if stream is not None:
        return stream if type(stream) is int else stream.cuda_stream
    import torch
    if torch.cuda.is_available():
        return torch.cuda.current_stream().cuda_stream
    return None


def _i32(a) -> np.ndarray:
    if type(a) is np.ndarray and a.dtype == np.int32 and a.flags.c_contiguous:
        return a
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


class _Cached:
    """Keeps the C struct of a dataclass until one of its fields is assigned."""

    def __setattr__(self, k, v):
        object.__setattr__(self, k, v)
        if k != "_cs":
            object.__setattr__(self, "_cs", None)

    def c(self):
        cs = self.__dict__.get("_cs")
        if cs is None:
            cs = self._make_c()
            object.__setattr__(self, "_cs", cs)
        return cs


@dataclass(eq=False)
class Cache(_Cached):
    """One layer's KV cache; holds the tensors so their memory stays alive."""
    dtype: str                    # "bf16" or "fp8"
    hq: int
    hkv: int
    k_pool: object = None         # [num_pages][hkv][256][128] bf16 (or int16) / uint8
    v_pool: object = None
    k_scale: object = None        # float32 [hkv] (fp8)
    v_scale: object = None
    err_flag: object = None       # int32 [1]
    num_pages: int = 0

    def _make_c(self) -> tfpa_cache:
        return tfpa_cache(BF16 if self.dtype == "bf16" else FP8_E4M3, self.hq, self.hkv,
                          HEAD_DIM, _ptr(self.k_pool), _ptr(self.v_pool), self.num_pages,
                          _ptr(self.k_scale), _ptr(self.v_scale), _ptr(self.err_flag))


@dataclass(eq=False)
class Seg(_Cached):
    """One stream: a device page table or a pair of slabs."""
    seq_len: int
    page_table: object = None         # device int32 [>= ceil(seq_len/256)]
    page_table_host: object = None    # optional host int32 mirror (validated)
    k_slab: object = None             # [hkv][slab_cap][128]
    v_slab: object = None
    slab_cap: int = 0

    def _make_c(self) -> tfpa_seg:
        host = None
        if self.page_table_host is not None:
            object.__setattr__(self, "page_table_host", _i32(self.page_table_host))
            host = _ptr(self.page_table_host)
        return tfpa_seg(int(self.seq_len), _ptr(self.page_table), host, _ptr(self.k_slab),
                        _ptr(self.v_slab), int(self.slab_cap))


@dataclass(eq=False)
class Scratch(_Cached):
    part_o: object
    part_ml: object
    cap_rows: int
    max_splits: int = MAX_SPLITS
    arrive: object = None             # uint32 [cap_rows][hq] zeros: merge in the partial kernel

    def _make_c(self) -> tfpa_scratch:
        return tfpa_scratch(_ptr(self.part_o), _ptr(self.part_ml), self.cap_rows, self.max_splits,
                            _ptr(self.arrive))


def make_scratch(cap_rows: int, hq: int, max_splits: int = MAX_SPLITS, device="cuda",
                 fused_merge: bool = True) -> Scratch:
    """Scratch for cap_rows rows; with fused_merge (the default) it carries
    the zeroed arrival counters that let tfpa_decode merge streams of up to
    four splits inside the partial kernel (one launch instead of two)."""
    import torch
    o = torch.empty(cap_rows * hq * max_splits * HEAD_DIM, dtype=torch.float32, device=device)
    ml = torch.empty(cap_rows * hq * max_splits * 2, dtype=torch.float32, device=device)
    arrive = torch.zeros(cap_rows * hq, dtype=torch.int32, device=device) if fused_merge else None
    return Scratch(o, ml, cap_rows, max_splits, arrive)


class SegTable:
    """The call's segments as one C array, built once.  A decode loop moves
    each stream's length forward in place (``set_seq_len``) instead of
    rebuilding the table for every call; every entry point that takes
    ``segs`` accepts a SegTable.  The Seg objects (and their tensors) stay
    referenced for as long as the table lives."""

    def __init__(self, segs: Sequence[Seg]):
        self.segs = list(segs)
        self.n = len(self.segs)
        self.arr = (tfpa_seg * max(1, self.n))(*[s.c() for s in self.segs])

    def __len__(self):
        return self.n

    def __getitem__(self, i):
        return self.segs[i]

    def set_seq_len(self, i: int, seq_len: int) -> None:
        """Stream i now holds seq_len keys (its page table, and the host mirror
        if one was given, must cover ceil(seq_len / 256) pages)."""
        self.arr[i].seq_len = seq_len
        seg = self.segs[i]
        object.__setattr__(seg, "seq_len", seq_len)
        cs = seg.__dict__.get("_cs")
        if cs is not None:
            cs.seq_len = seq_len


def _segs(segs):
    if type(segs) is SegTable:
        return segs.arr, segs.n
    arr = (tfpa_seg * max(1, len(segs)))(*[s.c() for s in segs])
    return arr, len(segs)


def tfpa_pages_per_split(seq_len: int) -> int:
    return lib().tfpa_pages_per_split(int(seq_len))


def tfpa_num_splits(seq_len: int) -> int:
    return lib().tfpa_num_splits(int(seq_len))


def tfpa_write_kv(cache: Cache, segs: Sequence[Seg], k_rows, v_rows, row_seg, row_pos,
                  stream=None) -> None:
    cs, n = _segs(segs)
    rs, rp = _i32(row_seg), _i32(row_pos)
    cc = cache.c()
    _check(lib().tfpa_write_kv(ctypes.byref(cc), cs, n, _ptr(k_rows), _ptr(v_rows), _ptr(rs),
                               _ptr(rp), len(rs), _stream(stream)), "tfpa_write_kv")


def tfpa_decode_partial(cache: Cache, segs: Sequence[Seg], q, row_seg, row_pos, softmax_scale,
                        scratch: Scratch, stream=None) -> None:
    cs, n = _segs(segs)
    rs, rp = _i32(row_seg), _i32(row_pos)
    cc, sc = cache.c(), scratch.c()
    _check(lib().tfpa_decode_partial(ctypes.byref(cc), cs, n, _ptr(q), _ptr(rs), _ptr(rp),
                                     len(rs), float(softmax_scale), ctypes.byref(sc),
                                     _stream(stream)), "tfpa_decode_partial")


def tfpa_row_splits(cache: Cache, segs: Sequence[Seg], row_seg, row_pos) -> np.ndarray:
    """Each row's split count as tfpa_decode_partial leaves it (for tfpa_merge)."""
    cs, n = _segs(segs)
    rs, rp = _i32(row_seg), _i32(row_pos)
    cc = cache.c()
    ns = np.zeros(len(rs), np.int32)
    _check(lib().tfpa_row_splits(ctypes.byref(cc), cs, n, _ptr(rs), _ptr(rp), len(rs), _ptr(ns)),
           "tfpa_row_splits")
    return ns


def tfpa_merge(scratch: Scratch, hq: int, nsplit, out, lse=None, stream=None) -> None:
    ns = _i32(nsplit)
    sc = scratch.c()
    _check(lib().tfpa_merge(ctypes.byref(sc), int(hq), len(ns), _ptr(ns), _ptr(out), _ptr(lse),
                            _stream(stream)), "tfpa_merge")


def tfpa_decode(cache: Cache, segs: Sequence[Seg], q, row_seg, row_pos, softmax_scale,
                scratch: Scratch, out, lse=None, stream=None) -> None:
    cs, n = _segs(segs)
    rs, rp = _i32(row_seg), _i32(row_pos)
    cc, sc = cache.c(), scratch.c()
    _check(lib().tfpa_decode(ctypes.byref(cc), cs, n, _ptr(q), _ptr(rs), _ptr(rp), len(rs),
                             float(softmax_scale), ctypes.byref(sc), _ptr(out), _ptr(lse),
                             _stream(stream)), "tfpa_decode")


def tfpa_decode_append(cache: Cache, segs: Sequence[Seg], k_rows, v_rows, q, row_seg, row_pos,
                       softmax_scale, scratch: Scratch, out, lse=None, stream=None) -> None:
    """Store the rows' K / V and decode the rows in one call (a decode step)."""
    cs, n = _segs(segs)
    rs, rp = _i32(row_seg), _i32(row_pos)
    cc, sc = cache.c(), scratch.c()
    _check(lib().tfpa_decode_append(ctypes.byref(cc), cs, n, _ptr(k_rows), _ptr(v_rows), _ptr(q),
                                    _ptr(rs), _ptr(rp), len(rs), float(softmax_scale),
                                    ctypes.byref(sc), _ptr(out), _ptr(lse), _stream(stream)),
           "tfpa_decode_append")


def tfpa_write_kv_rope(cache: Cache, segs: Sequence[Seg], k_rows, v_rows, row_seg, row_pos,
                       rope_cos, rope_sin, rope_pos=None, stream=None) -> None:
    """KV write with K rotated by each row's rotary position: ``rope_cos`` /
    ``rope_sin`` are device float32 ``[n][64]`` tables; ``rope_pos`` a device
    int32 tensor (one per row) or None for the storage positions."""
    cs, n = _segs(segs)
    rs, rp = _i32(row_seg), _i32(row_pos)
    cc = cache.c()
    _check(lib().tfpa_write_kv_rope(ctypes.byref(cc), cs, n, _ptr(k_rows), _ptr(v_rows),
                                    _ptr(rs), _ptr(rp), _ptr(rope_pos), _ptr(rope_cos),
                                    _ptr(rope_sin), int(rope_cos.shape[0]), len(rs),
                                    _stream(stream)), "tfpa_write_kv_rope")


def tfpa_keep_kv(cache: Cache, segs: Sequence[Seg], keep_seg, keep_src, keep_dst,
                 stream=None) -> None:
    """Copy stored K/V rows from keep_src to keep_dst positions (host tables)."""
    cs, n = _segs(segs)
    a, b, d = _i32(keep_seg), _i32(keep_src), _i32(keep_dst)
    if not (len(a) == len(b) == len(d)):
        raise ValueError("keep tables differ in length")
    cc = cache.c()
    _check(lib().tfpa_keep_kv(ctypes.byref(cc), cs, n, _ptr(a), _ptr(b), _ptr(d), len(a),
                              _stream(stream)), "tfpa_keep_kv")


class Pool:
    """The page pool's admission ledger (host only): claims are up front and
    all or nothing; ``claim`` raises TfpaError(TFPA_ELANEMEM) while the pool
    cannot hold the request and TfpaError(TFPA_ECAPACITY) if it never could."""

    def __init__(self, num_pages: int):
        self._p = lib().tfpa_pool_create(int(num_pages))
        if not self._p:
            raise TfpaError(TFPA_EINVAL, "tfpa_pool_create")
        self.num_pages = int(num_pages)

    def free(self) -> int:
        return int(lib().tfpa_pool_free(self._p))

    def fits(self, npages: int) -> bool:
        return bool(lib().tfpa_pool_fits(self._p, int(npages)))

    def claim(self, npages: int) -> np.ndarray:
        out = np.zeros(max(1, int(npages)), np.int32)
        _check(lib().tfpa_pool_claim(self._p, int(npages), out.ctypes.data), "tfpa_pool_claim")
        return out[: int(npages)]

    def release(self, pages) -> None:
        a = _i32(pages)
        _check(lib().tfpa_pool_release(self._p, _ptr(a), len(a)), "tfpa_pool_release")

    def __del__(self):
        if getattr(self, "_p", None):
            lib().tfpa_pool_destroy(self._p)
            self._p = None


def tfpa_stage_pages(page_table, first: int, pages, stream=None) -> None:
    """Write page ids into a device page table at [first, first + len) on the stream."""
    a = _i32(pages)
    _check(lib().tfpa_stage_pages(_ptr(page_table), int(first), _ptr(a), len(a),
                                  _stream(stream)), "tfpa_stage_pages")


def tfpa_save_kv(cache: Cache, seg: Seg, p0: int, p1: int, image, stream=None) -> None:
    """Stored rows [p0, p1) of one stream into ``image`` ([K, V][hkv][p1-p0][128])."""
    cs, _ = _segs([seg])
    cc = cache.c()
    _check(lib().tfpa_save_kv(ctypes.byref(cc), cs, int(p0), int(p1), _ptr(image),
                              _stream(stream)), "tfpa_save_kv")


def tfpa_restore_kv(cache: Cache, seg: Seg, p0: int, p1: int, image, stream=None) -> None:
    """The reverse of tfpa_save_kv: ``image`` back into rows [p0, p1) of the stream."""
    cs, _ = _segs([seg])
    cc = cache.c()
    _check(lib().tfpa_restore_kv(ctypes.byref(cc), cs, int(p0), int(p1), _ptr(image),
                                 _stream(stream)), "tfpa_restore_kv")


def tfpa_decode_tree(cache: Cache, segs: Sequence[Seg], q, row_seg, row_pos, row_anc,
                     softmax_scale, scratch: Scratch, out, lse=None, stream=None) -> None:
    """Draft-tree verify: ``row_anc`` is a device tensor of 64-bit ancestor
    masks, one per row (int64 or uint64 storage; only the bits matter)."""
    cs, n = _segs(segs)
    rs, rp = _i32(row_seg), _i32(row_pos)
    cc, sc = cache.c(), scratch.c()
    _check(lib().tfpa_decode_tree(ctypes.byref(cc), cs, n, _ptr(q), _ptr(rs), _ptr(rp),
                                  _ptr(row_anc), len(rs), float(softmax_scale),
                                  ctypes.byref(sc), _ptr(out), _ptr(lse), _stream(stream)),
           "tfpa_decode_tree")


def tfpa_decode_static(cache: Cache, segs: Sequence[Seg], q, row_seg, row_pos, softmax_scale,
                       out, lse=None, stream=None) -> None:
    """Decode without caller scratch: the partials live in an array compiled
    into the library, for callers that cannot allocate device memory."""
    cs, n = _segs(segs)
    rs, rp = _i32(row_seg), _i32(row_pos)
    cc = cache.c()
    _check(lib().tfpa_decode_static(ctypes.byref(cc), cs, n, _ptr(q), _ptr(rs), _ptr(rp),
                                    len(rs), float(softmax_scale), _ptr(out), _ptr(lse),
                                    _stream(stream)), "tfpa_decode_static")


def tfpa_prefill(cache: Cache, segs: Sequence[Seg], q, row_seg, row_pos, softmax_scale, out,
                 lse=None, max_rows_per_launch: int = 0, stream=None) -> None:
    cs, n = _segs(segs)
    rs, rp = _i32(row_seg), _i32(row_pos)
    cc = cache.c()
    _check(lib().tfpa_prefill(ctypes.byref(cc), cs, n, _ptr(q), _ptr(rs), _ptr(rp), len(rs),
                              float(softmax_scale), int(max_rows_per_launch), _ptr(out),
                              _ptr(lse), _stream(stream)), "tfpa_prefill")


class Plan:
    """Launches planned ahead (tfpa_plan_*): ``write_kv`` and ``decode`` take
    the arguments of tfpa_write_kv / tfpa_decode without a stream and do all
    of the call's host work; ``launch`` enqueues the planned launches."""

    def __init__(self):
        self._p = lib().tfpa_plan_create()
        if not self._p:
            raise MemoryError("tfpa_plan_create")

    def clear(self) -> None:
        lib().tfpa_plan_clear(self._p)

    def __len__(self) -> int:
        return int(lib().tfpa_plan_launches(self._p))

    def write_kv(self, cache: Cache, segs, k_rows, v_rows, row_seg, row_pos) -> None:
        cs, n = _segs(segs)
        rs, rp = _i32(row_seg), _i32(row_pos)
        _check(lib().tfpa_plan_write_kv(self._p, ctypes.byref(cache.c()), cs, n, _ptr(k_rows),
                                        _ptr(v_rows), _ptr(rs), _ptr(rp), len(rs)),
               "tfpa_plan_write_kv")

    def decode(self, cache: Cache, segs, q, row_seg, row_pos, softmax_scale, scratch: Scratch,
               out, lse=None) -> None:
        cs, n = _segs(segs)
        rs, rp = _i32(row_seg), _i32(row_pos)
        _check(lib().tfpa_plan_decode(self._p, ctypes.byref(cache.c()), cs, n, _ptr(q), _ptr(rs),
                                      _ptr(rp), len(rs), float(softmax_scale),
                                      ctypes.byref(scratch.c()), _ptr(out), _ptr(lse)),
               "tfpa_plan_decode")

    def decode_append(self, cache: Cache, segs, k_rows, v_rows, q, row_seg, row_pos,
                      softmax_scale, scratch: Scratch, out, lse=None) -> None:
        cs, n = _segs(segs)
        rs, rp = _i32(row_seg), _i32(row_pos)
        _check(lib().tfpa_plan_decode_append(self._p, ctypes.byref(cache.c()), cs, n,
                                             _ptr(k_rows), _ptr(v_rows), _ptr(q), _ptr(rs),
                                             _ptr(rp), len(rs), float(softmax_scale),
                                             ctypes.byref(scratch.c()), _ptr(out), _ptr(lse)),
               "tfpa_plan_decode_append")

    def launch(self, stream=None) -> None:
        _check(lib().tfpa_plan_launch(self._p, _stream(stream)), "tfpa_plan_launch")

    def set_device(self, dyn) -> None:
        """Device mode (tfpa_plan_set_device): ``dyn`` is a device tensor
        (kept alive by the plan) whose bytes hold the launches' dynamic
        data, or None for parameter mode."""
        nbytes = 0 if dyn is None else dyn.numel() * dyn.element_size()
        _check(lib().tfpa_plan_set_device(self._p, _ptr(dyn), nbytes), "tfpa_plan_set_device")
        self._dyn = dyn

    def dyn_bytes(self) -> int:
        return int(lib().tfpa_plan_dyn_bytes(self._p))

    def pack(self, host) -> None:
        """Writes the planned launches' dynamic data into the host tensor
        ``host`` (tfpa_plan_dyn_pack), for a copy to the device buffer."""
        _check(lib().tfpa_plan_dyn_pack(self._p, ctypes.c_void_p(host.data_ptr()),
                                        host.numel() * host.element_size()),
               "tfpa_plan_dyn_pack")

    def shape(self) -> int:
        return int(lib().tfpa_plan_shape(self._p))

    def capture(self, before=(), after=(), stream=None) -> None:
        """tfpa_plan_capture: `before` / `after` are (dst, src, nbytes)
        copies (tensors or addresses) around the plan's launches, captured
        with them as one CUDA graph on `stream` (a created stream)."""
        def arr(copies):
            a = (tfpa_copy * max(1, len(copies)))()
            for i, (dst, src, n) in enumerate(copies):
                a[i] = tfpa_copy(_ptr(dst), _ptr(src), int(n))
            return a
        b, a = arr(before), arr(after)
        _check(lib().tfpa_plan_capture(self._p, b, len(before), a, len(after), _stream(stream)),
               "tfpa_plan_capture")

    def replay(self, stream=None) -> None:
        _check(lib().tfpa_plan_replay(self._p, _stream(stream)), "tfpa_plan_replay")

    def __del__(self):
        if getattr(self, "_p", None):
            lib().tfpa_plan_destroy(self._p)
            self._p = None


@contextlib.contextmanager
def record_launches(dry_run: bool = True):
    """Collects the library's launches as dicts; with dry_run nothing runs."""
    records: List[dict] = []

    def _cb(rec, _user):
        r = rec.contents
        records.append(dict(kind=KINDS[r.kind], row0=r.row0, rows=r.rows, runs=r.runs,
                            items=r.items, grid=r.grid, q_offset=r.q_offset,
                            out_offset=r.out_offset))

    cb = HOOK(_cb)
    lib().tfpa_set_launch_hook(cb, None, 1 if dry_run else 0)
    try:
        yield records
    finally:
        lib().tfpa_set_launch_hook(HOOK(), None, 0)
