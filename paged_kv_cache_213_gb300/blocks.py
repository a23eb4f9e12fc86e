"""ctypes binding of the block manager and the copy-on-write block copy
(``include/pagedkv_blocks.h``).  Marshalling only; the logic is in the C++
library."""
from __future__ import annotations

import ctypes

import torch

from .binding import PagedKVError, _need, _ptr, _stream_handle, library

PKV_ERR_OUT_OF_BLOCKS = -6


class OutOfBlocks(PagedKVError):
    pass


_bound = False


def _lib():
    global _bound
    lib = library()
    if not _bound:
        c = ctypes
        p = c.c_void_p
        lib.pkv_bm_create.argtypes = [c.c_int64, c.c_int]
        lib.pkv_bm_create.restype = p
        lib.pkv_bm_destroy.argtypes = [p]
        lib.pkv_bm_destroy.restype = None
        lib.pkv_bm_add_sequence.argtypes = [p, c.c_int64]
        lib.pkv_bm_add_sequence.restype = c.c_int
        lib.pkv_bm_fork.argtypes = [p, c.c_int64, c.c_int64]
        lib.pkv_bm_fork.restype = c.c_int
        lib.pkv_bm_append_slot.argtypes = [p, c.c_int64, c.POINTER(c.c_int64),
                                           c.POINTER(c.c_int32), c.POINTER(c.c_int32),
                                           c.POINTER(c.c_int32)]
        lib.pkv_bm_append_slot.restype = c.c_int
        lib.pkv_bm_free_sequence.argtypes = [p, c.c_int64]
        lib.pkv_bm_free_sequence.restype = c.c_int
        lib.pkv_bm_num_free_blocks.argtypes = [p]
        lib.pkv_bm_num_free_blocks.restype = c.c_int64
        lib.pkv_bm_sequence_length.argtypes = [p, c.c_int64, c.POINTER(c.c_int64)]
        lib.pkv_bm_sequence_length.restype = c.c_int
        lib.pkv_bm_block_table.argtypes = [p, c.c_int64, p, c.c_int64, c.POINTER(c.c_int64)]
        lib.pkv_bm_block_table.restype = c.c_int
        lib.pkv_bm_block_info.argtypes = [p, c.c_int32, c.POINTER(c.c_int32),
                                          c.POINTER(c.c_int32)]
        lib.pkv_bm_block_info.restype = c.c_int
        lib.pkv_bm_prefix_groups.argtypes = [p, p, c.c_int, p, p, c.POINTER(c.c_int),
                                             c.POINTER(c.c_int), c.POINTER(c.c_int)]
        lib.pkv_bm_prefix_groups.restype = c.c_int
        lib.paged_kv_copy_blocks.argtypes = [p, p, p, p, p, c.c_int, c.c_int, c.c_int, c.c_int,
                                             c.c_int64, p, p]
        lib.paged_kv_copy_blocks.restype = c.c_int
        _bound = True
    return lib


def _check(func, rc):
    if rc == PKV_ERR_OUT_OF_BLOCKS:
        raise OutOfBlocks(func, rc)
    if rc != 0:
        raise PagedKVError(func, rc)


class BlockManager:
    """Pool of physical KV blocks with per-sequence block tables, fork and
    copy-on-write (the library's C++ manager)."""

    def __init__(self, num_blocks: int, block_size: int):
        self._lib = _lib()
        self._h = self._lib.pkv_bm_create(num_blocks, block_size)
        if not self._h:
            raise ValueError("bad pool size")
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            self._lib.pkv_bm_destroy(h)
            self._h = None

    def add_sequence(self, seq: int):
        _check("pkv_bm_add_sequence", self._lib.pkv_bm_add_sequence(self._h, seq))

    def fork(self, parent: int, child: int):
        _check("pkv_bm_fork", self._lib.pkv_bm_fork(self._h, parent, child))

    def append_slot(self, seq: int):
        """(slot, copy): copy is (src, dst, rows) for a copy-on-write, else None."""
        slot = ctypes.c_int64()
        src, dst, rows = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        _check("pkv_bm_append_slot",
               self._lib.pkv_bm_append_slot(self._h, seq, ctypes.byref(slot), ctypes.byref(src),
                                            ctypes.byref(dst), ctypes.byref(rows)))
        copy = None if src.value < 0 else (src.value, dst.value, rows.value)
        return slot.value, copy

    def free_sequence(self, seq: int):
        _check("pkv_bm_free_sequence", self._lib.pkv_bm_free_sequence(self._h, seq))

    def num_free(self) -> int:
        return int(self._lib.pkv_bm_num_free_blocks(self._h))

    def length(self, seq: int) -> int:
        n = ctypes.c_int64()
        _check("pkv_bm_sequence_length", self._lib.pkv_bm_sequence_length(self._h, seq,
                                                                          ctypes.byref(n)))
        return n.value

    def block_table(self, seq: int) -> list[int]:
        n = ctypes.c_int64()
        _check("pkv_bm_block_table", self._lib.pkv_bm_block_table(self._h, seq, None, 0,
                                                                  ctypes.byref(n)))
        buf = (ctypes.c_int32 * max(1, n.value))()
        _check("pkv_bm_block_table", self._lib.pkv_bm_block_table(self._h, seq, buf, n.value,
                                                                  ctypes.byref(n)))
        return list(buf[: n.value])

    def prefix_groups(self, seq_ids):
        """Groups of consecutive batch rows sharing leading blocks, for
        paged_decode_attention_prefix_shared: (offsets int32 [G+1], prefix
        tokens int32 [G], largest group, longest prefix) as numpy arrays and
        ints."""
        import numpy as np
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        n = int(ids.size)
        offs = np.zeros(n + 1, dtype=np.int32)
        pref = np.zeros(max(n, 1), dtype=np.int32)
        g, most, longest = ctypes.c_int(), ctypes.c_int(), ctypes.c_int()
        _check("pkv_bm_prefix_groups",
               self._lib.pkv_bm_prefix_groups(self._h, ids.ctypes.data_as(ctypes.c_void_p), n,
                                              offs.ctypes.data_as(ctypes.c_void_p),
                                              pref.ctypes.data_as(ctypes.c_void_p),
                                              ctypes.byref(g), ctypes.byref(most),
                                              ctypes.byref(longest)))
        return offs[: g.value + 1].copy(), pref[: g.value].copy(), most.value, longest.value

    def block_info(self, block: int):
        """(refcount, filled rows) of a physical block."""
        r, t = ctypes.c_int32(), ctypes.c_int32()
        _check("pkv_bm_block_info", self._lib.pkv_bm_block_info(self._h, block, ctypes.byref(r),
                                                                ctypes.byref(t)))
        return r.value, t.value


def paged_kv_copy_blocks(k_cache, v_cache, src, dst, tokens=None, err_word=None):
    """Copy rows [0, tokens[i]) (all rows if None) of block src[i] to dst[i],
    all KV heads, in both caches, on the current stream."""
    dev = k_cache.device
    _need(k_cache, "k_cache", torch.float16, dev)
    _need(v_cache, "v_cache", torch.float16, dev)
    _need(src, "src", torch.int32, dev)
    _need(dst, "dst", torch.int32, dev)
    if tokens is not None:
        _need(tokens, "tokens", torch.int32, dev)
    if err_word is not None:
        _need(err_word, "err_word", torch.int32, dev)
    NB, Hk, bs, d = k_cache.shape
    n = src.numel()
    if dst.numel() != n or (tokens is not None and tokens.numel() != n):
        raise ValueError("src, dst, tokens must have the same length")
    with torch.cuda.device(dev):
        rc = _lib().paged_kv_copy_blocks(_ptr(k_cache), _ptr(v_cache), _ptr(src), _ptr(dst),
                                         _ptr(tokens), n, Hk, d, bs, NB, _ptr(err_word),
                                         _stream_handle(dev))
    _check("paged_kv_copy_blocks", rc)
