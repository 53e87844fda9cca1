"""Python handle on the library's host block allocator (pa_alloc_* in the C ABI).

Block pool with a free stack, reference counts, fork and copy-on-write, as the
"PagedAttention实现" page's PagedKVManager describes, producing the block tables
and slot mappings the kernels consume. Host memory only; no GPU needed.
"""
from __future__ import annotations

import ctypes
from dataclasses import dataclass

import numpy as np

from . import PA_OK, PagedAttnError, _decl, lib

_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64


class _Stats(ctypes.Structure):
    _fields_ = [("num_blocks", _i64), ("num_free", _i64), ("num_used", _i64), ("peak_used", _i64),
                ("num_cow_copies", _i64), ("num_seqs", _i64)]


_decl("pa_alloc_create", [_i64, _i32, ctypes.POINTER(_vp)])
_decl("pa_alloc_destroy", [_vp], None)
_decl("pa_alloc_add_seq", [_vp, _i64])
_decl("pa_alloc_fork", [_vp, _i64, _i64])
_decl("pa_alloc_append", [_vp, _i64, _i64, _vp, _vp, _i64, ctypes.POINTER(_i64)])
_decl("pa_alloc_free_seq", [_vp, _i64])
_decl("pa_alloc_block_table", [_vp, _i64, _vp, _i64, ctypes.POINTER(_i64)])
_decl("pa_alloc_seq_len", [_vp, _i64, ctypes.POINTER(_i64)])
_decl("pa_alloc_export", [_vp, _vp, _i64, _vp, _i32, _vp])
_decl("pa_alloc_block", [_vp, ctypes.POINTER(ctypes.c_int32)])
_decl("pa_alloc_decref", [_vp, ctypes.c_int32])
_decl("pa_alloc_refcount", [_vp, ctypes.c_int32, ctypes.POINTER(ctypes.c_int32)])
_decl("pa_alloc_get_stats", [_vp, ctypes.POINTER(_Stats)])
_decl("pa_alloc_snapshot", [_vp, _vp, _i64, ctypes.POINTER(_i64)])
_decl("pa_alloc_restore", [_vp, _i64, ctypes.POINTER(_vp)])


@dataclass
class AllocStats:
    num_blocks: int
    num_free: int
    num_used: int
    peak_used: int
    num_cow_copies: int
    num_seqs: int


def _ok(rc, what):
    if rc != PA_OK:
        raise PagedAttnError(rc, what)


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int):
        self._L = lib()
        h = _vp()
        _ok(self._L.pa_alloc_create(num_blocks, block_size, ctypes.byref(h)), "pa_alloc_create")
        self._h = h
        self.num_blocks = num_blocks
        self.block_size = block_size

    def __del__(self):
        h = getattr(self, "_h", None)
        if h is not None and h.value:
            self._L.pa_alloc_destroy(h)
            self._h = None

    def add_seq(self, seq_id: int) -> None:
        _ok(self._L.pa_alloc_add_seq(self._h, seq_id), "pa_alloc_add_seq")

    def fork(self, parent: int, child: int) -> None:
        _ok(self._L.pa_alloc_fork(self._h, parent, child), "pa_alloc_fork")

    def append(self, seq_id: int, n_tokens: int):
        """Returns (slots int32 [n_tokens], cow_pairs int32 [n_cow, 2])."""
        slots = np.empty(max(n_tokens, 1), np.int32)
        pairs = np.empty((1, 2), np.int32)   # an append copies at most one block
        n = _i64(0)
        _ok(self._L.pa_alloc_append(self._h, seq_id, n_tokens, slots.ctypes.data, pairs.ctypes.data, 1,
                                    ctypes.byref(n)), "pa_alloc_append")
        return slots[:n_tokens].copy(), pairs[: n.value].copy()

    def free_seq(self, seq_id: int) -> None:
        _ok(self._L.pa_alloc_free_seq(self._h, seq_id), "pa_alloc_free_seq")

    def block_table(self, seq_id: int) -> list[int]:
        n = _i64(0)
        _ok(self._L.pa_alloc_block_table(self._h, seq_id, None, 0, ctypes.byref(n)), "pa_alloc_block_table")
        out = np.empty(max(n.value, 1), np.int32)
        _ok(self._L.pa_alloc_block_table(self._h, seq_id, out.ctypes.data, n.value, ctypes.byref(n)),
            "pa_alloc_block_table")
        return out[: n.value].tolist()

    def length(self, seq_id: int) -> int:
        n = _i64(0)
        _ok(self._L.pa_alloc_seq_len(self._h, seq_id, ctypes.byref(n)), "pa_alloc_seq_len")
        return int(n.value)

    def export(self, seq_ids, max_blocks_per_seq: int):
        """(block_tables int32 [n, max_blocks_per_seq] padded with -1, context_lens int32 [n])."""
        ids = np.ascontiguousarray(seq_ids, dtype=np.int64)
        tables = np.empty((ids.shape[0], max_blocks_per_seq), np.int32)
        lens = np.empty(ids.shape[0], np.int32)
        _ok(self._L.pa_alloc_export(self._h, ids.ctypes.data, ids.shape[0], tables.ctypes.data,
                                    max_blocks_per_seq, lens.ctypes.data), "pa_alloc_export")
        return tables, lens

    def alloc(self) -> int:
        b = ctypes.c_int32(0)
        _ok(self._L.pa_alloc_block(self._h, ctypes.byref(b)), "pa_alloc_block")
        return int(b.value)

    def decref(self, block: int) -> None:
        _ok(self._L.pa_alloc_decref(self._h, block), "pa_alloc_decref")

    def refcount(self, block: int) -> int:
        c = ctypes.c_int32(0)
        _ok(self._L.pa_alloc_refcount(self._h, block, ctypes.byref(c)), "pa_alloc_refcount")
        return int(c.value)

    def snapshot(self) -> bytes:
        """The allocator's whole state as bytes (see pa_alloc_snapshot)."""
        n = _i64(0)
        _ok(self._L.pa_alloc_snapshot(self._h, None, 0, ctypes.byref(n)), "pa_alloc_snapshot")
        buf = ctypes.create_string_buffer(max(n.value, 1))
        _ok(self._L.pa_alloc_snapshot(self._h, buf, n.value, ctypes.byref(n)), "pa_alloc_snapshot")
        return buf.raw[: n.value]

    @classmethod
    def restore(cls, image: bytes) -> "BlockAllocator":
        """A new allocator in the state a snapshot recorded (see pa_alloc_restore)."""
        L = lib()
        h = _vp()
        data = bytes(image)
        _ok(L.pa_alloc_restore(data, len(data), ctypes.byref(h)), "pa_alloc_restore")
        self = cls.__new__(cls)
        self._L, self._h = L, h
        st = self.stats()
        self.num_blocks, self.block_size = st.num_blocks, int.from_bytes(data[16:24], "little", signed=True)
        return self

    def stats(self) -> AllocStats:
        s = _Stats()
        _ok(self._L.pa_alloc_get_stats(self._h, ctypes.byref(s)), "pa_alloc_get_stats")
        return AllocStats(s.num_blocks, s.num_free, s.num_used, s.peak_used, s.num_cow_copies, s.num_seqs)
