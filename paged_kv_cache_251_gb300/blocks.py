"""Thin ctypes binding of the host block manager (include/pa_block_manager.h)."""
from __future__ import annotations

import ctypes

import torch

from .pa import PagedAttentionError, _lib

P, I, I64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
_lib.pa_bm_create.argtypes = [I, I, I, I, P]
_lib.pa_bm_create.restype = P
_lib.pa_bm_destroy.argtypes = [P]
_lib.pa_bm_destroy.restype = None
_lib.pa_bm_add_sequence.argtypes = [P, I, I]
_lib.pa_bm_add_sequence.restype = I
_lib.pa_bm_fork.argtypes = [P, I, I]
_lib.pa_bm_fork.restype = I
_lib.pa_bm_free_sequence.argtypes = [P, I]
_lib.pa_bm_free_sequence.restype = I
_lib.pa_bm_append.argtypes = [P, P, I, P, P, I, P, P]
_lib.pa_bm_append.restype = I
_lib.pa_bm_length.argtypes = [P, I]
_lib.pa_bm_length.restype = ctypes.c_longlong
_lib.pa_bm_tables.argtypes = [P, P, P]
_lib.pa_bm_tables.restype = I
_lib.pa_bm_refcount.argtypes = [P, I]
_lib.pa_bm_refcount.restype = I
_lib.pa_bm_num_free.argtypes = [P]
_lib.pa_bm_num_free.restype = I


def _check(st: int):
    if st != 0:
        raise PagedAttentionError(st, "block manager")


class BlockManager:
    """Pool of physical blocks, per-sequence block tables, reference counts,
    copy-on-write and sliding-window rings (all in native code)."""

    def __init__(self, num_blocks: int, block_size: int, max_seqs: int, max_blocks_per_seq: int,
                 free_order=None):
        self.num_blocks, self.block_size = num_blocks, block_size
        self.max_seqs, self.max_blocks_per_seq = max_seqs, max_blocks_per_seq
        fo = None
        if free_order is not None:
            fo = torch.as_tensor(free_order, dtype=torch.int32).contiguous()
            assert fo.numel() == num_blocks
        self._h = _lib.pa_bm_create(num_blocks, block_size, max_seqs, max_blocks_per_seq,
                                    None if fo is None else ctypes.c_void_p(fo.data_ptr()))
        if not self._h:
            raise ValueError("bad block manager arguments")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            _lib.pa_bm_destroy(h)
            self._h = None

    def add_sequence(self, seq: int, ring_blocks: int = 0) -> None:
        _check(_lib.pa_bm_add_sequence(self._h, seq, ring_blocks))

    def fork(self, parent: int, child: int) -> None:
        _check(_lib.pa_bm_fork(self._h, parent, child))

    def free_sequence(self, seq: int) -> None:
        _check(_lib.pa_bm_free_sequence(self._h, seq))

    def append(self, seqs, pairs_cap: int | None = None):
        """Place one token at the end of each listed sequence (in order).
        Returns (slots int64 [n], copy pairs int64 [k, 2])."""
        s = torch.as_tensor(seqs, dtype=torch.int32).contiguous()
        n = s.numel()
        cap = n if pairs_cap is None else pairs_cap
        slots = torch.empty(n, dtype=torch.int64)
        pairs = torch.empty((max(cap, 1), 2), dtype=torch.int64)
        np_, placed = ctypes.c_int(0), ctypes.c_int(0)
        st = _lib.pa_bm_append(self._h, ctypes.c_void_p(s.data_ptr()), n, ctypes.c_void_p(slots.data_ptr()),
                               ctypes.c_void_p(pairs.data_ptr()), cap, ctypes.byref(np_), ctypes.byref(placed))
        if st != 0:
            raise PagedAttentionError(st, f"block manager append stopped after {placed.value} tokens")
        return slots, pairs[:np_.value].clone()

    def extend(self, seq: int, ntokens: int):
        """Place ntokens tokens at the end of one sequence."""
        return self.append([seq] * ntokens)

    def length(self, seq: int) -> int:
        return int(_lib.pa_bm_length(self._h, seq))

    def tables(self):
        """(block_tables int32 [max_seqs, max_blocks_per_seq], lengths int32 [max_seqs])."""
        t = torch.empty((self.max_seqs, self.max_blocks_per_seq), dtype=torch.int32)
        lens = torch.empty(self.max_seqs, dtype=torch.int32)
        _check(_lib.pa_bm_tables(self._h, ctypes.c_void_p(t.data_ptr()), ctypes.c_void_p(lens.data_ptr())))
        return t, lens

    def refcount(self, block: int) -> int:
        return int(_lib.pa_bm_refcount(self._h, block))

    def num_free(self) -> int:
        return int(_lib.pa_bm_num_free(self._h))
