"""Block-table bookkeeping models for the oracle (plain Python, small state).

TEST INFRASTRUCTURE ONLY (see the package docstring).

CowModel follows "PagedAttention — 把 KV cache 当虚拟内存页来管理", 实践案例
案例 3 (copy-on-write serving several candidates): blocks carry a reference
count; a write into a block whose count is above one first drops one
reference, takes a fresh block, copies the old block into it (one whole block
is the copy unit) and writes there; a sole owner writes in place.  New blocks
come from a free list on demand (核心要点: a sequence holds a list of block
numbers, not one contiguous region).

RingModel follows "KV Cache与长上下文管理", section "让 Round Robin / Sliding
Window 变成 O(1) 操作", and "PagedAttention的终极用途": a sliding window keeps a
fixed ring of physical pages; moving into a new page recycles the oldest one
and changes only the page table — no K/V bytes move.
"""
from __future__ import annotations

from collections import deque


class CowModel:
    """Reference counts, per-sequence block tables and copy-on-write."""

    def __init__(self, block_size: int, free_blocks):
        self.bs = int(block_size)
        self.free = deque(int(b) for b in free_blocks)
        self.ref: dict[int, int] = {}
        self.tables: dict[int, list[int]] = {}

    def _take(self) -> int:
        if not self.free:
            raise MemoryError("block pool exhausted")
        b = self.free.popleft()
        self.ref[b] = 1
        return b

    def add_sequence(self, sid: int) -> None:
        self.tables[sid] = []

    def fork(self, parent: int, child: int) -> None:
        """The child shares every block of the parent (one more reference each)."""
        self.tables[child] = list(self.tables[parent])
        for b in self.tables[child]:
            self.ref[b] += 1

    def write(self, sid: int, pos: int):
        """Place token ``pos`` of sequence ``sid``.  Returns (slot, copy) where
        copy is (src, dst) when the write had to copy a shared block first."""
        table = self.tables[sid]
        logical, offset = divmod(pos, self.bs)
        if logical == len(table):
            table.append(self._take())
        elif logical > len(table):
            raise ValueError("tokens are written in order")
        block = table[logical]
        copy = None
        if self.ref[block] > 1:
            self.ref[block] -= 1
            fresh = self._take()
            copy = (block, fresh)
            table[logical] = fresh
            block = fresh
        return block * self.bs + offset, copy

    def free_sequence(self, sid: int) -> None:
        for b in self.tables.pop(sid):
            self.ref[b] -= 1
            if self.ref[b] == 0:
                del self.ref[b]
                self.free.append(b)


class RingModel:
    """One sequence whose K/V lives in a fixed ring of physical blocks.

    Logical block ``lb`` is stored in ``ring[lb % len(ring)]``; the block table
    row is rewritten when the sequence moves into a new logical block.  Table
    entries of logical blocks that the ring has recycled are set to
    ``stale`` (they must never be read).
    """

    def __init__(self, block_size: int, ring_blocks, table_len: int, stale: int = -1):
        self.bs = int(block_size)
        self.ring = [int(b) for b in ring_blocks]
        self.table = [stale] * int(table_len)
        self.stale = stale
        self.length = 0
        self.data_moves = 0  # bytes of K/V the model ever moved (stays 0)

    def write(self, pos: int) -> int:
        """Place token ``pos`` (tokens arrive in order) and return its slot."""
        if pos != self.length:
            raise ValueError("tokens are written in order")
        logical, offset = divmod(pos, self.bs)
        if offset == 0:
            r = len(self.ring)
            if logical >= r:
                self.table[logical - r] = self.stale   # its page is recycled now
            self.table[logical] = self.ring[logical % r]
        self.length += 1
        return self.table[logical] * self.bs + offset
