"""Plain-Python block manager of the paged KV cache (test infrastructure only).

Restates, in the simplest possible data structures, the allocation rules of
"Distributed LLM Inference Serving Platform":
  * section 2: blocks come from one pool when needed; the prompt's blocks are
    shared by parallel completions with a reference count and cloned only
    when a diverging token is appended (copy-on-write);
  * section 7, PagedBlockManager: a LIFO free list (pop the last id, push
    freed ids at the end; initial list 0 .. N-1), allocation fails with an
    out-of-memory error when the list is empty, free = reference count - 1
    and return to the list at 0;
  * Lab 1 worked solution: fork copies the parent's table and raises every
    block's count; an append into a shared, partially filled tail clones it
    (the clone holds the tail's tokens plus the new one and replaces the tail
    in the appender's table); the last sharer writes in place; full prefix
    blocks stay shared.  A full tail block is followed by a fresh block.

Independent of the library's C++ manager: the tests compare the two.
"""
from __future__ import annotations


class OutOfBlocks(RuntimeError):
    pass


class BlockManagerOracle:
    def __init__(self, num_blocks: int, block_size: int):
        self.block_size = block_size
        self.free = list(range(num_blocks))
        self.ref = [0] * num_blocks
        self.filled = [0] * num_blocks
        self.tables: dict[int, list[int]] = {}
        self.lengths: dict[int, int] = {}

    def _allocate(self) -> int:
        if not self.free:
            raise OutOfBlocks("GPU out of memory: no free physical block")
        b = self.free.pop()
        self.ref[b] = 1
        self.filled[b] = 0
        return b

    def add_sequence(self, seq: int):
        if seq in self.tables:
            raise ValueError("sequence exists")
        self.tables[seq] = []
        self.lengths[seq] = 0

    def fork(self, parent: int, child: int):
        if parent not in self.tables or child in self.tables:
            raise ValueError("bad fork")
        self.tables[child] = list(self.tables[parent])
        self.lengths[child] = self.lengths[parent]
        for b in self.tables[child]:
            self.ref[b] += 1

    def append_slot(self, seq: int):
        """(slot, copy) where copy is (src, dst, rows) or None."""
        table = self.tables[seq]
        copy = None
        if not table or self.filled[table[-1]] == self.block_size:
            table.append(self._allocate())
        elif self.ref[table[-1]] > 1:
            tail = table[-1]
            new = self._allocate()
            self.ref[tail] -= 1
            self.filled[new] = self.filled[tail]
            copy = (tail, new, self.filled[tail])
            table[-1] = new
        tail = table[-1]
        slot = tail * self.block_size + self.filled[tail]
        self.filled[tail] += 1
        self.lengths[seq] += 1
        return slot, copy

    def free_sequence(self, seq: int):
        for b in self.tables.pop(seq):
            self.ref[b] -= 1
            if self.ref[b] <= 0:
                self.ref[b] = 0
                self.filled[b] = 0
                self.free.append(b)
        del self.lengths[seq]

    def num_free(self) -> int:
        return len(self.free)
