"""Plain-Python model of paged block tables (test infrastructure; see the
package docstring).

Sources (page title, section):
  * "Module 10: inference and serving", section "Mapping logical positions to
    physical blocks": storage is split into fixed-size blocks; a sequence's
    block table maps logical block numbers to physical blocks of a shared pool;
    a growing request takes one more block instead of reserving its future;
    at most block_size - 1 tail slots per sequence are unused.
  * same page, section "Share only identical state": continuations of one
    prompt reference the same full prefix blocks; a reference count records
    how many sequences use each block; a write into a shared block that is
    not yet full first gets a private copy (copy-on-write); full prefix blocks
    stay shared.
  * "Ch. 6 Inference efficiency and serving", section 6.4: branches with the
    same prefix point at the same read-only physical block and get a new block
    when the fork writes.

Readings where the pages are silent:
  * append at logical position pos (the length before the append): if pos
    starts a new block and the table has no block there, allocate one; if the
    block holding pos is shared (count > 1), copy-on-write: allocate a private
    block, point the table at it, drop one reference to the old block, and
    report (old, new) so the caller copies the contents on the device.
  * fork(n_tokens) shares every block that holds one of the first n_tokens
    tokens, the partial last one included; the first write into that partial
    block takes the copy-on-write path above.
  * allocation is all-or-nothing; on failure nothing changes.
"""
from __future__ import annotations

from typing import Iterable, List, Optional, Sequence, Tuple


class OutOfBlocks(Exception):
    pass


class BlockError(Exception):
    pass


class BlockModel:
    def __init__(self, num_blocks: int):
        if num_blocks <= 0:
            raise BlockError("num_blocks must be positive")
        self.num_blocks = num_blocks
        self.ref = [0] * num_blocks

    # -- pool -------------------------------------------------------------
    def num_free(self) -> int:
        return sum(1 for r in self.ref if r == 0)

    def refcount(self, i: int) -> int:
        if not 0 <= i < self.num_blocks:
            return -1
        return self.ref[i]

    def allocate(self, n: int, chosen: Optional[Sequence[int]] = None) -> List[int]:
        """Take n free blocks (count 1 each).  `chosen` lets a test replay the
        ids another allocator picked; they must be distinct and free."""
        if n < 0:
            raise BlockError("negative count")
        if n > self.num_free():
            raise OutOfBlocks()
        if chosen is None:
            ids = [i for i, r in enumerate(self.ref) if r == 0][:n]
        else:
            ids = list(chosen)
            if len(ids) != n or len(set(ids)) != n:
                raise BlockError("chosen ids must be n distinct ids")
            for i in ids:
                if not 0 <= i < self.num_blocks or self.ref[i] != 0:
                    raise BlockError("chosen id %d is not free" % i)
        for i in ids:
            self.ref[i] = 1
        return ids

    def share(self, ids: Iterable[int]) -> None:
        ids = list(ids)
        for i in ids:
            if not 0 <= i < self.num_blocks or self.ref[i] == 0:
                raise BlockError("share of a block that is not allocated: %d" % i)
        for i in ids:
            self.ref[i] += 1

    def release(self, ids: Iterable[int]) -> None:
        ids = list(ids)
        need = {}
        for i in ids:
            need[i] = need.get(i, 0) + 1
        for i, c in need.items():
            if not 0 <= i < self.num_blocks or self.ref[i] < c:
                raise BlockError("release of a block with too few references: %d" % i)
        for i in ids:
            self.ref[i] -= 1

    # -- block tables -----------------------------------------------------
    def append_slot(self, row: List[int], pos: int, block_size: int,
                    chosen: Optional[int] = None) -> Tuple[int, int]:
        """Make the slot of logical position `pos` writable in table `row`
        (entries -1 when unassigned).  Returns (cow_src, cow_dst), both -1
        when no copy is needed."""
        j = pos // block_size
        if pos < 0 or j >= len(row):
            raise BlockError("position outside the table row")
        if row[j] < 0:
            # a block opens only at its first slot, right after the previous one
            if pos % block_size != 0 or (j > 0 and row[j - 1] < 0):
                raise BlockError("gap in the table row")
            (new,) = self.allocate(1, None if chosen is None else [chosen])
            row[j] = new
            return -1, -1
        old = row[j]
        if self.refcount(old) <= 0:
            raise BlockError("table points at a free block")
        if self.ref[old] > 1:
            (new,) = self.allocate(1, None if chosen is None else [chosen])
            row[j] = new
            self.release([old])
            return old, new
        return -1, -1

    def fork(self, src_row: Sequence[int], n_tokens: int, block_size: int,
             dst_row: List[int]) -> None:
        nblk = (n_tokens + block_size - 1) // block_size
        if nblk > len(dst_row) or nblk > len(src_row):
            raise BlockError("fork longer than the table row")
        ids = list(src_row[:nblk])
        self.share(ids)
        for j, i in enumerate(ids):
            dst_row[j] = i


def blocks_for(n_tokens: int, block_size: int) -> int:
    """Blocks a sequence of n_tokens holds: ceil(n / bs)."""
    return (n_tokens + block_size - 1) // block_size
