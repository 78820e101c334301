"""Free-block stack of the physical block pool (test infrastructure only).

Restates the allocator of the mini-infer BlockPool ("Paged KV-Cache Memory
Management", section "Python Implementation: Physical Block Pool"): the free
list starts as the ids 0..num_blocks-1 in increasing order, an allocation takes
the id at the END of the list (so the first one handed out is num_blocks-1),
an exhausted pool raises MemoryError("Out of KV-Cache Physical Blocks"), and
freeing appends the id back to the end (so it is the next one handed out).

The pages do not check double frees or foreign ids; this oracle does, the
plainest reading of a pool that must never hand one block to two sequences.
"""
from __future__ import annotations

from typing import Iterable, List


class FreeBlockStack:
    def __init__(self, num_blocks: int):
        if num_blocks <= 0:
            raise ValueError("num_blocks must be positive")
        self.num_blocks = num_blocks
        self.free_blocks: List[int] = list(range(num_blocks))
        self._in_use = [False] * num_blocks

    def seed(self, order: Iterable[int]) -> None:
        """Replace the free list by a permutation of all ids (all must be free)."""
        order = [int(x) for x in order]
        if any(self._in_use):
            raise ValueError("seed requires every block to be free")
        if sorted(order) != list(range(self.num_blocks)):
            raise ValueError("seed order must be a permutation of 0..num_blocks-1")
        self.free_blocks = order

    def allocate_block(self) -> int:
        if not self.free_blocks:
            raise MemoryError("Out of KV-Cache Physical Blocks")
        blk = self.free_blocks.pop()
        self._in_use[blk] = True
        return blk

    def free_block(self, block_id: int) -> None:
        if not (0 <= block_id < self.num_blocks):
            raise ValueError(f"block id {block_id} outside the pool")
        if not self._in_use[block_id]:
            raise ValueError(f"block {block_id} freed twice")
        self._in_use[block_id] = False
        self.free_blocks.append(block_id)

    def num_free(self) -> int:
        return len(self.free_blocks)
