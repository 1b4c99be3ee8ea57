"""Reference model of the host-side paged KV block allocator and slot mapper.

Test infrastructure only.  The library's C++ allocator must reproduce this model bit for
bit (same block ids, same order, same errors) on any sequence of calls.

Source: "GPU waiting, not working" (nanoserve notes), the change table's "faster way of
mapping tokens to cache slots"; "NanoFlow: ..." page, "Runtime details that keep the pipeline
fed": KV lives in fragmented PagedAttention pages.  The policy details are this library's
own reading (the pages give none):

* The pool has ``num_blocks`` blocks of ``block_size`` token slots.  The free list starts as
  0, 1, ..., num_blocks-1; ``alloc`` takes from the front and ``release`` appends to the back
  (first-in first-out reuse).
* ``prepare_step``: for each request b in order, position p = positions[b]; when p is the
  first slot of a block (p % bs == 0) a block is taken and stored at table[b][p // bs]; the
  slot is table[b][p // bs] * bs + p % bs.  Running out of blocks or past the table width is an
  error, raised before anything is changed.
"""
from __future__ import annotations

from collections import deque
from typing import Iterable, List

import numpy as np


class AllocatorError(RuntimeError):
    pass


class BlockAllocator:
    def __init__(self, num_blocks: int, block_size: int):
        if num_blocks <= 0 or block_size <= 0:
            raise AllocatorError("invalid pool size")
        self.num_blocks = num_blocks
        self.block_size = block_size
        self.free = deque(range(num_blocks))

    def free_count(self) -> int:
        return len(self.free)

    def alloc(self, n: int) -> List[int]:
        if n < 0 or n > len(self.free):
            raise AllocatorError("out of blocks")
        return [self.free.popleft() for _ in range(n)]

    def release(self, ids: Iterable[int]) -> None:
        ids = list(ids)
        for i in ids:
            if not 0 <= i < self.num_blocks:
                raise AllocatorError("block id out of range")
        self.free.extend(ids)

    def prepare_step(self, block_tables: np.ndarray, positions: np.ndarray) -> np.ndarray:
        """Allocate blocks for this step's tokens in place; return int64 slot_mapping [B]."""
        bs = self.block_size
        B, mb = block_tables.shape
        need = 0
        for b in range(B):
            p = int(positions[b])
            if p < 0 or p // bs >= mb:
                raise AllocatorError("position beyond the block table")
            if p % bs == 0:
                need += 1
        if need > len(self.free):
            raise AllocatorError("out of blocks")
        slots = np.empty(B, dtype=np.int64)
        for b in range(B):
            p = int(positions[b])
            if p % bs == 0:
                block_tables[b, p // bs] = self.free.popleft()
            slots[b] = int(block_tables[b, p // bs]) * bs + p % bs
        return slots
