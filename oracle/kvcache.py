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
* A block belongs to at most one request (a slot holds one token of one request), so
  ``release`` accepts only blocks that were handed out and not yet returned, each once per
  call; anything else is an error raised before anything is changed.
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
        self.held = set()

    def free_count(self) -> int:
        return len(self.free)

    def _take(self) -> int:
        i = self.free.popleft()
        self.held.add(i)
        return i

    def alloc(self, n: int) -> List[int]:
        if n < 0 or n > len(self.free):
            raise AllocatorError("out of blocks")
        return [self._take() for _ in range(n)]

    def release(self, ids: Iterable[int]) -> None:
        ids = [int(i) for i in ids]
        for i in ids:
            if not 0 <= i < self.num_blocks:
                raise AllocatorError("block id out of range")
        if len(set(ids)) != len(ids) or not self.held.issuperset(ids):
            raise AllocatorError("block not in use (already free, or twice in one release)")
        self.held.difference_update(ids)
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
                block_tables[b, p // bs] = self._take()
            slots[b] = int(block_tables[b, p // bs]) * bs + p % bs
        return slots


# ------------------------------------------------------------------------------------------
# KV offload rows ("NanoFlow: ..." page, "Runtime details that keep the pipeline fed": K/V
# leave for the host as contiguous vectors right after the KQV projection; on reload they land
# contiguously on the device and are then scattered into the fragmented pages).  The row
# layout is this library's reading (the page gives none): row (layer l, token t) is the K of
# every kv head of that token, heads in order, then its V, in the cache's storage type.
# ------------------------------------------------------------------------------------------

def kv_rows(k_pools: List[np.ndarray], v_pools: List[np.ndarray], slots: Iterable[int]) -> np.ndarray:
    """[n_layers][n][2 * Hkv * d] rows of the tokens at ``slots`` from per-layer pools shaped
    [num_blocks, Hkv, bs, d], copied element for element (no arithmetic)."""
    slots = [int(s) for s in slots]
    L = len(k_pools)
    _, hkv, bs, d = k_pools[0].shape
    out = np.empty((L, len(slots), 2 * hkv * d), dtype=k_pools[0].dtype)
    for l in range(L):
        for t, s in enumerate(slots):
            blk, off = s // bs, s % bs
            for h in range(hkv):
                out[l, t, h * d:(h + 1) * d] = k_pools[l][blk, h, off, :]
                out[l, t, (hkv + h) * d:(hkv + h + 1) * d] = v_pools[l][blk, h, off, :]
    return out


def kv_scatter(k_pools: List[np.ndarray], v_pools: List[np.ndarray], rows: np.ndarray,
               slots: Iterable[int]) -> None:
    """Inverse of ``kv_rows``: write row (l, t) into every layer's pools at slots[t], in place."""
    slots = [int(s) for s in slots]
    _, hkv, bs, d = k_pools[0].shape
    for l in range(len(k_pools)):
        for t, s in enumerate(slots):
            blk, off = s // bs, s % bs
            for h in range(hkv):
                k_pools[l][blk, h, off, :] = rows[l, t, h * d:(h + 1) * d]
                v_pools[l][blk, h, off, :] = rows[l, t, (hkv + h) * d:(hkv + h + 1) * d]


def request_slots(block_table_row: np.ndarray, first_pos: int, n_tokens: int, block_size: int) -> np.ndarray:
    """Slots of positions first_pos .. first_pos + n_tokens - 1 through one block-table row."""
    return np.array([int(block_table_row[p // block_size]) * block_size + p % block_size
                     for p in range(first_pos, first_pos + n_tokens)], dtype=np.int64)
