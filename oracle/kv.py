"""KV block pool bookkeeping (oracle side).

TEST INFRASTRUCTURE ONLY (see the package docstring).

Source: AX Engine page, "Core Technical Architecture & Methods": the KV
cache grows inside preallocated buffers, a speculation rollback is O(1)
because only the sequence length moves, and the scheduler and KV manager
recover memory blocks.  The page does not fix the block layout; the reading
used here (and by the GPU library):

* the buffers are a pool of num_blocks blocks of block_size positions; a
  sequence's positions 0, 1, ... live in the blocks of its table, in order;
* before a forward that writes `extra` more positions, a sequence holds
  ceil((kv_len + extra) / block_size) blocks (at most max_blocks; short when
  the pool or the table row runs out, keeping what it got);
* a rollback moves kv_len only; trimming returns the blocks past
  ceil(kv_len / block_size); a finished sequence returns all its blocks;
* free blocks form a stack holding num_blocks - 1, ..., 0 from the bottom, so
  a lone sequence takes blocks 0, 1, 2, ... in that order.

The sequences are served one after another in index order here; the device
serves them at once, so with several sequences only the counts, not which
block went where, are unique (when the pool runs short, only the totals).

Pinned by: tests/test_oracle_kv.py (hand-worked pool traces, the conservation
of blocks, ceil-division closed forms).
"""
from __future__ import annotations

import math
from typing import List


def blocks_for(length: int, block_size: int) -> int:
    """Blocks that hold `length` positions (negative lengths count as 0)."""
    return math.ceil(max(int(length), 0) / block_size)


class KvPool:
    def __init__(self, num_blocks: int, B: int, max_blocks: int, block_size: int):
        self.num_blocks, self.B, self.max_blocks, self.block_size = num_blocks, B, max_blocks, block_size
        self.free: List[int] = list(range(num_blocks - 1, -1, -1))  # top of the stack = end of the list
        self.tables: List[List[int]] = [[] for _ in range(B)]
        self.short = False

    def reserve(self, kv_len, extra: int):
        for b in range(self.B):
            want = blocks_for(int(kv_len[b]) + extra, self.block_size)
            if want > self.max_blocks:
                self.short = True
                want = self.max_blocks
            while len(self.tables[b]) < want:
                if not self.free:
                    self.short = True
                    break
                self.tables[b].append(self.free.pop())

    def trim(self, kv_len):
        for b in range(self.B):
            keep = min(len(self.tables[b]), blocks_for(int(kv_len[b]), self.block_size))
            for blk in self.tables[b][keep:]:
                self.free.append(blk)
            del self.tables[b][keep:]

    def release(self, done):
        for b in range(self.B):
            if int(done[b]) != 0:
                self.free.extend(self.tables[b])
                self.tables[b] = []

    def counts(self):
        return [len(t) for t in self.tables]
