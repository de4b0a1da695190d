"""Host-side block manager: free list, reference counts, prefix sharing, COW.

Plumbing around the GPU path, not part of it.  Semantics follow the pages:

* aiqz.cc "paged-attention-mechanism", section "分页核心思想": blocks are
  taken on demand as a sequence grows (ceil(tokens / B) blocks);
  section "前缀共享机制": shared blocks are read-only and counted by reference;
  a write into a block whose count is above one first takes a new block,
  copies the old contents, writes, and drops the old count by one;
  section "Python 演示": free blocks are handed out from the front of a queue,
  a fork shares the first ceil(n / B) blocks of its parent, and a new token
  takes a fresh block exactly when the last one is full.
* cf-1.com news/5879632, section 3.2: on release, each table entry is unmapped
  first and its count decremented after; a block returns to the pool only at
  count zero.  Section 4.3: all count changes go through inc_ref/dec_ref, and
  a debug audit compares the sum of counts with the table references.
* ipipp.com "PagedAttention原理是什么？…", section "分页式KV缓存的底层设计":
  a table is an append-only logical -> physical list.

The copy itself is left to the device (``pa_copy_blocks``): ``append_slot``
returns the (src, dst) pair to copy before the token's K/V is written.
"""
from __future__ import annotations

from collections import deque
from typing import Hashable, Iterable, Optional

import numpy as np


class PoolExhausted(RuntimeError):
    """No free physical block is left; the manager's state is unchanged."""


class BlockManagerError(RuntimeError):
    """Misuse: unknown sequence, double free, or a broken invariant."""


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Iterable[int]] = None):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(p) for p in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the pool ids")
        self.refs = [0] * self.num_blocks
        self.free = deque(order)
        self.tables: dict[Hashable, list[int]] = {}
        self.used: dict[Hashable, int] = {}

    # -- reference counting (the only places counts change) ------------------
    def inc_ref(self, pid: int) -> None:
        if self.refs[pid] <= 0:
            raise BlockManagerError(f"inc_ref on free block {pid}")
        self.refs[pid] += 1

    def dec_ref(self, pid: int) -> None:
        if self.refs[pid] <= 0:
            raise BlockManagerError(f"dec_ref on free block {pid} (double free)")
        self.refs[pid] -= 1
        if self.refs[pid] == 0:
            self.free.append(pid)

    def _alloc(self) -> int:
        if not self.free:
            raise PoolExhausted("no free physical block")
        pid = self.free.popleft()
        self.refs[pid] = 1
        return pid

    # -- sequence operations ---------------------------------------------------
    def blocks_for(self, tokens: int) -> int:
        return -(-int(tokens) // self.block_size)

    def allocate(self, seq: Hashable, num_tokens: int) -> list[int]:
        """Prefill: a new sequence holding ``num_tokens`` tokens."""
        if seq in self.tables:
            raise BlockManagerError(f"sequence {seq!r} exists")
        need = self.blocks_for(num_tokens)
        if need > len(self.free):
            raise PoolExhausted(f"need {need} blocks, {len(self.free)} free")
        self.tables[seq] = [self._alloc() for _ in range(need)]
        self.used[seq] = int(num_tokens)
        return list(self.tables[seq])

    def fork(self, child: Hashable, parent: Hashable, num_tokens: Optional[int] = None) -> list[int]:
        """Share the first ``num_tokens`` tokens (default: all) of ``parent``."""
        if child in self.tables:
            raise BlockManagerError(f"sequence {child!r} exists")
        if parent not in self.tables:
            raise BlockManagerError(f"unknown sequence {parent!r}")
        n = self.used[parent] if num_tokens is None else int(num_tokens)
        if n > self.used[parent]:
            raise BlockManagerError("cannot share more tokens than the parent holds")
        shared = self.tables[parent][: self.blocks_for(n)]
        for pid in shared:
            self.inc_ref(pid)
        self.tables[child] = list(shared)
        self.used[child] = n
        return list(shared)

    def append_slot(self, seq: Hashable) -> tuple[int, Optional[tuple[int, int]]]:
        """Make room for one new token.

        Returns (slot, cow): ``slot = pid * B + offset`` where the token's K/V
        goes, and ``cow = (src, dst)`` when the last block was shared and had
        to be copied first (``None`` otherwise).
        """
        if seq not in self.tables:
            raise BlockManagerError(f"unknown sequence {seq!r}")
        table = self.tables[seq]
        pos = self.used[seq] % self.block_size
        cow = None
        if pos == 0:
            table.append(self._alloc())
        else:
            last = table[-1]
            if self.refs[last] > 1:
                new = self._alloc()
                table[-1] = new          # remap first ...
                self.dec_ref(last)       # ... then drop the shared count
                cow = (last, new)
        self.used[seq] += 1
        return table[-1] * self.block_size + pos, cow

    def free_seq(self, seq: Hashable) -> None:
        """Release a sequence: unmap its table, then drop each block's count."""
        if seq not in self.tables:
            raise BlockManagerError(f"unknown sequence {seq!r} (double free?)")
        table = self.tables.pop(seq)
        del self.used[seq]
        for pid in table:
            self.dec_ref(pid)

    # -- views -------------------------------------------------------------------
    def block_tables(self, seqs: list, width: Optional[int] = None, pad: int = -1) -> np.ndarray:
        width = max((len(self.tables[s]) for s in seqs), default=0) if width is None else width
        out = np.full((len(seqs), width), pad, dtype=np.int32)
        for i, s in enumerate(seqs):
            row = self.tables[s]
            if len(row) > width:
                raise BlockManagerError("table wider than requested width")
            out[i, : len(row)] = row
        return out

    def context_lens(self, seqs: list) -> np.ndarray:
        return np.array([self.used[s] for s in seqs], dtype=np.int32)

    def num_free(self) -> int:
        return len(self.free)

    def num_used_blocks(self) -> int:
        return sum(1 for r in self.refs if r > 0)

    def check(self) -> None:
        """Audit: counts equal table references; free list holds exactly the count-0 blocks."""
        counted = [0] * self.num_blocks
        for s, row in self.tables.items():
            if len(row) != self.blocks_for(self.used[s]):
                raise BlockManagerError(f"sequence {s!r}: {len(row)} blocks for {self.used[s]} tokens")
            for pid in row:
                counted[pid] += 1
        if counted != self.refs:
            bad = [p for p in range(self.num_blocks) if counted[p] != self.refs[p]][:8]
            raise BlockManagerError(f"reference counts disagree with tables at blocks {bad}")
        free = list(self.free)
        if len(set(free)) != len(free):
            raise BlockManagerError("a block is twice in the free list")
        if set(free) != {p for p in range(self.num_blocks) if self.refs[p] == 0}:
            raise BlockManagerError("free list does not match the zero-count blocks")
