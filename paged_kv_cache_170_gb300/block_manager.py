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

import heapq
from collections import deque
from typing import Hashable, Iterable, Optional

import numpy as np


class PoolExhausted(RuntimeError):
    """No free physical block is left; the manager's state is unchanged."""


class BlockManagerError(RuntimeError):
    """Misuse: unknown sequence, double free, or a broken invariant."""


class BlockManager:
    """``policy`` picks the free block a sequence gets:

    * ``"queue"`` (the demo's): the front of the free queue (``free_order``,
      then blocks in the order they were freed);
    * ``"contiguous"``: the block right after the sequence's last one when it
      is free, else the lowest free id; a new sequence takes the first run of
      consecutive free ids long enough for it.  This is the pages' remedy for
      scattered blocks (cf-1.com news/5879632, section 5.1: keep a sequence's
      blocks physically together so reads stay linear).
    """

    def __init__(self, num_blocks: int, block_size: int, free_order: Optional[Iterable[int]] = None,
                 policy: str = "queue"):
        if num_blocks <= 0 or block_size <= 0:
            raise ValueError("num_blocks and block_size must be positive")
        if policy not in ("queue", "contiguous"):
            raise ValueError(f"unknown policy {policy!r}")
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        self.policy = policy
        order = list(range(num_blocks)) if free_order is None else [int(p) for p in free_order]
        if sorted(order) != list(range(num_blocks)):
            raise ValueError("free_order must be a permutation of the pool ids")
        self.refs = [0] * self.num_blocks
        self._nfree = self.num_blocks
        # queue policy: the free queue; contiguous policy: a heap of free ids
        # (count 0 marks a block free; entries of blocks taken since are skipped)
        self.free = deque(order) if policy == "queue" else deque()
        self._free_heap = list(order) if policy == "contiguous" else []
        heapq.heapify(self._free_heap)
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
            self._nfree += 1
            if self.policy == "queue":
                self.free.append(pid)
            else:
                heapq.heappush(self._free_heap, pid)

    def _take(self, pid: int) -> int:
        self.refs[pid] = 1
        self._nfree -= 1
        return pid

    def _alloc(self, after: Optional[int] = None) -> int:
        """One free block (after ``after``, the sequence's last block, when the
        contiguous policy can)."""
        if self._nfree == 0:
            raise PoolExhausted("no free physical block")
        if self.policy == "queue":
            return self._take(self.free.popleft())
        if after is not None and after + 1 < self.num_blocks and self.refs[after + 1] == 0:
            return self._take(after + 1)
        while self.refs[self._free_heap[0]] != 0:  # entries of blocks taken since
            heapq.heappop(self._free_heap)
        return self._take(heapq.heappop(self._free_heap))

    def _alloc_run(self, n: int) -> list[int]:
        """n blocks for a new sequence: the first run of n consecutive free ids
        (contiguous policy), else one by one."""
        if self.policy == "contiguous" and n > 1:
            run = 0
            for pid in range(self.num_blocks):
                run = run + 1 if self.refs[pid] == 0 else 0
                if run == n:
                    return [self._take(p) for p in range(pid - n + 1, pid + 1)]
        out: list[int] = []
        for _ in range(n):
            out.append(self._alloc(out[-1] if out else None))
        return out

    # -- sequence operations ---------------------------------------------------
    def blocks_for(self, tokens: int) -> int:
        return -(-int(tokens) // self.block_size)

    def allocate(self, seq: Hashable, num_tokens: int) -> list[int]:
        """Prefill: a new sequence holding ``num_tokens`` tokens."""
        if seq in self.tables:
            raise BlockManagerError(f"sequence {seq!r} exists")
        need = self.blocks_for(num_tokens)
        if need > self._nfree:
            raise PoolExhausted(f"need {need} blocks, {self._nfree} free")
        self.tables[seq] = self._alloc_run(need)
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
            table.append(self._alloc(table[-1] if table else None))
        else:
            last = table[-1]
            if self.refs[last] > 1:
                new = self._alloc(table[-2] if len(table) > 1 else None)
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
        return self._nfree

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
        zero = {p for p in range(self.num_blocks) if self.refs[p] == 0}
        if len(zero) != self._nfree:
            raise BlockManagerError("free count does not match the zero-count blocks")
        if self.policy == "queue":
            free = list(self.free)
            if len(set(free)) != len(free):
                raise BlockManagerError("a block is twice in the free list")
            if set(free) != zero:
                raise BlockManagerError("free list does not match the zero-count blocks")
        elif not zero <= set(self._free_heap):
            raise BlockManagerError("a free block is missing from the free heap")


def pool_report(block_tables, context_lens, block_size: int, bytes_per_token: int,
                max_len: Optional[int] = None) -> dict:
    """The pages' memory figures for a set of block tables (host, no GPU).

    aiqz.cc "paged-attention-mechanism", section "显存收益分析": the waste
    ratio eta = (M_alloc - M_used) / M_alloc, and its estimate for paged
    allocation, eta' ~ 1 / (2 N_blocks) (on average half of each request's
    last block is empty); section "前缀共享机制": a prefix of N_p blocks
    shared by R requests saves M_saved = N_p * B * bytes * (R - 1).

    Here M_alloc counts each distinct physical block a table references once;
    M_used counts the tokens stored in those blocks (a shared block holds the
    most tokens any of its sharers has in it); M_saved sums, over the
    referenced blocks, (references - 1) * B * bytes, which is the pages'
    formula for a prefix shared by R; eta_prime is the pages' estimate
    averaged over the requests holding at least one block.  With ``max_len``
    the report adds what reserving max_len tokens per request up front would
    take (the contiguous scheme the pages compare against) and its use.
    ``bytes_per_token`` is the K plus V bytes of one token over all kv heads.
    """
    tables = np.asarray(block_tables)
    lens = np.asarray(context_lens, dtype=np.int64)
    B = int(block_size)
    refs: dict[int, int] = {}
    fill: dict[int, int] = {}
    eta_prime, logical_blocks = [], 0
    for s in range(len(lens)):
        L = int(max(lens[s], 0))
        nb = -(-L // B)
        logical_blocks += nb
        if nb:
            eta_prime.append(1.0 / (2 * nb))
        for i in range(nb):
            pid = int(tables[s, i])
            refs[pid] = refs.get(pid, 0) + 1
            fill[pid] = max(fill.get(pid, 0), min(B, L - i * B))
    m_alloc = len(refs) * B * bytes_per_token
    m_used = sum(fill.values()) * bytes_per_token
    out = {
        "requests": int(len(lens)),
        "tokens": int(lens.clip(min=0).sum()),
        "blocks_referenced": int(logical_blocks),
        "blocks_distinct": int(len(refs)),
        "m_alloc_bytes": int(m_alloc),
        "m_used_bytes": int(m_used),
        "eta_waste": (m_alloc - m_used) / m_alloc if m_alloc else 0.0,
        "eta_prime_estimate": float(np.mean(eta_prime)) if eta_prime else 0.0,
        "m_saved_bytes": int(sum(r - 1 for r in refs.values()) * B * bytes_per_token),
    }
    if max_len is not None:
        reserved = len(lens) * int(max_len) * bytes_per_token
        out["contiguous_reserved_bytes"] = int(reserved)
        out["contiguous_utilisation"] = out["tokens"] * bytes_per_token / reserved if reserved else 0.0
        out["paged_utilisation"] = m_used / m_alloc if m_alloc else 0.0
    return out
