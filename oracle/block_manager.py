"""Reference-counted block manager (oracle; test infrastructure only).

Follows the pages step by step:

* A block holds ``block_size`` consecutive tokens; a sequence takes a new
  block only when its last one is full ("PagedAttention" (tensortonic),
  section 3: with 4-token blocks, 6 tokens use 2 blocks and token 9 opens a
  third; "PagedAttention and vLLM: Paging the KV Cache Like an OS", Step 3,
  request A's walk-through).
* Free blocks wait in a first-in-first-out queue; a finished sequence's blocks
  go back to it ("vLLM's PagedAttention ...", section 7 skeleton and section
  2.4 free queue).
* Forking a sequence copies its block table and raises each block's reference
  count ("PagedAttention and vLLM ...", Step 4, beam search paragraph).
* A write into a block that others still hold (count above one) goes to a
  fresh copy of it: the writer's table entry is switched to the copy and the
  shared block's count drops by one; a writer that holds the block alone
  (count one) writes straight into it ("PagedAttention and vLLM ...", Step 4,
  parallel sampling paragraph).

The manager tracks metadata only.  The copies it asks for are returned as
(src, dst) pairs; ``paged_ops.copy_blocks`` moves the bytes.
"""
from __future__ import annotations

from collections import deque
from typing import Dict, Iterable, List, Optional, Tuple


class OutOfBlocks(RuntimeError):
    pass


class BlockManager:
    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Optional[Iterable[int]] = None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        assert sorted(order) == list(range(num_blocks)), "free order must be a permutation"
        self.free: deque = deque(order)
        self.refcount: List[int] = [0] * self.num_blocks
        self.tables: Dict[int, List[int]] = {}
        self.lens: Dict[int, int] = {}
        self.copies: List[Tuple[int, int]] = []   # every CoW (src, dst) so far

    # -- allocation -------------------------------------------------------
    def _pop_free(self) -> int:
        if not self.free:
            raise OutOfBlocks("no free block left")
        b = self.free.popleft()
        assert self.refcount[b] == 0
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        assert self.refcount[b] > 0
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self.free.append(b)

    # -- sequence operations ------------------------------------------------
    def add_sequence(self, seq: int) -> None:
        assert seq not in self.tables
        self.tables[seq] = []
        self.lens[seq] = 0

    def append(self, seq: int) -> Tuple[int, Optional[Tuple[int, int]]]:
        """Reserve the slot for the sequence's next token.

        Returns (slot, cow) where slot = physical_block * block_size + offset
        and cow is the (src, dst) block copy that must run before the write,
        or None.
        """
        table = self.tables[seq]
        n = self.lens[seq]
        offset = n % self.block_size
        cow = None
        if offset == 0:
            # the last block is full (or there is none): take a fresh one
            table.append(self._pop_free())
        else:
            last = table[-1]
            if self.refcount[last] > 1:
                fresh = self._pop_free()
                self.refcount[last] -= 1      # still > 0: others share it
                table[-1] = fresh
                cow = (last, fresh)
                self.copies.append(cow)
        slot = table[n // self.block_size] * self.block_size + offset
        self.lens[seq] = n + 1
        return slot, cow

    def append_tokens(self, seq: int, count: int):
        slots, cows = [], []
        for _ in range(count):
            s, c = self.append(seq)
            slots.append(s)
            if c is not None:
                cows.append(c)
        return slots, cows

    def fork(self, parent: int, child: int) -> None:
        assert child not in self.tables
        self.tables[child] = list(self.tables[parent])
        self.lens[child] = self.lens[parent]
        for b in self.tables[child]:
            self.refcount[b] += 1

    def free_sequence(self, seq: int) -> None:
        for b in self.tables.pop(seq):
            self._release(b)
        del self.lens[seq]

    # -- queries ------------------------------------------------------------
    def num_used_blocks(self) -> int:
        return self.num_blocks - len(self.free)

    def slot_of(self, seq: int, pos: int) -> int:
        """Physical slot holding token ``pos`` (0-based) of ``seq``."""
        assert 0 <= pos < self.lens[seq]
        return self.tables[seq][pos // self.block_size] * self.block_size + pos % self.block_size

    def check_invariants(self) -> None:
        total_refs = sum(self.refcount)
        total_entries = sum(len(t) for t in self.tables.values())
        assert total_refs == total_entries, (total_refs, total_entries)
        free = set(self.free)
        assert len(free) == len(self.free), "a block is queued twice"
        for b in range(self.num_blocks):
            assert (self.refcount[b] == 0) == (b in free), b
        for s, t in self.tables.items():
            n = self.lens[s]
            assert len(t) == -(-n // self.block_size), (s, len(t), n)
