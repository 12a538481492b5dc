"""Block manager with a prefix cache (oracle; test infrastructure only).

Follows the block pool and hash chain of "PagedAttention and vLLM: Paging the
KV Cache Like an OS" ... section 2.4 ("V1's block pool and hash chain") and
its summary point 5:

* Free blocks wait in one queue ordered by recency of release: released blocks
  go to the back, allocation takes the front, and a block taken from the front
  that still holds cached prefix content is first removed from the cache.  The
  queue order is the eviction order; there is no other LRU structure.
* A hash -> block map finds cached blocks.  Only full blocks are cached.
* A block's key is chained: SHA-256 over (the previous block's key, this
  block's tokens, an extra key such as an adapter id).  The first block's
  previous key is the root value.  One differing token changes every later key.
* A new request walks its prompt's chain block by block; each hit raises the
  block's reference count (taking it out of the free queue if it was there)
  and its tokens need no prefill; the walk stops at the first miss.  A full
  hit still recomputes the last prompt token (its logits are needed), so hits
  only cover blocks inside the first prompt_len - 1 tokens.
* Cached blocks are full and never written again, so sharing them needs no
  copy-on-write: each request fills its own last block.

Readings where the pages are silent (each stated beside the code below): the
byte layout of the hashed message, the root key, the order in which a
finished sequence's blocks enter the free queue, and what happens when a block
fills with content that is already cached.
"""
from __future__ import annotations

import hashlib
import struct
from typing import Dict, Iterable, List, Optional, Sequence, Tuple

ROOT_KEY = bytes(32)   # reading: the first block's "previous key" is 32 zero bytes


class OutOfBlocks(RuntimeError):
    pass


def block_key(parent: bytes, tokens: Sequence[int], extra_key: int) -> bytes:
    """Chained key of one full block.  Reading for the message layout: the
    parent's 32 bytes, each token id as 4 little-endian bytes, then the extra
    key as 8 little-endian bytes."""
    msg = bytes(parent) + b"".join(struct.pack("<I", int(t) & 0xFFFFFFFF) for t in tokens)
    msg += struct.pack("<Q", int(extra_key) & 0xFFFFFFFFFFFFFFFF)
    return hashlib.sha256(msg).digest()


def chain_keys(tokens: Sequence[int], block_size: int, extra_key: int = 0) -> List[bytes]:
    """Keys of every full block of ``tokens``, in order."""
    keys, parent = [], ROOT_KEY
    for i in range(len(tokens) // block_size):
        parent = block_key(parent, tokens[i * block_size:(i + 1) * block_size], extra_key)
        keys.append(parent)
    return keys


class _Seq:
    def __init__(self, extra_key: int):
        self.extra_key = extra_key
        self.table: List[int] = []
        self.keys: List[bytes] = []       # keys of the full blocks, in order
        self.tail: List[int] = []         # tokens of the partly filled last block
        self.len = 0


class PrefixCache:
    def __init__(self, num_blocks: int, block_size: int,
                 free_order: Optional[Iterable[int]] = None):
        self.num_blocks = int(num_blocks)
        self.block_size = int(block_size)
        order = list(range(num_blocks)) if free_order is None else [int(b) for b in free_order]
        assert sorted(order) == list(range(num_blocks)), "free order must be a permutation"
        self.free: List[int] = order            # front = next to allocate / evict
        self.refcount: List[int] = [0] * self.num_blocks
        self.block_hash: List[Optional[bytes]] = [None] * self.num_blocks
        self.cache: Dict[bytes, int] = {}
        self.seqs: Dict[int, _Seq] = {}

    # -- pool -------------------------------------------------------------------
    def _allocate(self) -> int:
        if not self.free:
            raise OutOfBlocks("no free block left")
        b = self.free.pop(0)
        h = self.block_hash[b]
        if h is not None:                       # evict its cached content
            if self.cache.get(h) == b:
                del self.cache[h]
            self.block_hash[b] = None
        assert self.refcount[b] == 0
        self.refcount[b] = 1
        return b

    def _release(self, b: int) -> None:
        assert self.refcount[b] > 0
        self.refcount[b] -= 1
        if self.refcount[b] == 0:
            self.free.append(b)

    # -- requests -----------------------------------------------------------------
    def add_sequence(self, seq: int, prompt: Sequence[int], extra_key: int = 0) -> int:
        """Start a request: take over the cached blocks of the prompt's longest
        cached prefix.  Returns the number of prompt tokens that need no
        prefill (a multiple of block_size, at most len(prompt) - 1)."""
        assert seq not in self.seqs
        s = _Seq(extra_key)
        B = self.block_size
        usable = max(0, len(prompt) - 1) // B     # the last token is always recomputed
        parent = ROOT_KEY
        for i in range(usable):
            key = block_key(parent, prompt[i * B:(i + 1) * B], extra_key)
            b = self.cache.get(key)
            if b is None:
                break
            if self.refcount[b] == 0:
                self.free.remove(b)
            self.refcount[b] += 1
            s.table.append(b)
            s.keys.append(key)
            parent = key
        s.len = len(s.table) * B
        self.seqs[seq] = s
        return s.len

    def append(self, seq: int, tokens: Sequence[int]) -> List[int]:
        """Reserve slots for ``tokens`` (the sequence's next tokens, in order);
        each block that becomes full is keyed and, when its key is not cached
        yet, entered in the cache.  Reading: when the key is already cached
        (the same content filled twice), the existing block stays the cached
        one and the new block stays uncached."""
        s = self.seqs[seq]
        B = self.block_size
        need = sum(1 for i in range(len(tokens)) if (s.len + i) % B == 0)
        if need > len(self.free):
            raise OutOfBlocks("not enough free blocks")
        slots = []
        for t in tokens:
            off = s.len % B
            if off == 0:
                s.table.append(self._allocate())
            blk = s.table[-1]
            slots.append(blk * B + off)
            s.tail.append(int(t))
            s.len += 1
            if len(s.tail) == B:
                parent = s.keys[-1] if s.keys else ROOT_KEY
                key = block_key(parent, s.tail, s.extra_key)
                s.keys.append(key)
                s.tail = []
                if key not in self.cache:
                    self.cache[key] = blk
                    self.block_hash[blk] = key
        return slots

    def free_sequence(self, seq: int) -> None:
        """Release a finished request's blocks.  Reading: last block first, so
        that eviction from the front of the queue drops the deepest blocks of a
        chain before the ones every longer hit also needs."""
        s = self.seqs.pop(seq)
        for b in reversed(s.table):
            self._release(b)

    # -- inspection -----------------------------------------------------------------
    def table(self, seq: int) -> Tuple[List[int], int]:
        s = self.seqs[seq]
        return list(s.table), s.len

    def check_invariants(self) -> None:
        refs = [0] * self.num_blocks
        for s in self.seqs.values():
            for b in s.table:
                refs[b] += 1
        assert refs == self.refcount
        assert sorted(self.free) == [b for b in range(self.num_blocks) if refs[b] == 0]
        for key, b in self.cache.items():
            assert self.block_hash[b] == key
        assert sum(h is not None for h in self.block_hash) == len(self.cache)
