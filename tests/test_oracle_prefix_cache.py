"""The prefix-cache oracle against what the pages state ("PagedAttention and
vLLM: Paging the KV Cache Like an OS" ..., section 2.4 and summary point 5),
a brute-force prefix matcher on histories without eviction, invariants, and
planted mistakes that these checks must catch."""
import random

import pytest

import oracle.prefix_cache as pcm
from oracle.prefix_cache import PrefixCache


def _fill(pc, seq, prompt, extra=0):
    """A request as a serving loop runs it: look up, then prefill the rest."""
    cached = pc.add_sequence(seq, prompt, extra)
    pc.append(seq, prompt[cached:])
    return cached


# ---- the pages' statements ---------------------------------------------------

def check_full_hit_recomputes_last_token():
    pc = PrefixCache(32, 4)
    prompt = list(range(100, 116))                 # 4 full blocks
    assert _fill(pc, 1, prompt) == 0
    assert _fill(pc, 2, prompt) == 12              # 3 blocks: token 15 is recomputed
    longer = prompt + [7]
    assert _fill(pc, 3, longer) == 16              # 4 blocks, token 16 recomputed


def check_one_token_breaks_the_chain():
    pc = PrefixCache(64, 4)
    base = list(range(1, 25))                      # 6 blocks
    _fill(pc, 1, base)
    first = [999] + base[1:]
    assert _fill(pc, 2, first) == 0               # token 0 differs: no block hits
    mid = base[:9] + [999] + base[10:]             # token 9 is in block 2
    assert _fill(pc, 3, mid) == 8                  # blocks 0 and 1 only


def check_same_block_after_different_prefix():
    pc = PrefixCache(64, 4)
    a = [1, 2, 3, 4, 5, 6, 7, 8, 0]
    b = [9, 9, 9, 9, 5, 6, 7, 8, 0]                # block 1 equal, block 0 not
    _fill(pc, 1, a)
    assert _fill(pc, 2, b) == 0
    ka = pcm.chain_keys(a, 4)
    kb = pcm.chain_keys(b, 4)
    assert ka[1] != kb[1]                          # the parent salts the key


def check_extra_key_separates():
    pc = PrefixCache(64, 4)
    p = list(range(30, 47))
    _fill(pc, 1, p, extra=5)
    assert _fill(pc, 2, p, extra=6) == 0
    assert _fill(pc, 3, p, extra=5) == 16


def check_lru_eviction_order():
    # 8 blocks of 4.  A fills 3 blocks and finishes: its blocks go to the back
    # of the free queue last-first, so the deepest is evicted first.
    pc = PrefixCache(8, 4)
    a = list(range(1, 13))
    _fill(pc, 1, a)
    t, _ = pc.table(1)
    pc.free_sequence(1)
    assert pc.free[-3:] == t[::-1]
    _fill(pc, 2, list(range(50, 74)))              # 6 blocks: the 5 never-cached ones, then A's last
    assert t[2] in pc.table(2)[0] and len(pc.cache) == 2 + 6   # A keeps 2, request 2 adds 6
    pc.free_sequence(2)
    assert _fill(pc, 3, a + [0]) == 8              # A's first two blocks still hit


def check_hit_leaves_free_queue_and_shares():
    pc = PrefixCache(16, 4)
    p = list(range(1, 10))
    _fill(pc, 1, p)
    t1, _ = pc.table(1)
    pc.free_sequence(1)
    assert all(b in pc.free for b in t1)
    assert _fill(pc, 2, p) == 8
    assert _fill(pc, 3, p) == 8
    for b in t1[:2]:
        assert b not in pc.free and pc.refcount[b] == 2
    pc.free_sequence(2)
    assert all(pc.refcount[b] == 1 for b in t1[:2])


def check_no_write_into_shared_blocks():
    pc = PrefixCache(64, 4)
    rnd = random.Random(3)
    system = [rnd.randrange(1000) for _ in range(10)]
    for seq in range(6):
        prompt = system + [rnd.randrange(1000) for _ in range(rnd.randrange(1, 9))]
        cached = pc.add_sequence(seq, prompt)
        slots = pc.append(seq, prompt[cached:])
        slots += pc.append(seq, [rnd.randrange(1000) for _ in range(5)])
        for sl in slots:
            assert pc.refcount[sl // 4] == 1
        pc.check_invariants()


def check_against_brute_force_prefix_matching():
    # no eviction (a large pool): a request's hits are the longest prefix, in
    # whole blocks inside its first len - 1 tokens, that equals the start of a
    # token stream filled earlier under the same extra key
    rnd = random.Random(11)
    B = 4
    pc = PrefixCache(4096, B)
    history = []                                   # (extra key, tokens filled)
    roots = [[rnd.randrange(50) for _ in range(rnd.randrange(4, 30))] for _ in range(5)]
    for seq in range(120):
        extra = rnd.randrange(2)
        base = roots[rnd.randrange(len(roots))]
        cut = rnd.randrange(len(base) + 1)
        prompt = base[:cut] + [rnd.randrange(50) for _ in range(rnd.randrange(1, 12))]
        expect = 0
        for k in range((len(prompt) - 1) // B, 0, -1):
            if any(e == extra and len(h) >= k * B and h[:k * B] == prompt[:k * B]
                   for e, h in history):
                expect = k * B
                break
        cached = pc.add_sequence(seq, prompt, extra)
        assert cached == expect, (seq, cached, expect)
        pc.append(seq, prompt[cached:])
        gen = [rnd.randrange(50) for _ in range(rnd.randrange(0, 9))]
        pc.append(seq, gen)
        history.append((extra, prompt + gen))
        if rnd.random() < 0.5:
            pc.free_sequence(seq)
        pc.check_invariants()


CHECKS = [check_full_hit_recomputes_last_token, check_one_token_breaks_the_chain,
          check_same_block_after_different_prefix, check_extra_key_separates,
          check_lru_eviction_order, check_hit_leaves_free_queue_and_shares,
          check_no_write_into_shared_blocks, check_against_brute_force_prefix_matching]


@pytest.mark.parametrize("check", CHECKS, ids=lambda f: f.__name__)
def test_prefix_cache_check(check):
    check()


def test_out_of_blocks_is_refused():
    pc = PrefixCache(2, 4)
    pc.add_sequence(0, [1, 2, 3])
    with pytest.raises(pcm.OutOfBlocks):
        pc.append(0, list(range(9)))


# ---- planted mistakes ------------------------------------------------------------

_orig_key = pcm.block_key
_orig_free = PrefixCache.free_sequence
_orig_alloc = PrefixCache._allocate
_orig_add = PrefixCache.add_sequence


def _key_unchained(parent, tokens, extra_key):
    return _orig_key(pcm.ROOT_KEY, tokens, extra_key)


def _key_no_extra(parent, tokens, extra_key):
    return _orig_key(parent, tokens, 0)


def _free_in_order(self, seq):
    s = self.seqs.pop(seq)
    for b in s.table:
        self._release(b)


def _alloc_keeps_cache(self):
    b = self.free.pop(0)
    self.refcount[b] = 1
    return b


def _add_full_hit(self, seq, prompt, extra_key=0):
    # hits allowed to cover the whole prompt
    return _orig_add(self, seq, list(prompt) + [0], extra_key)


MUTANTS = {
    "key not chained": ("block_key", pcm, _key_unchained),
    "extra key ignored": ("block_key", pcm, _key_no_extra),
    "blocks freed first-first": ("free_sequence", PrefixCache, _free_in_order),
    "eviction keeps the cache entry": ("_allocate", PrefixCache, _alloc_keeps_cache),
    "full hit without recompute": ("add_sequence", PrefixCache, _add_full_hit),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_checks_catch_mutant(name, monkeypatch):
    attr, owner, fn = MUTANTS[name]
    monkeypatch.setattr(owner, attr, fn)
    caught = []
    for check in CHECKS:
        try:
            check()
        except (AssertionError, KeyError, ValueError, IndexError, pcm.OutOfBlocks):
            caught.append(check.__name__)
    assert caught, f"no check caught: {name}"
