"""Pins for the oracle's block manager and sizing arithmetic, against the
numbers the pages print (fixtures under tests/golden/, each with its source)."""
import json
import math
import os
import random

import pytest

from oracle.block_manager import BlockManager, OutOfBlocks
from oracle import sizing

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_four_token_blocks():
    g = golden("four_token_blocks.json")
    B = g["block_size"]
    for case in g["cases"]:
        bm = BlockManager(64, B)
        bm.add_sequence(0)
        bm.append_tokens(0, case["tokens"])
        assert len(bm.tables[0]) == case["blocks"], case
        assert len(bm.tables[0]) * B - bm.lens[0] == case["free_slots_in_last"], case
        bm.check_invariants()


def test_token_nine_opens_third_block_and_earlier_entries_stay():
    bm = BlockManager(16, 4, free_order=[3, 0, 6] + [b for b in range(16) if b not in (3, 0, 6)])
    bm.add_sequence(0)
    slots, _ = bm.append_tokens(0, 8)
    assert bm.tables[0] == [3, 0]
    slot9, cow = bm.append(0)
    assert cow is None
    assert bm.tables[0] == [3, 0, 6]           # the table of section 5
    assert slot9 == 6 * 4 + 0
    assert slots == [12, 13, 14, 15, 0, 1, 2, 3]


def test_request_a_walkthrough():
    g = golden("request_a_walkthrough.json")
    B = g["block_size"]
    head = g["free_order_head"]
    order = head + [b for b in range(64) if b not in head]
    bm = BlockManager(64, B, free_order=order)
    bm.add_sequence(0)
    bm.append_tokens(0, g["prompt_tokens"])
    assert bm.tables[0] == g["after_prefill"]["table"]
    assert len(bm.tables[0]) * B - bm.lens[0] == g["after_prefill"]["empty_slots_in_block_3"]
    bm.append_tokens(0, g["decode_steps"])
    assert bm.lens[0] == g["after_decode"]["tokens"]
    assert len(bm.tables[0]) * B - bm.lens[0] == g["after_decode"]["free_slots_in_block_3"]
    while bm.lens[0] < g["block_3_full_at_token"]:
        bm.append(0)
    assert bm.tables[0] == [7, 1, 3]           # block 3 full at token 48, no new block yet
    assert len(bm.tables[0]) * B == bm.lens[0]
    bm.append(0)                               # token 49
    assert len(bm.tables[0]) == 4 and g["token_49_needs_new_block"]
    before = bm.num_used_blocks()
    bm.free_sequence(0)                        # a finished request returns its blocks
    assert bm.num_used_blocks() == before - 4 == 0


def test_waste_example():
    g = golden("waste_example.json")
    reqs = g["requests_prompt_generated_final"]
    c = g["contiguous"]
    reserved = len(reqs) * g["max_len"]
    used = sum(p + q for p, q, f in reqs)
    assert reserved == c["reserved_slots"] and used == c["used_slots"]
    assert sum(f - (p + q) for p, q, f in reqs) == c["later_slots"]
    assert sum(g["max_len"] - f for p, q, f in reqs) == c["never_slots"]
    assert round(used / reserved, 4) == c["utilization_4dp"]
    kib = g["per_token_kib"]
    assert reserved * kib / 1024 == c["reserved_mib"]
    assert used * kib / 1024 == c["used_mib"]
    # the paged layout, driven through the block manager
    B = g["paged_block_size"]
    bm = BlockManager(1024, B)
    for i, (p, q, f) in enumerate(reqs):
        bm.add_sequence(i)
        bm.append_tokens(i, p + q)
    bm.check_invariants()
    blocks = bm.num_used_blocks()
    assert blocks == g["paged"]["blocks"]
    assert blocks == sum(sizing.blocks_for_tokens(p + q, B) for p, q, f in reqs)
    assert round(used / (blocks * B), 4) == g["paged"]["utilization_4dp"]
    assert blocks * B * kib / 1024 == g["paged"]["allocated_mib"]
    assert sizing.max_waste_slots(B) == g["max_waste"]["slots"]
    assert sizing.max_waste_slots(B) * kib == g["max_waste"]["kib"]


def test_unshared_waste_bounded_by_block_minus_one():
    rnd = random.Random(5)
    for B in (1, 4, 8, 16, 32):
        bm = BlockManager(40 * 300, B)
        for s in range(40):
            bm.add_sequence(s)
            bm.append_tokens(s, rnd.randint(1, 300))
            waste = len(bm.tables[s]) * B - bm.lens[s]
            assert 0 <= waste <= B - 1
        bm.check_invariants()


def test_cow_parallel_sampling_arithmetic():
    g = golden("cow_parallel_sampling.json")
    B, P, n, gen = g["block_size"], g["prompt_tokens"], g["samples"], g["generated_per_sample"]
    assert n * sizing.blocks_for_tokens(P + gen, B) == g["unshared_blocks"]
    bm = BlockManager(1024, B)
    bm.add_sequence(0)
    bm.append_tokens(0, P)
    for i in range(1, n):
        bm.fork(0, i)
    full_prompt_blocks = P // B
    assert full_prompt_blocks == g["shared_full_prompt_blocks"]
    shared_prefix = list(bm.tables[0][:full_prompt_blocks])
    cows = []
    for step in range(gen):
        for i in range(n):
            _, cow = bm.append(i)
            if cow:
                cows.append((i, cow))
        bm.check_invariants()
    assert bm.num_used_blocks() == g["shared_total_blocks"]
    assert bm.num_used_blocks() * g["block_mib"] == g["shared_mib"]
    assert round(100 * (1 - g["shared_total_blocks"] / g["unshared_blocks"])) == g["saving_percent_rounded"]
    # the full prompt blocks stay shared by all samples and are never copied
    for i in range(n):
        assert bm.tables[i][:full_prompt_blocks] == shared_prefix
        assert len(bm.tables[i]) - full_prompt_blocks == g["private_blocks_per_sample"]
    for b in shared_prefix:
        assert bm.refcount[b] == n
    # only the partial prompt block is copied: once by every writer that saw
    # a count above one; the last sharer writes in place
    assert [i for i, _ in cows] == list(range(n - 1))
    src = {c[0] for _, c in cows}
    assert len(src) == 1 and src.pop() == bm.tables[n - 1][full_prompt_blocks]


def test_fork_and_free_refcounts():
    bm = BlockManager(32, 4)
    bm.add_sequence(0)
    bm.append_tokens(0, 10)
    bm.fork(0, 1)
    bm.fork(1, 2)
    assert all(bm.refcount[b] == 3 for b in bm.tables[0])
    bm.free_sequence(1)
    assert all(bm.refcount[b] == 2 for b in bm.tables[0])
    bm.free_sequence(0)
    bm.free_sequence(2)
    assert bm.num_used_blocks() == 0
    bm.check_invariants()


def test_shared_block_bytes_never_change_while_shared():
    """A shared block is copied before any write, so a sharer's view never
    changes ("PagedAttention" (tensortonic), section 7)."""
    bm = BlockManager(64, 4)
    bm.add_sequence(0)
    bm.append_tokens(0, 6)
    bm.fork(0, 1)
    shared_last = bm.tables[0][-1]
    slot, cow = bm.append(1)
    assert cow == (shared_last, bm.tables[1][-1])
    assert slot // 4 == bm.tables[1][-1] != shared_last
    slot0, cow0 = bm.append(0)                 # count is back to one: in place
    assert cow0 is None and slot0 // 4 == shared_last


def test_pool_exercise():
    g = golden("pool_exercise.json")
    B = g["block_size"]
    bm = BlockManager(g["pool_blocks"], B)
    for i in range(g["short"]["count"]):
        bm.add_sequence(i)
        bm.append_tokens(i, g["short"]["prompt"] + g["short"]["generated"])
        assert len(bm.tables[i]) == g["short"]["blocks_each"]
    assert bm.num_used_blocks() == g["short"]["blocks_total"]
    longs = range(1000, 1000 + g["long"]["count"])
    for i in longs:
        bm.add_sequence(i)
        bm.append_tokens(i, g["long"]["prompt"])
        assert len(bm.tables[i]) == g["long"]["blocks_each"]
    assert bm.num_used_blocks() == g["both_total"]
    for i in longs:
        bm.append_tokens(i, 100)
    assert bm.num_used_blocks() == g["after_long_generate_100"]
    assert (bm.num_used_blocks() < g["pool_blocks"] / 2) == g["under_half_pool"]
    bm.check_invariants()


def test_out_of_blocks_raises():
    bm = BlockManager(2, 4)
    bm.add_sequence(0)
    bm.append_tokens(0, 8)
    with pytest.raises(OutOfBlocks):
        bm.append(0)


def test_kv_sizing():
    for c in golden("kv_sizing.json")["cases"]:
        bpt = sizing.kv_bytes_per_token(c["layers"], c["kv_heads"], c["head_dim"], c["bytes"])
        assert bpt == c["bytes_per_token"], c["model"]
        if "kb_per_token" in c:
            assert bpt / 1024 == c["kb_per_token"]
        if "request_gb_approx" in c:
            gb = bpt * c["tokens"] / 1e9
            gib = bpt * c["tokens"] / 2 ** 30
            assert abs(gb - c["request_gb_approx"]) < 0.1 or abs(gib - c["request_gb_approx"]) < 0.1
        if "block_bytes" in c:
            bb = sizing.kv_bytes_per_block(c["block_size"], c["layers"], c["kv_heads"],
                                          c["head_dim"], c["bytes"])
            assert bb == c["block_bytes"]
            assert bb // c["layers"] == c["block_bytes_per_layer"]
            blocks = c["free_bytes_h100"] / bb
            assert abs(blocks - c["pool_blocks_approx"]) < 1
            assert abs(math.floor(blocks) * c["block_size"] - c["pool_tokens_approx"]) < 100


def test_random_ops_keep_invariants():
    """Refcount bookkeeping under a random mix of appends, forks and frees."""
    rnd = random.Random(11)
    bm = BlockManager(512, 8, free_order=rnd.sample(range(512), 512))
    live = []
    nxt = 0
    for _ in range(3000):
        op = rnd.random()
        if op < 0.1 or not live:
            bm.add_sequence(nxt); live.append(nxt); nxt += 1
        elif op < 0.2:
            bm.fork(rnd.choice(live), nxt); live.append(nxt); nxt += 1
        elif op < 0.27:
            s = rnd.choice(live); live.remove(s); bm.free_sequence(s)
        else:
            s = rnd.choice(live)
            try:
                bm.append(s)
            except Exception:
                s2 = live.pop(0); bm.free_sequence(s2)
        bm.check_invariants()
