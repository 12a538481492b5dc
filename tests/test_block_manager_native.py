"""The library's native block manager (pkv_bm_* through the binding) against
the pages' worked examples and, step by step, against the oracle's manager
(an independent implementation of the same rules)."""
import json
import os
import random

import pytest

import paged_kv_cache_117_gb300 as pkv
from oracle.block_manager import BlockManager as OracleBM
from paged_kv_cache_117_gb300 import build as pbuild

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module", autouse=True)
def _lib():
    pbuild.build()
    pkv.load()


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def test_four_token_blocks():
    g = golden("four_token_blocks.json")
    for case in g["cases"]:
        bm = pkv.BlockManager(64, g["block_size"])
        bm.add_sequence(0)
        bm.append_tokens(0, case["tokens"])
        table, n = bm.table(0)
        assert len(table) == case["blocks"]
        assert len(table) * g["block_size"] - n == case["free_slots_in_last"]


def test_request_a_walkthrough():
    g = golden("request_a_walkthrough.json")
    order = g["free_order_head"] + [b for b in range(64) if b not in g["free_order_head"]]
    bm = pkv.BlockManager(64, g["block_size"], order)
    bm.add_sequence(0)
    bm.append_tokens(0, g["prompt_tokens"])
    assert bm.table(0)[0] == g["after_prefill"]["table"]
    bm.append_tokens(0, g["block_3_full_at_token"] - g["prompt_tokens"])
    assert bm.table(0) == ([7, 1, 3], 48)
    bm.append(0 for _ in range(1))
    assert len(bm.table(0)[0]) == 4
    bm.free_sequence(0)
    assert bm.num_used_blocks() == 0


def test_waste_example_blocks():
    g = golden("waste_example.json")
    bm = pkv.BlockManager(1024, g["paged_block_size"])
    for i, (p, q, f) in enumerate(g["requests_prompt_generated_final"]):
        bm.add_sequence(i)
        bm.append_tokens(i, p + q)
    assert bm.num_used_blocks() == g["paged"]["blocks"]


def test_cow_parallel_sampling():
    g = golden("cow_parallel_sampling.json")
    bm = pkv.BlockManager(1024, g["block_size"])
    bm.add_sequence(0)
    bm.append_tokens(0, g["prompt_tokens"])
    n = g["samples"]
    for i in range(1, n):
        bm.fork(0, i)
    copies = []
    for _ in range(g["generated_per_sample"]):
        slots, pairs = bm.append(range(n))
        copies += pairs.tolist()
    assert bm.num_used_blocks() == g["shared_total_blocks"]
    assert len(copies) == n - 1 and len({src for src, _ in copies}) == 1
    shared = bm.table(0)[0][: g["shared_full_prompt_blocks"]]
    assert all(bm.refcount(b) == n for b in shared)


def test_pool_exercise():
    g = golden("pool_exercise.json")
    bm = pkv.BlockManager(g["pool_blocks"], g["block_size"])
    for i in range(g["short"]["count"]):
        bm.add_sequence(i)
        bm.append_tokens(i, g["short"]["prompt"] + g["short"]["generated"])
    for i in range(1000, 1000 + g["long"]["count"]):
        bm.add_sequence(i)
        bm.append_tokens(i, g["long"]["prompt"])
    assert bm.num_used_blocks() == g["both_total"]
    for i in range(1000, 1000 + g["long"]["count"]):
        bm.append_tokens(i, 100)
    assert bm.num_used_blocks() == g["after_long_generate_100"]


def test_errors():
    with pytest.raises(ValueError):
        pkv.BlockManager(4, 4, [0, 1, 1, 2])           # not a permutation
    bm = pkv.BlockManager(2, 4)
    bm.add_sequence(0)
    with pytest.raises(pkv.PkvError):
        bm.add_sequence(0)
    with pytest.raises(pkv.PkvError):
        bm.fork(7, 8)
    bm.append_tokens(0, 8)
    with pytest.raises(pkv.PkvError) as e:
        bm.append([0])
    assert e.value.status == 9                           # too few free blocks
    assert bm.table(0) == (bm.table(0)[0], 8)            # unchanged


class _noop:
    def __enter__(self):
        return self

    def __exit__(self, *a):
        return False


def _needs(ref, batch):
    """Blocks an append batch takes, counted on a copy of the oracle's state."""
    import copy
    r = copy.deepcopy(ref)
    before = len(r.free)
    try:
        for s in batch:
            r.append(s)
    except Exception:
        return before + 1
    return before - len(r.free)


def test_differential_against_oracle_manager():
    rnd = random.Random(117)
    N, B = 300, 4
    order = rnd.sample(range(N), N)
    ours, ref = pkv.BlockManager(N, B, order), OracleBM(N, B, order)
    live, nxt = [], 0
    for step in range(4000):
        op = rnd.random()
        if op < 0.08 or not live:
            ours.add_sequence(nxt); ref.add_sequence(nxt); live.append(nxt); nxt += 1
        elif op < 0.16:
            p = rnd.choice(live)
            ours.fork(p, nxt); ref.fork(p, nxt); live.append(nxt); nxt += 1
        elif op < 0.22:
            s = rnd.choice(live); live.remove(s)
            ours.free_sequence(s); ref.free_sequence(s)
        else:
            batch = [rnd.choice(live) for _ in range(rnd.randint(1, 6))]
            if len(ref.free) < len(batch):
                with pytest.raises(pkv.PkvError) if _needs(ref, batch) > len(ref.free) else _noop():
                    slots, pairs = ours.append(batch)
                    for s in batch:
                        ref.append(s)
                    continue
                s = live.pop(0); ours.free_sequence(s); ref.free_sequence(s)
                continue
            slots, pairs = ours.append(batch)
            want_slots, want_pairs = [], []
            for s in batch:
                slot, cow = ref.append(s)
                want_slots.append(slot)
                if cow:
                    want_pairs.append(list(cow))
            assert slots.tolist() == want_slots, step
            assert pairs.tolist() == want_pairs, step
        if step % 50 == 0:
            for s in live:
                assert ours.table(s) == (ref.tables[s], ref.lens[s])
            assert ours.num_free() == len(ref.free)
            assert [ours.refcount(b) for b in range(N)] == ref.refcount


def test_bench_shared_step_matches_oracle_plan():
    """The benchmark builds the shared-prefix step with the library's manager;
    the parity tests build it with the oracle's: the two must agree."""
    import bench
    from paged_kv_cache_117_gb300 import workloads as wl
    from tests import gpu_harness as gh
    w = wl.SHARED
    lens, tables, width, slots, pairs, setup = bench.build_shared_step(w)
    plan = gh.plan_step(w)
    assert lens == plan.lens and tables == plan.tables
    assert slots.tolist() == plan.slots
    assert pairs.tolist() == [list(p) for p in plan.step_pairs] and len(plan.step_pairs) == 16
    assert setup == [list(p) for p in plan.setup_pairs]


def test_bench_beam_step_matches_oracle_plan():
    """Beam search: the benchmark's history (library manager) and the parity
    tests' history (oracle manager) agree step by step."""
    import bench
    from paged_kv_cache_117_gb300 import workloads as wl
    from tests import gpu_harness as gh
    w = wl.BEAM
    lens, tables, width, slots, pairs, hist = bench.build_beam_step(w)
    ref = gh.plan_beam(w)
    assert lens == ref.lens and tables == ref.tables and width >= ref.width
    assert len(hist) + 1 == len(ref.steps)
    for (p, s), (rp, rs, _) in zip(hist + [(pairs, slots)], ref.steps):
        assert p.tolist() == [list(x) for x in rp]
        assert s.tolist() == rs
    assert len(ref.steps[-1][0]) > 0              # the measured step copies blocks
    assert sum(len(p) for p, _, _ in ref.steps) > 1000
