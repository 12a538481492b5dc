"""Plant plausible mistakes in the oracle (on the CPU, by patching the oracle
module) and check that the pins catch every one of them.  A pin set that let
any of these through would not be pinning the oracle."""
import pytest
import torch

import oracle.paged_ops as ops
import oracle.block_manager as bmmod
from tests import oracle_checks as oc
from tests import test_oracle_block_manager as bmt

_orig_attend_one = ops.attend_one
_orig_gather = ops.gather_logical
_orig_attend = ops.attend


def _attend_one_no_scale(q, k, v, scale):
    return _orig_attend_one(q, k, v, 1.0)


def _attend_one_scale_twice(q, k, v, scale):
    return _orig_attend_one(q, k, v, scale * scale)


def _attend_one_swapped_kv(q, k, v, scale):
    return _orig_attend_one(q, v, k, scale)


def _attend_one_wrong_axis(q, keys, values, scale):
    q64 = q.to(torch.float64)
    if keys.shape[0] == 0:
        return torch.zeros_like(q64)
    z = (q64 @ keys.to(torch.float64).T) * scale
    w = torch.exp(z - z.max())
    return (w / w.sum(dim=0, keepdim=True)) @ values.to(torch.float64)


def _gather_one_short(cache, table, length):
    return _orig_gather(cache, table, max(0, length - 1))


def _gather_one_long(cache, table, length):
    B = cache.shape[1]
    cap = sum(1 for _ in table) * B
    return _orig_gather(cache, table, min(cap, length + 1))


def _gather_wrong_offset(cache, table, length):
    B = cache.shape[1]
    rows = [cache[int(table[p // B]), (p + 1) % B] for p in range(length)]
    if not rows:
        return cache.new_zeros((0,) + tuple(cache.shape[2:]))
    return torch.stack(rows)


def _gather_block_major_confusion(cache, table, length):
    """Reads logical block j from table[j] but walks slots as p // B."""
    B = cache.shape[1]
    rows = [cache[int(table[p % max(1, -(-length // B))]), p // max(1, -(-length // B)) % B]
            for p in range(length)]
    if not rows:
        return cache.new_zeros((0,) + tuple(cache.shape[2:]))
    return torch.stack(rows)


def _attend_wrong_gqa(q, k_cache, v_cache, block_tables, context_lens, scale):
    S, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    scale = float(torch.tensor(scale, dtype=torch.float32))
    out = torch.zeros((S, Hq, D), dtype=torch.float64)
    for s in range(S):
        L = int(context_lens[s])
        keys = ops.gather_logical(k_cache, block_tables[s], L)
        vals = ops.gather_logical(v_cache, block_tables[s], L)
        for hq in range(Hq):
            h = hq % Hkv
            out[s, hq] = ops.attend_one(q[s, hq:hq + 1], keys[:, h], vals[:, h], scale)[0]
    return out


def _attend_per_block(q, k_cache, v_cache, block_tables, context_lens, scale):
    S, Hq, D = q.shape
    B, Hkv = k_cache.shape[1], k_cache.shape[2]
    G = Hq // Hkv
    scale = float(torch.tensor(scale, dtype=torch.float32))
    out = torch.zeros((S, Hq, D), dtype=torch.float64)
    for s in range(S):
        L = int(context_lens[s])
        for j in range(-(-L // B)):
            n = min(B, L - j * B)
            blk = int(block_tables[s][j])
            for hq in range(Hq):
                h = hq // G
                out[s, hq] += ops.attend_one(q[s, hq:hq + 1], k_cache[blk, :n, h],
                                             v_cache[blk, :n, h], scale)[0]
    return out


ATTENTION_MUTANTS = {
    "no_scale": ("attend_one", _attend_one_no_scale),
    "scale_twice": ("attend_one", _attend_one_scale_twice),
    "swapped_kv": ("attend_one", _attend_one_swapped_kv),
    "softmax_wrong_axis": ("attend_one", _attend_one_wrong_axis),
    "length_minus_one": ("gather_logical", _gather_one_short),
    "length_plus_one": ("gather_logical", _gather_one_long),
    "wrong_slot_offset": ("gather_logical", _gather_wrong_offset),
    "block_slot_confusion": ("gather_logical", _gather_block_major_confusion),
    "gqa_modulo_map": ("attend", _attend_wrong_gqa),
    "per_block_softmax": ("attend", _attend_per_block),
}


def _run_checks():
    failed = []
    for check in oc.ALL_CHECKS:
        try:
            check()
        except (AssertionError, RuntimeError, IndexError, ValueError) as e:
            failed.append(check.__name__)
    return failed


@pytest.mark.parametrize("name", sorted(ATTENTION_MUTANTS))
def test_attention_mutant_is_caught(name, monkeypatch):
    attr, fn = ATTENTION_MUTANTS[name]
    monkeypatch.setattr(ops, attr, fn)
    failed = _run_checks()
    assert failed, f"mutant {name} passed every attention pin"


def test_unmutated_oracle_passes_all():
    assert _run_checks() == []


# -- block manager mutants ---------------------------------------------------

def _append_no_decrement(self, seq):
    table = self.tables[seq]
    n = self.lens[seq]
    offset = n % self.block_size
    cow = None
    if offset == 0:
        table.append(self._pop_free())
    else:
        last = table[-1]
        if self.refcount[last] > 1:
            fresh = self._pop_free()
            table[-1] = fresh
            cow = (last, fresh)
    slot = table[n // self.block_size] * self.block_size + offset
    self.lens[seq] = n + 1
    return slot, cow


def _append_off_by_one(self, seq):
    table = self.tables[seq]
    n = self.lens[seq]
    if n % self.block_size == 1 or not table:
        table.append(self._pop_free())
    slot = table[-1] * self.block_size + n % self.block_size
    self.lens[seq] = n + 1
    return slot, None


def _append_never_copies(self, seq):
    table = self.tables[seq]
    n = self.lens[seq]
    if n % self.block_size == 0:
        table.append(self._pop_free())
    slot = table[n // self.block_size] * self.block_size + n % self.block_size
    self.lens[seq] = n + 1
    return slot, None


def _pop_lifo(self):
    if not self.free:
        raise bmmod.OutOfBlocks("empty")
    b = self.free.pop()
    self.refcount[b] = 1
    return b


BM_TESTS = [bmt.test_four_token_blocks, bmt.test_token_nine_opens_third_block_and_earlier_entries_stay,
            bmt.test_request_a_walkthrough, bmt.test_waste_example,
            bmt.test_cow_parallel_sampling_arithmetic, bmt.test_shared_block_bytes_never_change_while_shared,
            bmt.test_pool_exercise, bmt.test_random_ops_keep_invariants]

BM_MUTANTS = {
    "cow_keeps_count": ("append", _append_no_decrement),
    "new_block_one_token_late": ("append", _append_off_by_one),
    "write_shared_in_place": ("append", _append_never_copies),
    "free_list_lifo": ("_pop_free", _pop_lifo),
}


@pytest.mark.parametrize("name", sorted(BM_MUTANTS))
def test_block_manager_mutant_is_caught(name, monkeypatch):
    attr, fn = BM_MUTANTS[name]
    monkeypatch.setattr(bmmod.BlockManager, attr, fn)
    failed = []
    for t in BM_TESTS:
        try:
            t()
        except Exception:
            failed.append(t.__name__)
    assert failed, f"mutant {name} passed every block-manager pin"
