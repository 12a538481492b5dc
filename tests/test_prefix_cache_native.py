"""The library's prefix-cache manager (pkv_pc_*) against the oracle's
(`oracle.prefix_cache`): SHA-256 against Python's hashlib and the FIPS 180
example digests, chained keys against the oracle's, and long random request
streams (shared system prompts, evictions, adapters) compared step by step:
cached-token counts, slots, tables, counts, the free queue's order and every
block's cached key."""
import hashlib
import random

import pytest
import torch

import oracle.prefix_cache as opc
import paged_kv_cache_117_gb300 as pkv
from paged_kv_cache_117_gb300 import build as pbuild


@pytest.fixture(scope="module", autouse=True)
def lib():
    pbuild.build()
    return pkv.load()


def test_sha256_published_examples():
    # FIPS 180-2 appendix B examples
    assert pkv.sha256(b"abc").hex() == \
        "ba7816bf8f01cfea414140de5dae2223b00361a396177a9cb410ff61f20015ad"
    assert pkv.sha256(b"abcdbcdecdefdefgefghfghighijhijkijkljklmklmnlmnomnopnopq").hex() == \
        "248d6a61d20638b8e5c026930c3e6039a33ce45964ff2167f6ecedd419db06c1"
    assert pkv.sha256(b"").hex() == \
        "e3b0c44298fc1c149afbf4c8996fb92427ae41e4649b934ca495991b7852b855"


def test_sha256_matches_hashlib_every_padding_case():
    rnd = random.Random(1)
    for n in list(range(0, 200)) + [447, 448, 511, 512, 513, 4096]:
        msg = bytes(rnd.randrange(256) for _ in range(n))
        assert pkv.sha256(msg) == hashlib.sha256(msg).digest(), n


@pytest.mark.parametrize("B", [1, 4, 16, 32])
def test_chain_keys_match_oracle(B):
    rnd = random.Random(B)
    toks = [rnd.randrange(-5, 1 << 31) for _ in range(5 * B + 3)]
    for extra in (0, 1, (1 << 64) - 1):
        assert pkv.chain_keys(toks, B, extra) == opc.chain_keys(toks, B, extra)


def _same_state(ours, ref):
    assert ours.free_queue() == ref.free
    assert ours.num_free() == len(ref.free)
    assert ours.num_cached() == len(ref.cache)
    for b in range(ref.num_blocks):
        assert ours.refcount(b) == ref.refcount[b]
        assert ours.block_key(b) == ref.block_hash[b]


@pytest.mark.parametrize("seed,B,N", [(0, 4, 64), (1, 16, 48), (2, 8, 200), (3, 1, 40)])
def test_random_request_streams_match_oracle(seed, B, N):
    rnd = random.Random(seed)
    order = list(range(N))
    rnd.shuffle(order)
    ours, ref = pkv.PrefixCache(N, B, order), opc.PrefixCache(N, B, order)
    systems = [[rnd.randrange(100) for _ in range(rnd.randrange(B, 6 * B))] for _ in range(4)]
    live, next_id = [], 0
    for step in range(600):
        op = rnd.random()
        if op < 0.45 or not live:
            sysp = systems[rnd.randrange(len(systems))] if rnd.random() < 0.8 else []
            prompt = sysp + [rnd.randrange(100) for _ in range(rnd.randrange(1, 3 * B))]
            extra = rnd.randrange(2)
            c1 = ours.add_sequence(next_id, prompt, extra)
            c0 = ref.add_sequence(next_id, prompt, extra)
            assert c1 == c0
            try:
                s0 = ref.append(next_id, prompt[c0:])
            except opc.OutOfBlocks:
                with pytest.raises(pkv.PkvError):
                    ours.append(next_id, prompt[c1:])
                ref.free_sequence(next_id)
                ours.free_sequence(next_id)
            else:
                assert ours.append(next_id, prompt[c1:]).tolist() == s0
                live.append(next_id)
            next_id += 1
        elif op < 0.75:
            sq = rnd.choice(live)
            toks = [rnd.randrange(100) for _ in range(rnd.randrange(1, 2 * B))]
            try:
                s0 = ref.append(sq, toks)
            except opc.OutOfBlocks:
                with pytest.raises(pkv.PkvError):
                    ours.append(sq, toks)
            else:
                assert ours.append(sq, toks).tolist() == s0
        else:
            sq = live.pop(rnd.randrange(len(live)))
            ours.free_sequence(sq)
            ref.free_sequence(sq)
        for sq in live[-3:]:
            assert ours.table(sq) == ref.table(sq)
        if step % 25 == 0:
            ref.check_invariants()
            _same_state(ours, ref)
    _same_state(ours, ref)


def test_errors():
    with pytest.raises(ValueError):
        pkv.PrefixCache(4, 4, [0, 1, 1, 2])
    pc = pkv.PrefixCache(2, 4)
    pc.add_sequence(0, [1, 2, 3])
    with pytest.raises(pkv.PkvError):
        pc.add_sequence(0, [1])                     # exists
    with pytest.raises(pkv.PkvError):
        pc.append(0, list(range(9)))                # needs 3 blocks, 2 free
    assert pc.num_free() == 2 and pc.table(0) == ([], 0)   # refused whole
    with pytest.raises(pkv.PkvError):
        pc.free_sequence(7)


@pytest.mark.parametrize("bad", [
    torch.tensor([1, 2, 2**31], dtype=torch.int64),     # would wrap to a negative id
    torch.tensor([1.0, 2.0]),                             # not integers
    torch.tensor([True, False]),
    [1, 2**31],
])
def test_token_ids_that_do_not_fit_int32_are_refused(bad):
    """Token ids reach the C calls as int32: a value that does not fit (or a
    tensor that is not integral) is refused before the call, whether it comes
    as a tensor or a list, instead of being wrapped into another id."""
    pc = pkv.PrefixCache(8, 4)
    with pytest.raises(ValueError):
        pc.add_sequence(0, bad)
    with pytest.raises(ValueError):
        pkv.chain_keys(bad, 1)
    assert pc.num_free() == 8


def test_sequence_ids_that_do_not_fit_int64_are_refused():
    bm = pkv.BlockManager(8, 4)
    bm.add_sequence(0)
    with pytest.raises(ValueError):
        bm.append(torch.tensor([0.0]))
    with pytest.raises(ValueError):
        bm.append([2**63])
    assert bm.num_free() == 8
