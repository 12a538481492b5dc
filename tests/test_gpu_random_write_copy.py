"""Seeded random sweep of the pool-maintenance calls against the oracle.

paged_kv_write: random pool shapes (block size, KV heads, head_dim, dtype),
token counts from 0 up, distinct slots in random order with skipped
(negative) and out-of-pool slots mixed in.  paged_block_copy and
paged_block_copy_ws: random pair lists with the cases the block manager
never makes mixed in (a dst named twice, a dst that is another pair's src,
self copies, shared sources, blocks outside the pool).

Which pairs are copied follows the calls' stated contract, written out here
on the host: a pair naming a block outside the pool is skipped; among the
others, a pair whose dst is another in-pool pair's dst or src is skipped.
The pairs left never touch each other's blocks, so the oracle copies them in
list order.  Both checks (scan and counters) must give the same pool and the
same flags, and the whole pool is compared bit-exactly.
"""
import random

import pytest
import torch

import oracle.paged_ops as ops
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu
DTYPES = (torch.bfloat16, torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as pkv
    pkv.load()
    pkv.read_device_flags(clear=True)
    yield


def _pool(rnd, gen):
    N = rnd.randint(8, 300)
    B = rnd.choice((4, 8, 16, 32))
    H = rnd.choice((1, 2, 4, 8))
    D = rnd.choice((64, 128))
    dtype = rnd.choice(DTYPES)
    k = torch.randn((N, B, H, D), generator=gen).to(dtype)
    v = torch.randn((N, B, H, D), generator=gen).to(dtype)
    return k, v


def _same_bits(a, b):
    return torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("seed", range(32))
def test_write_random(seed):
    import paged_kv_cache_117_gb300 as pkv
    rnd = random.Random(5000 + seed)
    gen = torch.Generator().manual_seed(6000 + seed)
    k, v = _pool(rnd, gen)
    N, B, H, D = k.shape
    r = rnd.random()
    T = 0 if r < 0.1 else (1 if r < 0.2 else rnd.randint(2, min(700, N * B)))
    slots = rnd.sample(range(N * B), T)
    out_of_pool = False
    for t in range(T):
        r = rnd.random()
        if r < 0.08:
            slots[t] = rnd.choice((-1, -2, -(N * B), -(1 << 40)))   # skipped
        elif r < 0.12:
            slots[t] = N * B + rnd.choice((0, 1, 17, 1 << 33))      # skipped, flagged
            out_of_pool = True
    key = torch.randn((T, H, D), generator=gen).to(k.dtype)
    val = torch.randn((T, H, D), generator=gen).to(k.dtype)
    kr, vr = k.clone(), v.clone()
    ops.write_kv(kr, vr, key, val, [s if s < N * B else -1 for s in slots])
    kd, vd = k.cuda(), v.cuda()
    pkv.paged_kv_write(key.cuda(), val.cuda(), kd, vd,
                       torch.tensor(slots, dtype=torch.int64).reshape(T).cuda())
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == (pkv.FLAG_SLOT_RANGE if out_of_pool else 0)
    assert _same_bits(kd.cpu(), kr) and _same_bits(vd.cpu(), vr)


def _random_pairs(rnd, N):
    r = rnd.random()
    P = 0 if r < 0.1 else (1 if r < 0.2 else rnd.randint(2, min(200, N // 2)))
    perm = list(range(N))
    rnd.shuffle(perm)
    pairs = []
    for i in range(P):
        src, dst = perm[i], perm[N // 2 + i]          # disjoint halves: no clash
        r = rnd.random()
        if pairs and r < 0.06:
            dst = rnd.choice(pairs)[1]                 # a dst named twice
        elif pairs and r < 0.12:
            dst = rnd.choice(pairs)[0]                 # a dst that is a src
        elif pairs and r < 0.18:
            src = rnd.choice(pairs)[0]                 # a shared source (allowed)
        elif r < 0.22:
            dst = src                                  # a self copy
        elif r < 0.27:
            if rnd.random() < 0.5:
                src = rnd.choice((-1, N, N + 5, 1 << 40))
            else:
                dst = rnd.choice((-3, N, N + 1))
        pairs.append((src, dst))
    return pairs


def _expected(pairs, N):
    """(pairs copied, flags) under the calls' contract."""
    inpool = [0 <= s < N and 0 <= d < N for s, d in pairs]
    clean, conflict = [], False
    for p, (s, d) in enumerate(pairs):
        if not inpool[p]:
            continue
        clash = any(inpool[i] and i != p and (pairs[i][0] == d or pairs[i][1] == d)
                    for i in range(len(pairs)))
        if clash:
            conflict = True
        else:
            clean.append((s, d))
    import paged_kv_cache_117_gb300 as pkv
    flags = (pkv.FLAG_PAIR_RANGE if not all(inpool) else 0) | \
            (pkv.FLAG_PAIR_CONFLICT if conflict else 0)
    return clean, flags


@pytest.mark.parametrize("seed", range(32))
def test_copy_random(seed):
    import paged_kv_cache_117_gb300 as pkv
    rnd = random.Random(7000 + seed)
    gen = torch.Generator().manual_seed(8000 + seed)
    k, v = _pool(rnd, gen)
    N = k.shape[0]
    pairs = _random_pairs(rnd, N)
    clean, flags = _expected(pairs, N)
    kr, vr = k.clone(), v.clone()
    ops.copy_blocks(kr, vr, clean)
    pt = gh.pairs_tensor(pairs).cuda()
    for with_ws in (False, True):
        kd, vd = k.cuda(), v.cuda()
        ws = pkv.block_copy_workspace(kd) if with_ws else None
        pkv.paged_block_copy(kd, vd, pt, workspace=ws)
        torch.cuda.synchronize()
        assert pkv.read_device_flags(clear=True) == flags, (with_ws, pairs)
        assert _same_bits(kd.cpu(), kr) and _same_bits(vd.cpu(), vr), with_ws
        if with_ws:
            assert int(ws.count_nonzero()) == 0


def test_out_of_pool_pair_blocks_nothing():
    """A pair outside the pool copies nothing, so a pair whose dst it names
    is still copied: (5, 7) with (7, 99) on a 64-block pool copies block 5
    to 7 (and flags the range), in both checks."""
    import paged_kv_cache_117_gb300 as pkv
    gen = torch.Generator().manual_seed(13)
    k = torch.randn((64, 16, 2, 64), generator=gen).to(torch.bfloat16)
    v = torch.randn((64, 16, 2, 64), generator=gen).to(torch.bfloat16)
    pairs = [(5, 7), (7, 99), (-1, 9), (9, 11)]
    kr, vr = k.clone(), v.clone()
    ops.copy_blocks(kr, vr, [(5, 7), (9, 11)])
    for with_ws in (False, True):
        kd, vd = k.cuda(), v.cuda()
        ws = pkv.block_copy_workspace(kd) if with_ws else None
        pkv.paged_block_copy(kd, vd, gh.pairs_tensor(pairs).cuda(), workspace=ws)
        torch.cuda.synchronize()
        assert pkv.read_device_flags(clear=True) == pkv.FLAG_PAIR_RANGE
        assert _same_bits(kd.cpu(), kr) and _same_bits(vd.cpu(), vr)
