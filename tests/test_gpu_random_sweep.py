"""Seeded random sweep of the attention entry points against the fp64 oracle.

Each case draws its own shapes (KV heads, group size, head_dim, block size,
cache and output dtypes), lengths (empty, one-token and multi-block contexts,
lengths on and beside block and partition edges) and call options
(partition size, the write appended or separate, P format, mixed or chunked
call), so that combinations the hand-written tests do not list are still
checked.  Every case compares the whole pool bit-exactly and every output
element within 2e-3 (fp32 output) or max(2e-3, 1 ulp) of the once-rounded
oracle (16-bit outputs).
"""
import random

import pytest
import torch

import oracle.paged_ops as ops
from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu
ATOL = 2e-3
DTYPES = (torch.bfloat16, torch.float16)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as pkv
    pkv.load()
    pkv.read_device_flags(clear=True)
    yield


def _edge_len(rnd, B, lo, hi):
    """A length in [lo, hi], often on or next to a block edge."""
    r = rnd.random()
    if r < 0.4:
        k = rnd.randint(max(1, lo // B), max(1, hi // B))
        return min(hi, max(lo, k * B + rnd.choice((-1, 0, 1))))
    return rnd.randint(lo, hi)


@pytest.mark.parametrize("seed", range(48))
def test_decode_random(seed):
    """paged_attention_decode(_append) on a random batch."""
    import paged_kv_cache_117_gb300 as pkv
    rnd = random.Random(1000 + seed)
    G = rnd.choice((1, 2, 3, 4, 5, 8, 12, 16, 24))
    Hkv = rnd.choice([h for h in (1, 2, 4, 8) if G * h <= 64])
    D = rnd.choice((64, 128))
    B = rnd.choice((4, 8, 16, 32))
    dtype = rnd.choice(DTYPES)
    S = rnd.randint(1, 7)
    lens = [rnd.choice((1, 2)) if rnd.random() < 0.2 else _edge_len(rnd, B, 1, 2400)
            for _ in range(S)]
    if rnd.random() < 0.3:
        lens[rnd.randrange(S)] = 0   # an idle sequence: zeros out
    N = sum((L + B - 1) // B for L in lens) + rnd.randint(4, 40)
    pt = rnd.choice((0, B, 4 * B, 16 * B, 512 if 512 % B == 0 else 0))
    w = wl.Workload(f"rand{seed}", S, G * Hkv, Hkv, D, B, N, dtype, pt, 2000 + seed,
                    "fixed", tuple(lens))
    out_dtype = rnd.choice((torch.float32, dtype))
    append = rnd.random() < 0.5 and all(L > 0 for L in lens)
    plan = gh.plan_step(w)
    k, v = wl.make_pool(w, "cpu")
    q, key, value = wl.make_step_inputs(w, "cpu")
    ref = gh.oracle_step(plan, k, v, list(range(N)), q, key, value, range(S))
    kd, vd = k.cuda(), v.cuda()
    out = gh.run_gpu_step(plan, kd, vd, q.cuda(), key.cuda(), value.cuda(), out_dtype, pt,
                          append=append)
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    assert torch.equal(kd.cpu(), ref.k_blocks) and torch.equal(vd.cpu(), ref.v_blocks)
    gh.assert_close_to_oracle(out, ref.out, ATOL)


@pytest.mark.parametrize("seed", range(48))
def test_multiquery_random(seed):
    """paged_attention_chunked or paged_attention_mixed on a random batch of
    prompt chunks, decode tokens and idle sequences."""
    import paged_kv_cache_117_gb300 as pkv
    rnd = random.Random(3000 + seed)
    G = rnd.choice((1, 2, 3, 4, 5, 8, 16, 32))
    Hkv = rnd.choice([h for h in (1, 2, 4) if G * h <= 32])
    D = rnd.choice((64, 128))
    B = rnd.choice((8, 16, 32))
    dtype = rnd.choice(DTYPES)
    p_format = rnd.choice(("hilo", "f16"))
    mixed = rnd.random() < 0.5
    S = rnd.randint(1, 5)
    prior, counts = [], []
    for _ in range(S):
        kind = rnd.random()
        if kind < 0.25:
            n = 1                                        # a decode token
        elif kind < 0.35:
            n = 0                                        # idle
        else:
            n = _edge_len(rnd, 128 // G if G <= 128 else 1, 2, 140)   # a chunk, near tile edges
        prior.append(_edge_len(rnd, B, 0, 700) if rnd.random() < 0.8 else 0)
        counts.append(n)
    if sum(counts) == 0:
        counts[0] = 1
    N = sum((c + n + B - 1) // B for c, n in zip(prior, counts)) + rnd.randint(4, 40)
    w = wl.Workload(f"mq{seed}", 0, G * Hkv, Hkv, D, B, N, dtype, 0, 4000 + seed, "fixed", ())
    step = gh.plan_chunked(w, prior, counts, None)
    T = step.query_start[-1]
    k, v = wl.make_pool(w, "cpu")
    gen = torch.Generator().manual_seed(w.seed + 77)
    q = torch.randn((T, w.num_q_heads, w.head_dim), generator=gen).to(dtype)
    key, val = wl.make_rows(w, 0, T)
    kd, vd = k.cuda(), v.cuda()
    ops.write_kv(k, v, key, val, step.slots)
    ref = ops.attend_chunked(q, k, v, step.tables, step.lens, step.query_start, w.scale)
    pkv.paged_kv_write(key.cuda(), val.cuda(), kd, vd,
                       torch.tensor(step.slots, dtype=torch.int64, device="cuda"))
    out_dtype = rnd.choice((torch.float32, dtype))
    out = torch.full((T, w.num_q_heads, D), float("nan"), dtype=out_dtype, device="cuda")
    args = (out, q.cuda(), kd, vd, wl.pad_tables(step.tables, step.width).cuda(),
            torch.tensor(step.lens, dtype=torch.int32, device="cuda"),
            torch.tensor(step.query_start, dtype=torch.int32, device="cuda"), w.scale)
    if mixed:
        pkv.paged_attention_mixed(*args, max_query_len=max(counts), p_format=p_format,
                                  partition_tokens=rnd.choice((0, B, 8 * B)))
    else:
        pkv.paged_attention_chunked(*args, max_query_len=max(counts), p_format=p_format)
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    assert torch.equal(kd.cpu().view(torch.int16), k.view(torch.int16))
    assert torch.equal(vd.cpu().view(torch.int16), v.view(torch.int16))
    gh.assert_close_to_oracle(out, ref, ATOL)
