"""Prefix caching on the GPU: requests whose prompts start with a system prompt
that an earlier (finished) request prefilled take its cached blocks over
(oracle prefix-cache manager), write only their own tokens, and attend over
the whole prompt with paged_attention_chunked -- compared with the oracle's
attention over the same pool; the pool is compared bit-exactly."""
import random

import pytest
import torch

import oracle.paged_ops as ops
from oracle.prefix_cache import PrefixCache
from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("B", [8, 16])
def test_prefix_hits_then_chunked_attention(B):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as pkv
    w = wl.Workload("prefix_small", 0, 8, 2, 128, B, 400, torch.bfloat16, 0, 600, "fixed", ())
    rnd = random.Random(B)
    pc = PrefixCache(w.num_blocks, B, wl.free_block_order(w))
    k, v = wl.make_pool(w, "cpu")
    kd, vd = k.cuda(), v.cuda()
    step = [0]

    def write(slots):
        key, val = wl.make_rows(w, step[0], len(slots))
        step[0] += 1
        ops.write_kv(k, v, key, val, slots)
        pkv.paged_kv_write(key.cuda(), val.cuda(), kd, vd,
                           torch.tensor(slots, dtype=torch.int64, device="cuda"))

    systems = [[rnd.randrange(1000) for _ in range(n)] for n in (5 * B + 3, 3 * B)]
    for i, sysp in enumerate(systems):          # earlier requests, finished
        sid = 100 + i
        c = pc.add_sequence(sid, sysp + [1])
        write(pc.append(sid, (sysp + [1])[c:]))
        pc.free_sequence(sid)
    prompts = [systems[r % 2] + [rnd.randrange(1000) for _ in range(rnd.randrange(1, 2 * B))]
               for r in range(7)]
    prompts.append([rnd.randrange(1000) for _ in range(3 * B + 1)])   # no hit at all
    counts, slots = [], []
    for r, prompt in enumerate(prompts):
        c = pc.add_sequence(r, prompt)
        assert c == ((len(systems[r % 2]) // B) * B if r < 7 else 0)
        slots += pc.append(r, prompt[c:])
        counts.append(len(prompt) - c)
    write(slots)
    pc.check_invariants()
    tables = [pc.table(r)[0] for r in range(len(prompts))]
    lens = [pc.table(r)[1] for r in range(len(prompts))]
    qs = [0]
    for n in counts:
        qs.append(qs[-1] + n)
    g = torch.Generator().manual_seed(B)
    q = torch.randn((qs[-1], w.num_q_heads, w.head_dim), generator=g).to(w.dtype)
    ref = ops.attend_chunked(q, k, v, tables, lens, qs, w.scale)
    out = torch.empty((qs[-1], w.num_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    pkv.paged_attention_chunked(out, q.cuda(), kd, vd, wl.pad_tables(tables).cuda(),
                                torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                torch.tensor(qs, dtype=torch.int32, device="cuda"), w.scale,
                                max_query_len=max(counts))
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    assert torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)
    gh.assert_close_to_oracle(out, ref, 2e-3)


def test_prefix_workload_full_size_sampled():
    """The benchmark's prefix workload at full size (32 requests over 2 cached
    2,048-token system prompts, 256 own tokens each), metadata from the
    oracle's prefix cache: every request takes 2,048 tokens over; the writes
    are bit-exact on the sampled requests' blocks and sampled rows match the
    oracle (a row at position p is decode attention over positions 0..p)."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as pkv
    w = wl.PREFIX
    plan = wl.prefix_plan(w)
    pc = PrefixCache(w.num_blocks, w.block_size, wl.free_block_order(w))
    kd, vd = wl.make_pool_chunked(w, "cuda")
    k, v = kd.cpu(), vd.cpu()
    step = [0]

    def write(slots):
        key, val = wl.make_rows(w, step[0], len(slots), "cuda")
        step[0] += 1
        ops.write_kv(k, v, key.cpu(), val.cpu(), slots)
        pkv.paged_kv_write(key, val, kd, vd, torch.tensor(slots, dtype=torch.int64, device="cuda"))

    for i, sysp in enumerate(plan.systems):
        sid = len(plan.prompts) + i
        c = pc.add_sequence(sid, sysp + [0])
        write(pc.append(sid, (sysp + [0])[c:]))
        pc.free_sequence(sid)
    counts, slots = [], []
    for r, prompt in enumerate(plan.prompts):
        c = pc.add_sequence(r, prompt)
        assert c == len(plan.systems[0])
        slots += pc.append(r, prompt[c:])
        counts.append(len(prompt) - c)
    write(slots)
    tables = [pc.table(r)[0] for r in range(len(plan.prompts))]
    lens = [pc.table(r)[1] for r in range(len(plan.prompts))]
    qs = [0]
    for n in counts:
        qs.append(qs[-1] + n)
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed + 3000)
    q = torch.randn((qs[-1], w.num_q_heads, w.head_dim), generator=g, device="cuda").to(w.dtype)
    out = torch.empty((qs[-1], w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    pkv.paged_attention_chunked(out, q, kd, vd, wl.pad_tables(tables, 4096 // w.block_size).cuda(),
                                torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                torch.tensor(qs, dtype=torch.int32, device="cuda"), w.scale,
                                max_query_len=max(counts))
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    seqs = [0, 1, 17, 31]
    ids = sorted({b for s in seqs for b in tables[s]})
    idx = torch.tensor(ids, device="cuda")
    assert torch.equal(kd[idx].cpu(), k[ids]) and torch.equal(vd[idx].cpu(), v[ids])
    assert torch.isfinite(out).all()
    qc = q.cpu()
    for s in seqs:
        n, L, r0 = counts[s], lens[s], qs[s]
        for i in (0, 1, 127, n - 1):
            ref = ops.attend(qc[r0 + i:r0 + i + 1], k, v, [tables[s]], [L - n + i + 1], w.scale)
            gh.assert_close_to_oracle(out[r0 + i:r0 + i + 1], ref, 2e-3)
