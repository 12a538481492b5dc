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
