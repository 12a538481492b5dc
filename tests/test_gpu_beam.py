"""Beam search on the paged cache: forks, prunes and copy-on-write copies over
many steps (copies and writes of every step run on the GPU), then attention
over the final beams -- all against the oracle.  The pool is compared
bit-exactly after the whole history."""
import pytest
import torch

import oracle.paged_ops as ops
from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("block_size", [4, 16])
def test_beam_history_matches_oracle(block_size):
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as pkv
    w = wl.Workload("beam_small", 16, 8, 2, 128, block_size, 300, torch.bfloat16, 64, 321,
                    "beam", (4, 37, 4, 2, 20))
    h = gh.plan_beam(w)
    total_pairs = sum(len(p) for p, _, _ in h.steps)
    assert total_pairs >= 10                       # the history exercises the copy kernel
    k, v = wl.make_pool(w, "cpu")
    kd, vd = k.cuda(), v.cuda()
    for t, (pairs, slots, order) in enumerate(h.steps):
        key, val = wl.make_rows(w, t, len(order))
        ops.copy_blocks(k, v, pairs)
        ops.write_kv(k, v, key, val, slots)
        pkv.paged_block_copy(kd, vd, gh.pairs_tensor(pairs).cuda())
        pkv.paged_kv_write(key.cuda(), val.cuda(), kd, vd,
                           torch.tensor(slots, dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    assert torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)
    q, _, _ = wl.make_step_inputs(w, "cpu")
    ref = ops.attend(q, k, v, h.tables, h.lens, w.scale)
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(out, q.cuda(), kd, vd, wl.pad_tables(h.tables).cuda(),
                               torch.tensor(h.lens, dtype=torch.int32, device="cuda"), w.scale,
                               partition_tokens=w.partition_tokens)
    torch.cuda.synchronize()
    gh.assert_close_to_oracle(out, ref, 2e-3)


def test_beam_full_size():
    """The benchmark's beam workload at full size (256 beams over 32 prompts,
    20 history steps, 512-token partitions, 128-block table rows): whole pool
    bit-exact after the history and the measured step, attention of sampled
    beams against the oracle."""
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import random
    import paged_kv_cache_117_gb300 as pkv
    w = wl.BEAM
    h = gh.plan_beam(w, width=2048 // w.block_size)
    kd, vd = wl.make_pool_chunked(w, "cuda")
    k, v = kd.cpu(), vd.cpu()
    for t, (pairs, slots, order) in enumerate(h.steps):
        if t + 1 < len(h.steps):
            key, val = wl.make_rows(w, t, len(order), "cuda")
        else:
            _, key, val = wl.make_step_inputs(w, "cuda")
        ops.copy_blocks(k, v, pairs)
        ops.write_kv(k, v, key.cpu(), val.cpu(), slots)
        pkv.paged_block_copy(kd, vd, gh.pairs_tensor(pairs).cuda())
        pkv.paged_kv_write(key, val, kd, vd, torch.tensor(slots, dtype=torch.int64, device="cuda"))
    q, _, _ = wl.make_step_inputs(w, "cuda")
    out = torch.empty(q.shape, dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(out, q, kd, vd, wl.pad_tables(h.tables, h.width).cuda(),
                               torch.tensor(h.lens, dtype=torch.int32, device="cuda"), w.scale,
                               partition_tokens=w.partition_tokens)
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    assert torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)
    seqs = sorted(random.Random(5).sample(range(len(h.lens)), 6))
    ref = ops.attend(q.cpu()[seqs], k, v, [h.tables[s] for s in seqs],
                     [h.lens[s] for s in seqs], w.scale)
    gh.assert_close_to_oracle(out[seqs], ref, 2e-3)
    assert torch.isfinite(out).all()
