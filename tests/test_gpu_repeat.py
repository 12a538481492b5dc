"""Repeated calls of the decode attention on batches whose sequences span many
split-context partitions, so that most units end in the completion counter
and many in the final merge: every repeat must give the same bits as the
first call (the kernel's arithmetic order does not depend on which CTA runs
which unit or which one merges), and the first call must match the fp64
oracle.  A release/acquire mistake in the counter hand-off (a merge reading a
record before it is written) would show up as a repeat that differs."""
import pytest
import torch

from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as pkv
    pkv.load()
    pkv.read_device_flags(clear=True)
    yield


@pytest.mark.parametrize("pt,repeats", [(16, 150), (64, 150), (512, 60)])
def test_many_partitions_repeat_bit_exactly(pt, repeats):
    import paged_kv_cache_117_gb300 as pkv
    # Qwen-shaped groups (8 query heads per KV head); 6 sequences of 1,500 to
    # 4,100 tokens: up to 256 partitions of 16 tokens per sequence
    w = wl.Workload("repeat", 6, 32, 4, 128, 16, 2000, torch.bfloat16, pt, 4242, "fixed",
                    (4100, 1500, 3333, 2049, 4096, 1777))
    plan = gh.plan_step(w)
    k, v = wl.make_pool(w, "cpu")
    q, key, value = wl.make_step_inputs(w, "cpu")
    ref = gh.oracle_step(plan, k, v, list(range(w.num_blocks)), q, key, value, range(w.num_seqs))
    kd, vd = k.cuda(), v.cuda()
    qd, keyd, vald = q.cuda(), key.cuda(), value.cuda()
    # the write once, then the attention call again and again over the same pool
    first = gh.run_gpu_step(plan, kd, vd, qd, keyd, vald, torch.float32, pt)
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    gh.assert_close_to_oracle(first, ref.out, 2e-3)
    tables = gh.table_tensor(plan).cuda()
    lens = torch.tensor(plan.lens, dtype=torch.int32, device="cuda")
    ws = torch.empty(pkv.paged_attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim,
                                                         tables.shape[1] * w.block_size, pt),
                     dtype=torch.uint8, device="cuda")
    outs = [torch.empty_like(first) for _ in range(repeats)]
    for o in outs:
        pkv.paged_attention_decode(o, qd, kd, vd, tables, lens, w.scale, partition_tokens=pt,
                                   workspace=ws)
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    bad = [i for i, o in enumerate(outs) if not torch.equal(o, first)]
    assert not bad, f"{len(bad)} of {repeats} repeats differ (first at {bad[0]})"
