"""The allocation-free decode entry point against the regular one.

paged_attention_decode_noalloc serves callers that cannot allocate device
memory for a workspace (a memory manager that owns all device memory, a
plugin with a fixed budget, a loop that must not call cudaMalloc); it uses a
scratch array inside the library instead.  This file calls it through the C
ABI several times in a row, with different queries and partition sizes, and
requires each result to equal, bit for bit, paged_attention_decode with a
caller-allocated workspace on the same inputs (the same kernel runs; only the
scratch differs), and to lie within the parity tests' tolerance of the fp64
oracle.  It is collected last so that a run
stopping at the first failure has already run every other test; it also runs
on its own in a fresh process.
"""
import pytest
import torch

from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

ATOL = 2e-3


@pytest.fixture(scope="module")
def pkv():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as m
    m.load()
    return m


def test_noalloc_matches_workspace_entry_point_twice(pkv):
    import oracle.paged_ops as ops
    w = wl.scaled(wl.LLAMA8B, 12, num_blocks=1500)
    plan = gh.plan_step(w)
    k, v = wl.make_pool(w, "cuda")
    q, key, value = wl.make_step_inputs(w, "cuda")
    q2 = torch.randn(q.shape, generator=torch.Generator().manual_seed(5)).to(q.dtype).cuda()
    tables = gh.table_tensor(plan).cuda()
    lens = torch.tensor(plan.lens, dtype=torch.int32, device="cuda")
    # several partitions per sequence; the later calls change the partition
    # size both ways, so a call finds the array holding counters and records
    # of a call with more (then fewer) partitions than its own
    calls = [(q, 64), (q2, 64), (q, 128), (q2, 16)]
    assert max(-(-L // 64) for L in plan.lens) > 1
    want = {}
    for qi, qc in enumerate((q, q2)):
        want[qi] = ops.attend(qc.cpu(), k.cpu(), v.cpu(), plan.tables, plan.lens, w.scale)
    for call, (qc, pt) in enumerate(calls):
        need = pkv.paged_attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim,
                                                   tables.shape[1] * w.block_size, pt)
        assert 0 < need <= pkv.NOALLOC_SCRATCH_BYTES
        ws = torch.empty(need, dtype=torch.uint8, device="cuda")
        ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        pkv.paged_attention_decode(ref, qc, k, v, tables, lens, w.scale, partition_tokens=pt,
                                   workspace=ws)
        got = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        pkv.paged_attention_decode_noalloc(got, qc, k, v, tables, lens, w.scale,
                                           partition_tokens=pt)
        torch.cuda.synchronize()
        # the same kernel on the same inputs, only the scratch differs: the
        # results must be identical bit for bit
        assert torch.equal(got, ref), f"call {call}: differs from the workspace entry point"
        err = (got.double().cpu() - want[0 if qc is q else 1]).abs().max().item()
        assert err <= ATOL, f"call {call}: max abs error {err:.3e} against the fp64 oracle"
    assert pkv.read_device_flags(clear=True) == 0


def test_noalloc_refuses_requests_beyond_its_scratch(pkv):
    # 4096 sequences x 64 heads x 16 partitions of records is far above the
    # fixed scratch: refused before any launch, with the workspace status
    lib = pkv.load()
    big = lib.paged_attention_decode_noalloc(1 << 20, 2, 2 << 20, 3 << 20, 4 << 20, 1, 5 << 20,
                                             512, 6 << 20, 4096, 64, 8, 128, 16, 8192, 0.1, 512,
                                             None)
    assert big == 7
    need = pkv.paged_attention_workspace_bytes(4096, 64, 128, 512 * 16, 512)
    assert need > pkv.NOALLOC_SCRATCH_BYTES
