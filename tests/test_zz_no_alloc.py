"""The allocation-free decode entry point against the regular one.

paged_attention_decode_noalloc serves callers that cannot allocate device
memory for a workspace (a memory manager that owns all device memory, a
plugin with a fixed budget, a loop that must not call cudaMalloc); it uses a
scratch array inside the library instead.  This file calls it through the C
ABI twice in a row, with different queries, and checks each result against
paged_attention_decode with a caller-allocated workspace on the same inputs,
at the tolerance the parity tests use.  It is collected last so that a run
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
    w = wl.scaled(wl.LLAMA8B, 12, num_blocks=1500)
    pt = 64                                   # several partitions per sequence
    plan = gh.plan_step(w)
    k, v = wl.make_pool(w, "cuda")
    q, key, value = wl.make_step_inputs(w, "cuda")
    tables = gh.table_tensor(plan).cuda()
    lens = torch.tensor(plan.lens, dtype=torch.int32, device="cuda")
    assert max(-(-L // pt) for L in plan.lens) > 1
    need = pkv.paged_attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim,
                                               tables.shape[1] * w.block_size, pt)
    assert 0 < need <= pkv.NOALLOC_SCRATCH_BYTES
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    for call in range(2):
        qc = q if call == 0 else torch.randn_like(q, dtype=torch.float32).to(q.dtype)
        ref = torch.empty(q.shape, dtype=torch.float32, device="cuda")
        pkv.paged_attention_decode(ref, qc, k, v, tables, lens, w.scale, partition_tokens=pt,
                                   workspace=ws)
        got = torch.full(q.shape, float("nan"), dtype=torch.float32, device="cuda")
        pkv.paged_attention_decode_noalloc(got, qc, k, v, tables, lens, w.scale,
                                           partition_tokens=pt)
        torch.cuda.synchronize()
        assert torch.isfinite(got).all()
        err = (got - ref).abs().max().item()
        assert err <= ATOL, f"call {call}: max abs diff {err:.3e}"
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
