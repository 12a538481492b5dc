"""paged_attention_decode_append -- the decode step's KV write and decode
attention in one call -- against the fp64 oracle doing the two steps the
pages describe one after the other (write this step's key/value at the slot
of position L - 1, then attend over all L positions): pools bit-exact,
outputs within 2e-3 (fp32 out) or max(2e-3, 1 ulp) (16-bit out)."""
import pytest
import torch

from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh
from tests.test_gpu_parity import ATOL, SMALL, _custom, _flags, _sample_seqs, run_full_compare

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as pkv
    pkv.load()
    pkv.read_device_flags(clear=True)
    yield


@pytest.mark.parametrize("name", list(SMALL))
def test_workloads_small(name):
    err, plan = run_full_compare(SMALL[name], append=True)
    if name == "shared":
        assert len(plan.step_pairs) == 16


@pytest.mark.parametrize("pt", [0, 4, 8, 16])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_tiny_partitions_and_out_dtypes(pt, out_dtype):
    run_full_compare(wl.TINY, out_dtype=out_dtype, partition_tokens=pt, append=True)


@pytest.mark.parametrize("pt", [0, 512])
def test_boundary_lengths(pt):
    # 0 (nothing appended), 1 (the new token is the whole context), block
    # edges, partition edges
    lens = [0, 1, 15, 16, 17, 511, 512, 513, 1024, 1025, 2047]
    run_full_compare(_custom("edges", lens, 8, 2, 128, 16, pt=pt), width=130, append=True)


@pytest.mark.parametrize("hq,hkv", [(3, 1), (12, 2), (16, 1), (24, 2), (8, 8), (40, 2), (64, 2)])
def test_group_sizes(hq, hkv):
    # groups above 16 heads run as several head chunks per KV head: each
    # substitutes the new row, only the first stores it
    run_full_compare(_custom("groups", [3, 40, 129, 300], hq, hkv, 64, 8, pt=64), append=True)


@pytest.mark.parametrize("b", [4, 8, 16, 32])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_block_sizes_dims_dtypes(b, d, dtype):
    w = _custom("shapes", [1, b - 1, b, 3 * b + 1, 700], 8, 2, d, b, dtype=dtype, pt=8 * b)
    run_full_compare(w, append=True)


def test_stale_new_slot_is_never_read():
    # the new slot holds NaN before the step and the tail slots NaN / Inf
    w = _custom("poison", [5, 21, 34, 7, 16, 33], 4, 2, 128, 16, pt=16)
    run_full_compare(w, poison_tail=True, poison_new_slot=True, append=True)


def test_same_as_separate_write_and_decode():
    """Bit-identical pools and outputs whether the step runs as two calls or
    as one (the attention arithmetic is the same)."""
    w = SMALL["llama8b"]
    plan = gh.plan_step(w)
    k, v = wl.make_pool(w, "cuda")
    q, key, value = wl.make_step_inputs(w, "cuda")
    k2, v2 = k.clone(), v.clone()
    o1 = gh.run_gpu_step(plan, k, v, q, key, value)
    o2 = gh.run_gpu_step(plan, k2, v2, q, key, value, append=True)
    torch.cuda.synchronize()
    assert _flags() == 0
    assert torch.equal(k, k2) and torch.equal(v, v2)
    assert torch.equal(o1, o2)


@pytest.mark.parametrize("name", ["llama8b", "qwen72b", "shared"])
def test_full_size_sampled(name):
    w = wl.WORKLOADS[name]
    width = {"llama8b": 8192 // 16, "qwen72b": 8192 // 16, "shared": 2048 // 16}[name]
    plan = gh.plan_step(w, width=width)
    k, v = wl.make_pool_chunked(w, "cuda")
    q, key, value = wl.make_step_inputs(w, "cuda")
    seqs = _sample_seqs(plan)
    ids = gh.needed_blocks(plan, seqs)
    idx = torch.tensor(ids, device="cuda")
    kb, vb = k[idx].cpu(), v[idx].cpu()
    ref = gh.oracle_step(plan, kb, vb, ids, q.cpu(), key.cpu(), value.cpu(), seqs)
    out = gh.run_gpu_step(plan, k, v, q, key, value, torch.float32, append=True)
    torch.cuda.synchronize()
    assert _flags() == 0
    gh.assert_close_to_oracle(out[seqs], ref.out, ATOL)
    assert torch.equal(k[idx].cpu(), ref.k_blocks)
    assert torch.equal(v[idx].cpu(), ref.v_blocks)
    # every sequence's new row landed in its slot
    B = w.block_size
    slots = torch.tensor(plan.slots, device="cuda")
    live = slots >= 0
    assert torch.equal(k.view(-1, w.num_kv_heads, w.head_dim)[slots[live]], key[live])
    assert torch.equal(v.view(-1, w.num_kv_heads, w.head_dim)[slots[live]], value[live])
    assert torch.isfinite(out).all()


def test_graph_captured_steps_match_oracle():
    """Three decode steps (copy -> append) captured once in a CUDA graph and
    replayed with new inputs copied into the captured buffers: the pool and
    every output match the oracle run step by step."""
    import oracle.paged_ops as ops
    import paged_kv_cache_117_gb300 as pkv
    from oracle.block_manager import BlockManager
    w = _custom("graph", [7, 16, 40, 1, 95], 8, 2, 128, 16, pt=32)
    S, B = w.num_seqs, w.block_size
    bm = BlockManager(w.num_blocks, B, wl.free_block_order(w))
    for s, L in enumerate(w.lens_args):
        bm.add_sequence(s)
        bm.append_tokens(s, L)
    k, v = wl.make_pool(w, "cpu")
    kd, vd = k.cuda(), v.cuda()
    width = 16
    tab = torch.zeros((S, width), dtype=torch.int32, device="cuda")
    lens = torch.zeros(S, dtype=torch.int32, device="cuda")
    q = torch.zeros((S, w.num_q_heads, w.head_dim), dtype=w.dtype, device="cuda")
    key = torch.zeros((S, w.num_kv_heads, w.head_dim), dtype=w.dtype, device="cuda")
    val = torch.zeros_like(key)
    out = torch.zeros((S, w.num_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    ws = torch.empty(pkv.paged_attention_workspace_bytes(S, w.num_q_heads, w.head_dim,
                                                         width * B, 32),
                     dtype=torch.uint8, device="cuda")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        pkv.paged_attention_decode_append(out, q, key, val, kd, vd, tab, lens, w.scale,
                                          partition_tokens=32, workspace=ws)
    gen = torch.Generator().manual_seed(77)
    for step in range(3):
        slots = [bm.append(s)[0] for s in range(S)]   # no sharing here: no copies
        tables = [list(bm.tables[s]) for s in range(S)]
        Ls = [bm.lens[s] for s in range(S)]
        qc = torch.randn((S, w.num_q_heads, w.head_dim), generator=gen).to(w.dtype)
        kc = torch.randn((S, w.num_kv_heads, w.head_dim), generator=gen).to(w.dtype)
        vc = torch.randn((S, w.num_kv_heads, w.head_dim), generator=gen).to(w.dtype)
        ops.write_kv(k, v, kc, vc, slots)
        ref = ops.attend(qc, k, v, tables, Ls, w.scale)
        tab.copy_(wl.pad_tables(tables, width))
        lens.copy_(torch.tensor(Ls, dtype=torch.int32))
        q.copy_(qc)
        key.copy_(kc)
        val.copy_(vc)
        g.replay()
        torch.cuda.synchronize()
        assert _flags() == 0
        assert torch.equal(kd.cpu(), k) and torch.equal(vd.cpu(), v)
        gh.assert_close_to_oracle(out, ref, ATOL)


def test_bad_metadata_is_flagged_and_nothing_stored():
    import paged_kv_cache_117_gb300 as pkv
    B, H, D, N = 16, 2, 64, 32
    k = torch.randn((N, B, H, D), device="cuda").to(torch.bfloat16)
    v = torch.randn((N, B, H, D), device="cuda").to(torch.bfloat16)
    k0, v0 = k.clone(), v.clone()
    q = torch.randn((3, 4, D), device="cuda").to(torch.bfloat16)
    key = torch.randn((3, H, D), device="cuda").to(torch.bfloat16)
    val = torch.randn((3, H, D), device="cuda").to(torch.bfloat16)
    # seq 0: the new token's block id is outside the pool; seq 1: a length
    # past the table (clamped, nothing appended); seq 2: nothing this step
    tables = torch.tensor([[1, 2, N + 5], [3, 4, 5], [6, 7, 8]], dtype=torch.int32,
                          device="cuda")
    lens = torch.tensor([40, 10_000, 0], dtype=torch.int32, device="cuda")
    out = torch.empty((3, 4, D), dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode_append(out, q, key, val, k, v, tables, lens, 0.125,
                                      partition_tokens=16)
    torch.cuda.synchronize()
    f = _flags()
    assert f & pkv.FLAG_BLOCK_RANGE and f & pkv.FLAG_LEN_RANGE
    assert torch.isfinite(out).all()
    assert torch.equal(k, k0) and torch.equal(v, v0)
    assert torch.equal(out[2], torch.zeros_like(out[2]))
