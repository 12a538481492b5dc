"""Parity of the CUDA library (through its C ABI) with the fp64 oracle.

Bit-exact for the KV write and the block copy (whole pool compared);
attention within 2e-3 max abs error for fp32 outputs, and within
max(2e-3, 1 ulp) of the once-rounded oracle for 16-bit outputs.
"""
import random

import pytest
import torch

from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu

ATOL = 2e-3


@pytest.fixture(scope="module", autouse=True)
def _lib():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    import paged_kv_cache_117_gb300 as pkv
    pkv.load()
    pkv.read_device_flags(clear=True)
    yield


def _flags():
    import paged_kv_cache_117_gb300 as pkv
    return pkv.read_device_flags(clear=True)


def run_full_compare(w, out_dtype=torch.float32, partition_tokens=None, width=None,
                     poison_tail=False, append=False, poison_new_slot=False):
    """Whole step on both sides; the full pool and every output compared.
    ``append``: the GPU side writes and attends in one call.
    ``poison_new_slot``: each sequence's new slot holds NaN before the step."""
    plan = gh.plan_step(w, width=width)
    k, v = wl.make_pool(w, "cpu")
    if poison_new_slot:
        for slot in plan.slots:
            if slot >= 0:
                k[slot // w.block_size, slot % w.block_size] = float("nan")
                v[slot // w.block_size, slot % w.block_size] = float("nan")
    if poison_tail:
        # unused slots of every last block hold NaN / Inf bit patterns
        for s, t in enumerate(plan.tables):
            L = plan.lens[s]
            if L % w.block_size:
                k[t[-1], L % w.block_size:] = float("nan")
                v[t[-1], L % w.block_size:] = float("inf")
    q, key, value = wl.make_step_inputs(w, "cpu")
    ids = list(range(w.num_blocks))
    ref = gh.oracle_step(plan, k, v, ids, q, key, value, range(w.num_seqs))
    kd, vd = k.cuda(), v.cuda()
    out = gh.run_gpu_step(plan, kd, vd, q.cuda(), key.cuda(), value.cuda(), out_dtype,
                          partition_tokens, append=append)
    torch.cuda.synchronize()
    assert _flags() == 0
    kg, vg = kd.cpu(), vd.cpu()
    if poison_tail:   # NaN != NaN: compare bit patterns
        assert torch.equal(kg.view(torch.int16), ref.k_blocks.view(torch.int16))
        assert torch.equal(vg.view(torch.int16), ref.v_blocks.view(torch.int16))
    else:
        assert torch.equal(kg, ref.k_blocks), "K pool differs from the oracle"
        assert torch.equal(vg, ref.v_blocks), "V pool differs from the oracle"
    return gh.assert_close_to_oracle(out, ref.out, ATOL), plan


# ---- the five workloads at sizes the oracle finishes in seconds -------------

SMALL = {
    "tiny": wl.TINY,
    "opt13b": wl.scaled(wl.OPT13B, 6, num_blocks=1000),
    "llama8b": wl.scaled(wl.LLAMA8B, 12, num_blocks=1500),
    "qwen72b": wl.scaled(wl.QWEN72B, 2, num_blocks=1100),
    "shared": wl.SHARED,
}


@pytest.mark.parametrize("name", list(SMALL))
def test_workload_small_full_compare(name):
    err, plan = run_full_compare(SMALL[name])
    if name == "shared":
        assert len(plan.step_pairs) == 16 and len(plan.setup_pairs) > 0
    if name == "tiny":
        assert plan.lens == [1, 6, 9, 17]


@pytest.mark.parametrize("pt", [0, 4, 8, 16])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16, torch.float16])
def test_tiny_partitions_and_out_dtypes(pt, out_dtype):
    run_full_compare(wl.TINY, out_dtype=out_dtype, partition_tokens=pt)


@pytest.mark.parametrize("pt", [0, 16, 64, 512])
def test_llama_small_partitions(pt):
    run_full_compare(SMALL["llama8b"], partition_tokens=pt)


def _custom(name, lens, hq, hkv, d, b, dtype=torch.bfloat16, pt=512, n=None):
    need = sum(-(-L // b) for L in lens) + 8
    return wl.Workload(name, len(lens), hq, hkv, d, b, n or need, dtype, pt, 500,
                       "fixed", tuple(lens))


@pytest.mark.parametrize("pt", [0, 512])
def test_boundary_lengths(pt):
    lens = [0, 1, 15, 16, 17, 511, 512, 513, 1024, 1025, 2047]
    w = _custom("edges", lens, 8, 2, 128, 16, pt=pt)
    err, plan = run_full_compare(w, width=130)


@pytest.mark.parametrize("hq,hkv", [(3, 1), (12, 2), (16, 1), (24, 2), (5, 5), (8, 8), (32, 4), (40, 2), (64, 2)])
def test_group_sizes(hq, hkv):
    w = _custom("groups", [3, 40, 129, 300], hq, hkv, 64, 8, pt=64)
    run_full_compare(w)


@pytest.mark.parametrize("b", [4, 8, 16, 32])
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_block_sizes_dims_dtypes(b, d, dtype):
    w = _custom("shapes", [1, b - 1, b, 3 * b + 1, 700], 8, 2, d, b, dtype=dtype, pt=8 * b)
    run_full_compare(w)


def test_tail_slots_with_nan_are_never_read():
    w = _custom("poison", [5, 21, 34, 7], 4, 2, 128, 16, pt=16)
    run_full_compare(w, poison_tail=True)


def test_deterministic():
    w = SMALL["llama8b"]
    plan = gh.plan_step(w)
    k, v = wl.make_pool(w, "cuda")
    q, key, value = wl.make_step_inputs(w, "cuda")
    o1 = gh.run_gpu_step(plan, k.clone(), v.clone(), q, key, value)
    o2 = gh.run_gpu_step(plan, k.clone(), v.clone(), q, key, value)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2)


# ---- full sizes, in the launch configuration the benchmark times ------------

def _sample_seqs(plan, count=6, seed=0):
    lens = plan.lens
    order = sorted(range(len(lens)), key=lambda s: lens[s])
    pick = {order[0], order[-1], order[len(order) // 2]}
    rnd = random.Random(seed)
    while len(pick) < min(count, len(lens)):
        pick.add(rnd.randrange(len(lens)))
    return sorted(pick)


@pytest.mark.parametrize("name", ["opt13b", "llama8b", "qwen72b", "shared"])
def test_workload_full_size_sampled(name):
    w = wl.WORKLOADS[name]
    width = {"opt13b": 2048 // 16, "llama8b": 8192 // 16, "qwen72b": 8192 // 16,
             "shared": 2048 // 16}[name]
    plan = gh.plan_step(w, width=width)
    k, v = wl.make_pool_chunked(w, "cuda")
    q, key, value = wl.make_step_inputs(w, "cuda")
    seqs = _sample_seqs(plan)
    ids = gh.needed_blocks(plan, seqs)
    idx = torch.tensor(ids, device="cuda")
    kb, vb = k[idx].cpu(), v[idx].cpu()            # inputs, before any library kernel
    ref = gh.oracle_step(plan, kb, vb, ids, q.cpu(), key.cpu(), value.cpu(), seqs)
    out = gh.run_gpu_step(plan, k, v, q, key, value, torch.float32)
    torch.cuda.synchronize()
    assert _flags() == 0
    gh.assert_close_to_oracle(out[seqs], ref.out, ATOL)
    assert torch.equal(k[idx].cpu(), ref.k_blocks)
    assert torch.equal(v[idx].cpu(), ref.v_blocks)
    # a property that holds for every sequence: each output row is a convex
    # combination of value rows, so it is finite and bounded by max |V|
    assert torch.isfinite(out).all()
    assert out.abs().max().item() <= max(v.abs().max().item(), value.abs().max().item()) + 1e-3
    # bf16 output of the same step equals the rounded fp32 output within 1 ulp
    if name == "llama8b":
        out16 = torch.empty_like(out, dtype=torch.bfloat16)
        import paged_kv_cache_117_gb300 as pkv
        pkv.paged_attention_decode(out16, q, k, v, gh.table_tensor(plan).cuda(),
                                   torch.tensor(plan.lens, dtype=torch.int32, device="cuda"),
                                   w.scale, partition_tokens=w.partition_tokens)
        gh.assert_close_to_oracle(out16[seqs], ref.out, ATOL)


@pytest.mark.parametrize("pt,append", [(512, False), (0, False), (512, True), (128, False)])
def test_longest_contexts_with_needles(pt, append):
    """Contexts far beyond the workloads': 131,072 tokens (256 partitions of
    512, 1,024 of 128 -- more records than the merge stages in shared memory
    -- or a single unit streaming all of it), 65,537 (its new token opens a
    fresh block), one token only, and 4,097.  In KV head 0 one key of each
    long sequence is planted to score ~90 above the rest, deep inside the
    context, so that one far partition dominates the merge."""
    lens = (131072, 65537, 1, 4097)
    nb = sum((L + 15) // 16 for L in lens)
    w = wl.Workload("longest", 4, 32, 8, 128, 16, nb + 64, torch.bfloat16, pt, 126,
                    "fixed", lens)
    plan = gh.plan_step(w)
    k, v = wl.make_pool_chunked(w, "cuda")
    q, key, value = wl.make_step_inputs(w, "cuda")
    for s, pos in ((0, 100_000), (1, 3), (3, 4000)):
        blk = plan.tables[s][pos // w.block_size]
        k[blk, pos % w.block_size, 0] = (q[s, 0].float() * 8).to(w.dtype)
    seqs = list(range(w.num_seqs))
    ids = gh.needed_blocks(plan, seqs)
    idx = torch.tensor(ids, device="cuda")
    kb, vb = k[idx].cpu(), v[idx].cpu()            # inputs, before any library kernel
    ref = gh.oracle_step(plan, kb, vb, ids, q.cpu(), key.cpu(), value.cpu(), seqs)
    # the needles dominate: query head 0 of sequence 0 returns (nearly) its V row
    pos = 100_000
    vrow = vb[ids.index(plan.tables[0][pos // 16]), pos % 16, 0].double()
    assert (ref.out[0, 0] - vrow).abs().max().item() < 1e-3
    out = gh.run_gpu_step(plan, k, v, q, key, value, torch.float32, append=append)
    torch.cuda.synchronize()
    assert _flags() == 0
    gh.assert_close_to_oracle(out, ref.out, ATOL)
    assert torch.equal(k[idx].cpu(), ref.k_blocks)
    assert torch.equal(v[idx].cpu(), ref.v_blocks)


# ---- write and copy on their own: whole pool, bit-exact ---------------------

@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_write_bitexact_whole_pool(dtype):
    import oracle.paged_ops as ops
    import paged_kv_cache_117_gb300 as pkv
    g = torch.Generator().manual_seed(9)
    N, B, H, D, T = 300, 16, 8, 128, 257
    k = torch.randn((N, B, H, D), generator=g).to(dtype)
    v = torch.randn((N, B, H, D), generator=g).to(dtype)
    key = torch.randn((T, H, D), generator=g).to(dtype)
    val = torch.randn((T, H, D), generator=g).to(dtype)
    slots = torch.randperm(N * B, generator=g)[:T].to(torch.int64)
    slots[::7] = -1
    kr, vr = k.clone(), v.clone()
    ops.write_kv(kr, vr, key, val, slots.tolist())
    kd, vd = k.cuda(), v.cuda()
    pkv.paged_kv_write(key.cuda(), val.cuda(), kd, vd, slots.cuda())
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kr) and torch.equal(vd.cpu(), vr)
    assert _flags() == 0


@pytest.mark.parametrize("b,d", [(16, 128), (4, 64), (32, 64)])
def test_copy_bitexact_whole_pool(b, d):
    import oracle.paged_ops as ops
    import paged_kv_cache_117_gb300 as pkv
    g = torch.Generator().manual_seed(10)
    N, H = 200, 4
    k = torch.randn((N, b, H, d), generator=g).to(torch.bfloat16)
    v = torch.randn((N, b, H, d), generator=g).to(torch.bfloat16)
    perm = torch.randperm(N, generator=g).tolist()
    pairs = [(perm[i], perm[100 + i]) for i in range(37)]     # distinct dst, dst not a src
    kr, vr = k.clone(), v.clone()
    ops.copy_blocks(kr, vr, pairs)
    kd, vd = k.cuda(), v.cuda()
    pkv.paged_block_copy(kd, vd, gh.pairs_tensor(pairs).cuda())
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kr) and torch.equal(vd.cpu(), vr)
    assert _flags() == 0


def test_conflicting_copy_pairs_are_skipped_and_flagged():
    """Copies of one call run in no order: pairs whose dst repeats another
    pair's dst, or is another pair's src, are skipped and flagged; the other
    pairs are copied (compared with the oracle copying only those)."""
    import oracle.paged_ops as ops
    import paged_kv_cache_117_gb300 as pkv
    g = torch.Generator().manual_seed(11)
    N, B, H, D = 64, 16, 2, 128
    k = torch.randn((N, B, H, D), generator=g).to(torch.bfloat16)
    v = torch.randn((N, B, H, D), generator=g).to(torch.bfloat16)
    pairs = [(1, 10), (2, 11), (3, 10),      # dst 10 twice: both skipped
             (4, 12), (12, 13),              # 12 is a dst and a src: (4, 12) skipped
             (5, 20), (6, 21)]               # clean
    kr, vr = k.clone(), v.clone()
    ops.copy_blocks(kr, vr, [(2, 11), (12, 13), (5, 20), (6, 21)])
    kd, vd = k.cuda(), v.cuda()
    pkv.paged_block_copy(kd, vd, gh.pairs_tensor(pairs).cuda())
    torch.cuda.synchronize()
    assert _flags() == pkv.FLAG_PAIR_CONFLICT
    assert torch.equal(kd.cpu(), kr) and torch.equal(vd.cpu(), vr)


@pytest.mark.parametrize("with_ws", [False, True])
def test_copy_4096_pairs_bitexact(with_ws):
    """A long pair list (4,096 copies in one call, as a scheduler moving many
    sequences would make): the whole pool equals the oracle's after the copy,
    with the scan check and with the counter workspace; the workspace is all
    zero again afterwards, ready for the next call."""
    import oracle.paged_ops as ops
    import paged_kv_cache_117_gb300 as pkv
    g = torch.Generator().manual_seed(12)
    N, B, H, D = 10_000, 16, 2, 64
    k = torch.randn((N, B, H, D), generator=g).to(torch.bfloat16)
    v = torch.randn((N, B, H, D), generator=g).to(torch.bfloat16)
    perm = torch.randperm(N, generator=g).tolist()
    pairs = [(perm[i], perm[4096 + i]) for i in range(4096)]
    pairs[7] = (pairs[7][1], pairs[7][1])          # a block copied onto itself clashes with none
    kr, vr = k.clone(), v.clone()
    ops.copy_blocks(kr, vr, pairs)
    kd, vd = k.cuda(), v.cuda()
    ws = pkv.block_copy_workspace(kd) if with_ws else None
    pt = gh.pairs_tensor(pairs).cuda()
    for _ in range(2):                             # the second call finds the workspace reset
        pkv.paged_block_copy(kd, vd, pt, workspace=ws)
    torch.cuda.synchronize()
    assert torch.equal(kd.cpu(), kr) and torch.equal(vd.cpu(), vr)
    assert _flags() == 0
    if with_ws:
        assert ws.numel() >= N * 8 and int(ws.count_nonzero()) == 0


def test_conflicting_copy_pairs_with_workspace():
    """The counter check finds the same conflicts as the scan, and leaves the
    workspace zeroed."""
    import oracle.paged_ops as ops
    import paged_kv_cache_117_gb300 as pkv
    g = torch.Generator().manual_seed(11)
    N, B, H, D = 64, 16, 2, 128
    k = torch.randn((N, B, H, D), generator=g).to(torch.bfloat16)
    v = torch.randn((N, B, H, D), generator=g).to(torch.bfloat16)
    pairs = [(1, 10), (2, 11), (3, 10),      # dst 10 twice: both skipped
             (4, 12), (12, 13),              # 12 is a dst and a src: (4, 12) skipped
             (5, 20), (6, 21), (30, 30),     # clean; a self copy is clean too
             (7, 99)]                        # out of the pool: skipped, range-flagged
    kr, vr = k.clone(), v.clone()
    ops.copy_blocks(kr, vr, [(2, 11), (12, 13), (5, 20), (6, 21)])
    kd, vd = k.cuda(), v.cuda()
    ws = pkv.block_copy_workspace(kd)
    pkv.paged_block_copy(kd, vd, gh.pairs_tensor(pairs).cuda(), workspace=ws)
    torch.cuda.synchronize()
    assert _flags() == pkv.FLAG_PAIR_CONFLICT | pkv.FLAG_PAIR_RANGE
    assert torch.equal(kd.cpu(), kr) and torch.equal(vd.cpu(), vr)
    assert int(ws.count_nonzero()) == 0


def test_empty_calls_launch_nothing():
    import paged_kv_cache_117_gb300 as pkv
    k = torch.zeros((4, 16, 2, 64), dtype=torch.bfloat16, device="cuda")
    v = torch.zeros_like(k)
    pkv.paged_block_copy(k, v, torch.zeros((0, 2), dtype=torch.int64, device="cuda"))
    e = torch.zeros((0, 2, 64), dtype=torch.bfloat16, device="cuda")
    pkv.paged_kv_write(e, e, k, v, torch.zeros((0,), dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()


# ---- bad device-side metadata: skipped or clamped, flagged, never a fault ---

def test_bad_metadata_is_flagged_not_faulted():
    import paged_kv_cache_117_gb300 as pkv
    B, H, D, N = 16, 2, 64, 32
    k = torch.randn((N, B, H, D), device="cuda").to(torch.bfloat16)
    v = torch.randn((N, B, H, D), device="cuda").to(torch.bfloat16)
    k0, v0 = k.clone(), v.clone()
    # slot past the pool: skipped, flagged
    key = torch.randn((2, H, D), device="cuda").to(torch.bfloat16)
    pkv.paged_kv_write(key, key, k, v, torch.tensor([N * B, -5], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert _flags() == pkv.FLAG_SLOT_RANGE
    assert torch.equal(k, k0) and torch.equal(v, v0)
    # copy pair naming a block outside the pool: skipped, flagged
    pkv.paged_block_copy(k, v, torch.tensor([[0, N], [-1, 3]], dtype=torch.int64, device="cuda"))
    torch.cuda.synchronize()
    assert _flags() == pkv.FLAG_PAIR_RANGE
    assert torch.equal(k, k0) and torch.equal(v, v0)
    # block id outside the pool and a length past the table: flagged, finite
    q = torch.randn((2, 4, D), device="cuda").to(torch.bfloat16)
    tables = torch.tensor([[1, N + 5, 2], [3, 4, 5]], dtype=torch.int32, device="cuda")
    lens = torch.tensor([40, 10_000], dtype=torch.int32, device="cuda")
    out = torch.empty((2, 4, D), dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(out, q, k, v, tables, lens, 0.125, partition_tokens=16)
    torch.cuda.synchronize()
    f = _flags()
    assert f & pkv.FLAG_BLOCK_RANGE and f & pkv.FLAG_LEN_RANGE
    assert torch.isfinite(out).all()
