"""Multi-query (chunked prefill + decode) paged attention on the GPU against
the oracle: the chunk's K/V rows written through paged_kv_write, then
paged_attention_chunked, every output row compared (fp32 output within 2e-3;
16-bit outputs within max(2e-3, 1 ulp) of the rounded oracle) and the pool
compared bit-exactly."""

import pytest
import torch

import oracle.paged_ops as ops
from paged_kv_cache_117_gb300 import workloads as wl
from tests import gpu_harness as gh

pytestmark = pytest.mark.gpu
ATOL = 2e-3


def _w(Hq, Hkv, D, B, dtype=torch.bfloat16, N=400, seed=500):
    return wl.Workload("chunk_case", 0, Hq, Hkv, D, B, N, dtype, 0, seed, "fixed", ())


def _run(w, prior, counts, out_dtype=torch.float32, poison=False, width=None, p_format="hilo",
         v_spike=None, mixed=False, partition_tokens=64):
    import paged_kv_cache_117_gb300 as pkv
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    step = gh.plan_chunked(w, prior, counts, width)
    T = step.query_start[-1]
    k, v = wl.make_pool(w, "cpu")
    if poison:   # slots no sequence owns hold NaN: never read, never allowed to leak
        for b, o in gh.unused_slots(step):
            k[b, o] = float("nan")
            v[b, o] = float("nan")
    g = torch.Generator().manual_seed(w.seed + 77)
    q = torch.randn((T, w.num_q_heads, w.head_dim), generator=g).to(w.dtype)
    key, val = wl.make_rows(w, 0, T)
    if v_spike is not None:   # one new V value far outside the f16 range
        val[0, 0, 0] = v_spike
    kd, vd = k.cuda(), v.cuda()
    ops.write_kv(k, v, key, val, step.slots)
    ref = ops.attend_chunked(q, k, v, step.tables, step.lens, step.query_start, w.scale)
    pkv.paged_kv_write(key.cuda(), val.cuda(), kd, vd,
                       torch.tensor(step.slots, dtype=torch.int64, device="cuda"))
    out = torch.full((T, w.num_q_heads, w.head_dim), float("nan"), dtype=out_dtype, device="cuda")
    args = (out, q.cuda(), kd, vd, wl.pad_tables(step.tables, step.width).cuda(),
            torch.tensor(step.lens, dtype=torch.int32, device="cuda"),
            torch.tensor(step.query_start, dtype=torch.int32, device="cuda"), w.scale)
    if mixed:
        pkv.paged_attention_mixed(*args, max_query_len=max(counts), p_format=p_format,
                                  partition_tokens=partition_tokens)
    else:
        pkv.paged_attention_chunked(*args, max_query_len=max(counts), p_format=p_format)
    torch.cuda.synchronize()
    flags = pkv.read_device_flags(clear=True)
    if v_spike is not None:
        assert flags == pkv.FLAG_V_RANGE and torch.isfinite(out).all()
        return None, step
    assert flags == 0
    assert torch.equal(kd.cpu().view(torch.int16), k.view(torch.int16))
    assert torch.equal(vd.cpu().view(torch.int16), v.view(torch.int16))
    return gh.assert_close_to_oracle(out, ref, ATOL), step


# ---- mixed batches: decode rows on the decode kernel, chunks on the tensor cores

@pytest.mark.parametrize("pt", [0, 16, 64])
def test_mixed_call_prefill_and_decode(pt):
    # prompt chunks at various offsets, decode tokens (one at the very first
    # position, one spanning several partitions), an idle sequence
    _run(_w(8, 2, 128, 16), [0, 200, 511, 37, 1000, 64, 5, 0],
         [130, 129, 1, 1, 256, 0, 3, 1], mixed=True, partition_tokens=pt)


def test_mixed_call_decode_only_and_chunks_only():
    _run(_w(8, 2, 128, 16), [0, 17, 300, 4000], [1, 1, 1, 1], mixed=True, width=300)
    _run(_w(8, 2, 128, 16), [0, 300], [40, 2], mixed=True)


@pytest.mark.parametrize("hq,hkv", [(4, 4), (16, 1), (40, 40), (64, 8)])
def test_mixed_call_group_sizes(hq, hkv):
    _run(_w(hq, hkv, 128, 16, N=500), [0, 150, 9, 77], [97, 1, 2, 1], mixed=True)


def test_mixed_call_f16_cache_16bit_outputs_and_f16_p():
    w = _w(8, 2, 64, 32, dtype=torch.float16)
    _run(w, [0, 90, 33], [150, 1, 70], out_dtype=torch.float16, mixed=True)
    _run(_w(8, 2, 128, 16), [0, 90, 5], [150, 1, 70], out_dtype=torch.bfloat16, mixed=True,
         p_format="f16")


def test_mixed_decode_rows_equal_the_decode_call():
    """A decode row of a mixed batch is computed exactly as paged_attention_decode
    computes it: the same kernel, partitions and merge order, so the rows are
    bit-identical; the chunk rows are the chunked kernel's."""
    import paged_kv_cache_117_gb300 as pkv
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = _w(32, 8, 128, 16, N=1200)
    prior, counts = [900, 0, 3000, 64, 2000], [1, 200, 1, 1, 77]
    step = gh.plan_chunked(w, prior, counts, None)
    T = step.query_start[-1]
    k, v = wl.make_pool(w, "cuda")
    g = torch.Generator().manual_seed(9)
    q = torch.randn((T, w.num_q_heads, w.head_dim), generator=g).to(w.dtype).cuda()
    key, val = wl.make_rows(w, 0, T, "cuda")
    pkv.paged_kv_write(key, val, k, v, torch.tensor(step.slots, dtype=torch.int64, device="cuda"))
    tab = wl.pad_tables(step.tables, step.width).cuda()
    lens = torch.tensor(step.lens, dtype=torch.int32, device="cuda")
    qs = torch.tensor(step.query_start, dtype=torch.int32, device="cuda")
    out = torch.empty((T, w.num_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    pkv.paged_attention_mixed(out, q, k, v, tab, lens, qs, w.scale, partition_tokens=256)
    chunk = torch.empty_like(out)
    pkv.paged_attention_chunked(chunk, q, k, v, tab, lens, qs, w.scale)
    dec = [s for s, n in enumerate(counts) if n == 1]
    rows = [step.query_start[s] for s in dec]
    dout = torch.empty((len(dec), w.num_q_heads, w.head_dim), dtype=torch.float32, device="cuda")
    pkv.paged_attention_decode(dout, q[rows].contiguous(), k, v, tab[dec].contiguous(),
                               lens[dec].contiguous(), w.scale, partition_tokens=256)
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    assert torch.equal(out[rows], dout)
    other = [r for r in range(T) if r not in rows]
    assert torch.equal(out[other], chunk[other])


def test_one_prompt_whole():
    # a fresh prompt in one chunk: 300 tokens, Llama-shaped group of 4
    _run(_w(8, 2, 128, 16), [0], [300])


def test_mixed_batch_prefill_and_decode():
    # prompt chunks at various offsets, decode tokens, an idle sequence
    _run(_w(8, 2, 128, 16), [0, 200, 511, 37, 1000, 64, 5],
         [130, 129, 1, 1, 256, 0, 3])


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 1), (16, 1), (10, 2), (12, 4), (64, 1), (128, 1)])
def test_group_sizes(hq, hkv):
    # G = 1, 8, 16, 5 (rows 125 of 128), 3, 64 and 128 (one token per tile)
    _run(_w(hq, hkv, 64, 16, N=300), [0, 150, 9], [97, 40, 2])


@pytest.mark.parametrize("b", [8, 16, 32])
@pytest.mark.parametrize("d", [64, 128])
def test_block_and_head_dim(b, d):
    _run(_w(8, 2, d, b, N=600), [0, 129, 300], [200, 127, 33])


def test_f16_cache_and_16bit_outputs():
    w = _w(8, 2, 128, 16, dtype=torch.float16)
    _run(w, [0, 90], [150, 70], out_dtype=torch.float16)
    _run(_w(8, 2, 128, 16), [0, 90], [150, 70], out_dtype=torch.bfloat16)


def test_tile_boundaries():
    # chunk and context lengths on and next to the 128-token tile edges
    _run(_w(8, 2, 128, 16, N=700), [0, 0, 128, 127, 255, 1, 0],
         [128, 256, 128, 1, 129, 127, 129])


def test_poisoned_unused_slots():
    # slots past each sequence's length hold NaN in the pool
    _run(_w(8, 2, 128, 16), [0, 45, 300], [77, 130, 12], poison=True)
    _run(_w(8, 2, 64, 32), [0, 5], [33, 100], poison=True)


def test_wide_table_and_long_context():
    # table rows wider than needed; one sequence with 3,000 tokens of context
    _run(_w(8, 2, 128, 16, N=800), [2900, 0], [100, 50], width=300)


@pytest.mark.parametrize("p_format", ["hilo", "f16"])
def test_longest_context(p_format):
    # 300 queries after 30,000 cached tokens (237 KV tiles, a 1,894-block table
    # row) next to two single-token decodes
    _run(_w(8, 2, 128, 16, N=2400), [30000, 0, 7], [300, 1, 1], p_format=p_format)


def test_prefill_full_size_sampled():
    """The benchmark's prefill workload at full size, in its launch
    configuration (16 chunks of 512 tokens after up to 7,168 cached tokens,
    512-block table rows, bf16 output): the chunk's writes bit-exact on the
    sampled sequences' blocks, and sampled rows against the oracle (a row at
    position p is decode attention over positions 0..p)."""
    import random
    import paged_kv_cache_117_gb300 as pkv
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = wl.PREFILL
    prior, counts = wl.chunk_plan(w)
    step = gh.plan_chunked(w, prior, counts, width=8192 // w.block_size)
    T = step.query_start[-1]
    k, v = wl.make_pool_chunked(w, "cuda")
    g = torch.Generator(device="cuda")
    g.manual_seed(w.seed + 3000)
    q = torch.randn((T, w.num_q_heads, w.head_dim), generator=g, device="cuda").to(w.dtype)
    key, val = wl.make_rows(w, 0, T, "cuda")
    lens = step.lens
    seqs = sorted({0, max(range(len(lens)), key=lambda s: lens[s]),
                   min(range(len(lens)), key=lambda s: lens[s])})
    ids = sorted({b for s in seqs for b in step.tables[s]})
    remap = {b: i for i, b in enumerate(ids)}
    idx = torch.tensor(ids, device="cuda")
    kb, vb = k[idx].cpu(), v[idx].cpu()
    B = w.block_size
    rows = [r for s in seqs for r in range(step.query_start[s], step.query_start[s + 1])]
    ops.write_kv(kb, vb, key.cpu()[rows], val.cpu()[rows],
                 [remap[step.slots[r] // B] * B + step.slots[r] % B for r in rows])
    out = torch.empty((T, w.num_q_heads, w.head_dim), dtype=torch.bfloat16, device="cuda")
    pkv.paged_kv_write(key, val, k, v, torch.tensor(step.slots, dtype=torch.int64, device="cuda"))
    pkv.paged_attention_chunked(out, q, k, v, wl.pad_tables(step.tables, step.width).cuda(),
                                torch.tensor(lens, dtype=torch.int32, device="cuda"),
                                torch.tensor(step.query_start, dtype=torch.int32, device="cuda"),
                                w.scale, max_query_len=max(counts))
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    assert torch.equal(k[idx].cpu(), kb) and torch.equal(v[idx].cpu(), vb)
    assert torch.isfinite(out).all()
    rnd = random.Random(3)
    qc = q.cpu()
    for s in seqs:
        n, L, r0 = counts[s], lens[s], step.query_start[s]
        for i in sorted({0, 1, 31, 32, 127, 128, n // 2, n - 1, rnd.randrange(n)}):
            p = L - n + i
            ref = ops.attend(qc[r0 + i:r0 + i + 1], kb, vb, [[remap[b] for b in step.tables[s]]],
                             [p + 1], w.scale)
            gh.assert_close_to_oracle(out[r0 + i:r0 + i + 1], ref, ATOL)


# ---- P as one f16 operand (V converted to f16 for a bf16 cache) -------------

@pytest.mark.parametrize("hq,hkv", [(8, 2), (16, 1), (10, 2), (64, 1)])
def test_f16_p_group_sizes(hq, hkv):
    _run(_w(hq, hkv, 64, 16, N=300), [0, 150, 9], [97, 40, 2], p_format="f16")


@pytest.mark.parametrize("b", [8, 16, 32])
@pytest.mark.parametrize("d", [64, 128])
def test_f16_p_block_and_head_dim(b, d):
    _run(_w(8, 2, d, b, N=600), [0, 129, 300], [200, 127, 33], p_format="f16")


def test_f16_p_f16_cache_mixed_batch_and_poison():
    _run(_w(8, 2, 128, 16, dtype=torch.float16), [0, 200, 511, 37], [130, 129, 1, 3],
         p_format="f16")
    _run(_w(8, 2, 128, 16), [0, 45, 300], [77, 130, 12], poison=True, p_format="f16")
    _run(_w(8, 2, 128, 16), [0, 0, 128, 127, 255], [128, 256, 128, 1, 129], p_format="f16",
         out_dtype=torch.bfloat16)


def test_f16_p_v_out_of_range_is_flagged():
    # a V value beyond +-65504 cannot be an f16 operand: it is clamped, the
    # output stays finite and the device flag word reports it
    _run(_w(8, 2, 128, 16), [0, 40], [30, 20], p_format="f16", v_spike=1.0e5)


def test_bad_metadata_is_flagged_not_faulted():
    """Device-side values the kernel cannot trust: a block id outside the
    pool is read as zeros and flagged; a length past the table is clamped and
    flagged; a sequence with more queries than tokens, or query_start out of
    order, is skipped (rows untouched) and flagged.  Nothing faults."""
    import paged_kv_cache_117_gb300 as pkv
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    B, H, D, N = 16, 2, 64, 32
    k = torch.randn((N, B, H, D), device="cuda").to(torch.bfloat16)
    v = torch.randn((N, B, H, D), device="cuda").to(torch.bfloat16)
    q = torch.randn((40, 8, D), device="cuda").to(torch.bfloat16)
    tables = torch.tensor([[1, N + 5, 2], [3, 4, 5], [6, 7, 8], [9, 10, 11]],
                          dtype=torch.int32, device="cuda")
    # seq 0: bad block id; seq 1: length past the table (clamped to 48);
    # seq 2: 10 queries but 5 tokens (skipped); seq 3: fine
    lens = torch.tensor([40, 10_000, 5, 30], dtype=torch.int32, device="cuda")
    qs = torch.tensor([0, 10, 20, 30, 40], dtype=torch.int32, device="cuda")
    out = torch.full((40, 8, D), 7.0, dtype=torch.float32, device="cuda")
    pkv.paged_attention_chunked(out, q, k, v, tables, lens, qs, 0.125, max_query_len=10)
    torch.cuda.synchronize()
    f = pkv.read_device_flags(clear=True)
    assert f & pkv.FLAG_BLOCK_RANGE and f & pkv.FLAG_LEN_RANGE
    assert not f & pkv.FLAG_TIMEOUT
    assert torch.isfinite(out).all()
    assert (out[20:30] == 7.0).all()                # skipped rows untouched
    # query_start running backwards: the sequence is skipped and flagged
    qs_bad = torch.tensor([0, 10, 5, 30, 40], dtype=torch.int32, device="cuda")
    out.fill_(7.0)
    pkv.paged_attention_chunked(out, q, k, v, tables, torch.tensor([10, 10, 10, 30], dtype=torch.int32,
                                device="cuda"), qs_bad, 0.125, max_query_len=25)
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) & pkv.FLAG_LEN_RANGE
    assert torch.isfinite(out).all()


def test_chunked_step_in_a_cuda_graph():
    """A chunked-prefill step (write + attention) captured in one CUDA graph
    and replayed: the call path does no host synchronisation when
    max_query_len is given, and replays match the oracle."""
    import paged_kv_cache_117_gb300 as pkv
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA GPU")
    w = _w(8, 2, 128, 16)
    step = gh.plan_chunked(w, [0, 100, 37], [90, 40, 1])
    T = step.query_start[-1]
    k, v = wl.make_pool(w, "cpu")
    kd, vd = k.cuda(), v.cuda()
    g = torch.Generator().manual_seed(5)
    q = torch.randn((T, 8, 128), generator=g).to(w.dtype)
    key, val = wl.make_rows(w, 0, T)
    ops.write_kv(k, v, key, val, step.slots)
    ref = ops.attend_chunked(q, k, v, step.tables, step.lens, step.query_start, w.scale)
    qd, keyd, vald = q.cuda(), key.cuda(), val.cuda()
    slots = torch.tensor(step.slots, dtype=torch.int64, device="cuda")
    tab = wl.pad_tables(step.tables).cuda()
    lens = torch.tensor(step.lens, dtype=torch.int32, device="cuda")
    qs = torch.tensor(step.query_start, dtype=torch.int32, device="cuda")
    out = torch.empty((T, 8, 128), dtype=torch.float32, device="cuda")
    pkv.load()
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        with torch.cuda.graph(graph, stream=side):
            pkv.paged_kv_write(keyd, vald, kd, vd, slots)
            pkv.paged_attention_chunked(out, qd, kd, vd, tab, lens, qs, w.scale, max_query_len=90)
    torch.cuda.current_stream().wait_stream(side)
    for _ in range(2):
        out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        assert pkv.read_device_flags(clear=True) == 0
        gh.assert_close_to_oracle(out, ref, ATOL)
