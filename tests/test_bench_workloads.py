"""The benchmark's workload selection on CPU: resizing a decode workload with
--seqs / --context keeps its heads, dtype, block size and partition, sizes
the pool and the table width for every sequence, names the result so that no
committed profile applies to it, and refuses the workloads whose sequences
share blocks or carry several query rows."""
import os
import sys

import pytest
import torch

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_cache_117_gb300 import workloads as wl  # noqa: E402


class Args:
    def __init__(self, workload="llama8b", seqs=None, context=None):
        self.workload, self.seqs, self.context = workload, seqs, context


def test_named_workload_is_unchanged():
    assert bench.select_workload(Args()) is wl.LLAMA8B


def test_fixed_batch_shape():
    w = bench.select_workload(Args(seqs=64, context=4096))
    base = wl.LLAMA8B
    assert (w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size, w.dtype,
            w.partition_tokens) == (base.num_q_heads, base.num_kv_heads, base.head_dim,
                                    base.block_size, base.dtype, base.partition_tokens)
    lens, tables, width, slots = bench.build_metadata(w)
    assert lens == [4096] * 64 and slots.shape == (64,)
    assert width == 4096 // 16
    assert all(len(t) == 256 for t in tables)
    # every block is distinct and inside the pool
    flat = [b for t in tables for b in t]
    assert len(set(flat)) == len(flat) and max(flat) < w.num_blocks
    assert w.name not in bench.TABLE_WIDTH_TOKENS
    assert bench.measured_traffic(w.name, w.partition_tokens, kv_write="append") is None


def test_more_sequences_keep_the_distribution():
    w = bench.select_workload(Args(seqs=32))
    assert w.lens_kind == wl.LLAMA8B.lens_kind and w.num_seqs == 32
    lens, tables, width, _ = bench.build_metadata(w)
    assert len(lens) == 32 and max(lens) <= width * w.block_size


def test_bytes_scale_with_the_batch():
    small = bench.select_workload(Args(seqs=8, context=1024))
    big = bench.select_workload(Args(seqs=16, context=1024))
    b_small = bench.algorithmic_bytes(small, *bench.build_metadata(small)[:3], 768, 2)
    b_big = bench.algorithmic_bytes(big, *bench.build_metadata(big)[:3], 768, 2)
    assert b_big["kv"] == 2 * b_small["kv"]
    assert b_small["kv"] == 8 * 1024 * small.num_kv_heads * small.head_dim * 2 * 2


@pytest.mark.parametrize("name", ["shared", "beam", "prefill", "prefix"])
def test_other_workloads_refuse_resizing(name):
    with pytest.raises(SystemExit):
        bench.select_workload(Args(workload=name, seqs=4, context=1024))


@pytest.mark.parametrize("name", ["tiny", "opt13b"])
def test_decode_state_from_the_native_manager_matches_the_oracle_manager(name):
    """The benchmark's decode state (tables, lengths and the step's slots)
    comes from the library's block manager through the C ABI; the oracle's
    manager, fed the same free queue and the same appends, assigns the same
    blocks and slots."""
    w = wl.scaled(wl.WORKLOADS[name], 16, 1024) if name != "tiny" else wl.TINY
    native = bench.build_metadata(w, manager="native")
    ref = bench.build_metadata(w, manager="oracle")
    assert native[:3] == ref[:3]
    assert native[3].tolist() == ref[3].tolist()
    # tiny: lengths 1, 6, 9, 17 in 4-token blocks; 1, 9 and 17 open a fresh block
    if name == "tiny":
        tables, slots = native[1], native[3].tolist()
        for s, L in enumerate(native[0]):
            assert len(tables[s]) == -(-L // 4)
            assert slots[s] // 4 == tables[s][-1] and slots[s] % 4 == (L - 1) % 4


def test_sizes_must_be_positive():
    with pytest.raises(SystemExit):
        bench.select_workload(Args(seqs=0, context=1024))
    with pytest.raises(SystemExit):
        bench.select_workload(Args(seqs=4, context=0))


def test_prefix_manager_cost_is_reported():
    cost = bench.prefix_manager_cost(wl.PREFIX, rounds=2)
    assert cost["requests"] == wl.PREFIX.num_seqs
    assert cost["prompt_tokens"] == 2048 + 256
    assert 0 < cost["us_per_request"] == cost["us_per_request_miss"] < 1e6
    assert 0 < cost["us_per_request_hit"] < 1e6
    # a new request finds its system prompt cached (128 full blocks of 16);
    # the same request again finds every full block cached but the one that
    # holds its last token, which is always recomputed
    assert cost["cached_tokens_per_request_miss"] == 2048
    assert cost["cached_tokens_per_request_hit"] == 2048 + 256 - 16


def _run_jobs(jobs):
    import oracle.paged_ops as ops
    return [bench.oracle_step(ops, j, j["k"].clone(), j["v"].clone()) for j in jobs]


def test_oracle_jobs_reproduce_the_whole_batch():
    """The CPU baseline splits a step by sequence into jobs on compact pools;
    together they compute what the oracle computes on the whole batch."""
    import oracle.paged_ops as ops
    w = wl.scaled(wl.SHARED, 24, num_blocks=600)
    w = bench.dataclasses.replace(w, lens_args=(3, 40, 8, 0, 9))
    lens, tables, width, slots, pairs, setup = bench.build_shared_step(w, bench.OracleManager)
    pairs = [tuple(p) for p in pairs.tolist()]
    assert pairs, "the step should contain copy-on-write copies"
    k, v = wl.make_pool(w)
    ops.copy_blocks(k, v, setup)
    q, key, value = wl.make_step_inputs(w)
    kw, vw = k.clone(), v.clone()
    ops.copy_blocks(kw, vw, pairs)
    ops.write_kv(kw, vw, key, value, slots.tolist())
    want = ops.attend(q, kw, vw, tables, lens, w.scale)
    parts = bench.split_by_work(range(len(lens)), lens, 5)
    assert len(parts) == 5 and sorted(s for p in parts for s in p) == list(range(len(lens)))
    fetch = lambda ids: (k[ids], v[ids])
    outs = _run_jobs(bench.oracle_jobs(w, "decode", parts, tables, lens, pairs, fetch, q, key,
                                       value, slots.tolist()))
    for part, out in zip(parts, outs):
        assert torch.equal(out, want[part])


def test_subchunk_jobs_reproduce_the_chunk():
    """The reference arm splits one sequence's chunk by query rows; each
    piece is the oracle's chunked call on a shorter sequence, and together
    they give exactly the rows of the whole chunk."""
    import oracle.paged_ops as ops
    w = bench.dataclasses.replace(wl.PREFILL, num_seqs=3, num_blocks=64, lens_args=(40, 2))
    lens, tables, width, slots, counts, qs, _ = bench.build_multiquery_step(
        w, bench.OracleManager)
    k, v = wl.make_pool(w)
    T = qs[-1]
    q = torch.randn((T, w.num_q_heads, w.head_dim),
                    generator=torch.Generator().manual_seed(1)).to(w.dtype)
    key, value = wl.make_rows(w, 0, T)
    kw, vw = k.clone(), v.clone()
    ops.write_kv(kw, vw, key, value, slots.tolist())
    want = ops.attend_chunked(q, kw, vw, tables, lens, qs, w.scale)
    fetch = lambda ids: (k[ids], v[ids])
    for seq in range(len(lens)):
        jobs = bench.subchunk_jobs(w, seq, lens, tables, counts, qs, fetch, q, key, value,
                                   slots.tolist(), 4)
        assert 1 < len(jobs) <= 4
        got = torch.cat(_run_jobs(jobs))
        assert torch.equal(got, want[qs[seq]:qs[seq + 1]])


def test_oracle_pool_reports_the_workers_it_used():
    w = wl.TINY
    lens, tables, width, slots = bench.build_metadata(w, manager="oracle")
    k, v = wl.make_pool(w)
    q, key, value = wl.make_step_inputs(w)
    pool = bench.OraclePool(3)
    try:
        cpu = bench.cpu_baseline_decode(pool, w, lens, tables, width, [],
                                        lambda ids: (k[ids], v[ids]), q, key, value, slots)
    finally:
        pool.close()
    assert cpu["cores"] == 3 and cpu["value"] > 0 and cpu["kind"] == "oracle"
