"""Builds one decode step of a workload and runs it through both sides.

The metadata (block tables, context lengths, slot mapping, copy-on-write
pairs) comes from the oracle's block manager; tensors come from the seeded
generators in ``paged_kv_cache_117_gb300.workloads``.  The GPU side runs
through the C ABI (binding); the oracle side runs ``oracle.paged_ops`` on CPU
copies of the same inputs -- taken before any library kernel touches them.
"""
from __future__ import annotations

from dataclasses import dataclass
from typing import List, Optional, Sequence

import torch

import oracle.paged_ops as ops
from oracle.block_manager import BlockManager
from paged_kv_cache_117_gb300 import workloads as wl


@dataclass
class StepPlan:
    w: wl.Workload
    lens: List[int]                 # after this step's token
    tables: List[List[int]]         # after this step
    width: int                      # block table row width (max_blocks)
    slots: List[int]                # this step's slot per sequence (-1: none)
    step_pairs: List[tuple]         # CoW copies this step (before the write)
    setup_pairs: List[tuple]        # CoW copies made while building the state


def plan_step(w: wl.Workload, width: Optional[int] = None) -> StepPlan:
    bm = BlockManager(w.num_blocks, w.block_size, wl.free_block_order(w))
    setup_pairs: List[tuple] = []
    if w.lens_kind == "shared":
        plan = wl.shared_prefix_plan(w)
        S = plan.prompts * plan.samples
        for p in range(plan.prompts):
            root = p * plan.samples
            bm.add_sequence(root)
            bm.append_tokens(root, plan.prompt_len)
            for i in range(1, plan.samples):
                bm.fork(root, root + i)
        for s in range(S):
            _, cows = bm.append_tokens(s, plan.own[s])
            setup_pairs += cows
        hist = None
    else:
        lens0 = wl.context_lens(w)
        S = len(lens0)
        for s, L in enumerate(lens0):
            bm.add_sequence(s)
            bm.append_tokens(s, max(0, L - 1))
        hist = lens0
    slots, step_pairs = [], []
    for s in range(S):
        if hist is not None and hist[s] == 0:
            slots.append(-1)
            continue
        slot, cow = bm.append(s)
        slots.append(slot)
        if cow is not None:
            step_pairs.append(cow)
    bm.check_invariants()
    lens = [bm.lens[s] for s in range(S)]
    tables = [list(bm.tables[s]) for s in range(S)]
    need = max(1, max(len(t) for t in tables))
    if width is None:
        width = need
    assert width >= need
    return StepPlan(w, lens, tables, width, slots, step_pairs, setup_pairs)


def table_tensor(plan: StepPlan) -> torch.Tensor:
    return wl.pad_tables(plan.tables, plan.width)


def pairs_tensor(pairs: Sequence[tuple]) -> torch.Tensor:
    if not pairs:
        return torch.zeros((0, 2), dtype=torch.int64)
    return torch.tensor([list(p) for p in pairs], dtype=torch.int64)


def needed_blocks(plan: StepPlan, seqs: Sequence[int]) -> List[int]:
    """Blocks the oracle needs to reproduce the chosen sequences' step: their
    tables' blocks plus the sources of any copy landing in one of them."""
    need = set()
    for s in seqs:
        need.update(plan.tables[s])
    for src, dst in plan.setup_pairs + plan.step_pairs:
        if dst in need:
            need.add(src)
    for src, dst in plan.setup_pairs:
        if dst in need:
            need.add(src)
    return sorted(need)


@dataclass
class OracleResult:
    out: torch.Tensor                # float64 [len(seqs), Hq, D]
    k_blocks: torch.Tensor           # pool blocks after the step, [len(ids), B, H, D]
    v_blocks: torch.Tensor
    block_ids: List[int]


def oracle_step(plan: StepPlan, k_pool_cpu_blocks, v_pool_cpu_blocks, block_ids,
                q_cpu, key_cpu, value_cpu, seqs: Sequence[int]) -> OracleResult:
    """Runs setup copies, step copies, the write and attention for ``seqs`` on
    a compact CPU pool holding ``block_ids`` (in that order)."""
    w = plan.w
    remap = {b: i for i, b in enumerate(block_ids)}
    kc = k_pool_cpu_blocks.clone()
    vc = v_pool_cpu_blocks.clone()
    local = lambda pairs: [(remap[a], remap[b]) for a, b in pairs if b in remap and a in remap]
    ops.copy_blocks(kc, vc, local(plan.setup_pairs))
    ops.copy_blocks(kc, vc, local(plan.step_pairs))
    B = w.block_size
    slots, rows = [], []
    for s, slot in enumerate(plan.slots):
        if slot >= 0 and slot // B in remap:
            slots.append(remap[slot // B] * B + slot % B)
            rows.append(s)
    if rows:
        ops.write_kv(kc, vc, key_cpu[rows], value_cpu[rows], slots)
    tables = [[remap[b] for b in plan.tables[s]] for s in seqs]
    lens = [plan.lens[s] for s in seqs]
    out = ops.attend(q_cpu[list(seqs)], kc, vc, tables, lens, w.scale)
    return OracleResult(out, kc, vc, list(block_ids))


def run_gpu_step(plan: StepPlan, k_cache, v_cache, q, key, value, out_dtype=torch.float32,
                 partition_tokens=None, run_setup=True, append=False):
    """Setup copies (if any), then the step: copy -> write -> attend, through
    the library (``append``: copy -> paged_attention_decode_append, the write
    and the attention in one call).  Returns out (device tensor)."""
    import paged_kv_cache_117_gb300 as pkv
    dev = k_cache.device
    if run_setup and plan.setup_pairs:
        pkv.paged_block_copy(k_cache, v_cache, pairs_tensor(plan.setup_pairs).to(dev))
    pkv.paged_block_copy(k_cache, v_cache, pairs_tensor(plan.step_pairs).to(dev))
    tables = table_tensor(plan).to(dev)
    lens = torch.tensor(plan.lens, dtype=torch.int32, device=dev)
    S = len(plan.lens)
    out = torch.empty((S, plan.w.num_q_heads, plan.w.head_dim), dtype=out_dtype, device=dev)
    pt = plan.w.partition_tokens if partition_tokens is None else partition_tokens
    if append:
        # the slot the call derives (position L - 1) is the manager's slot
        B = plan.w.block_size
        for s, slot in enumerate(plan.slots):
            L = plan.lens[s]
            assert slot == (plan.tables[s][(L - 1) // B] * B + (L - 1) % B if L else -1)
        pkv.paged_attention_decode_append(out, q, key, value, k_cache, v_cache, tables, lens,
                                          plan.w.scale, partition_tokens=pt)
        return out
    slots = torch.tensor(plan.slots, dtype=torch.int64, device=dev)
    pkv.paged_kv_write(key, value, k_cache, v_cache, slots)
    pkv.paged_attention_decode(out, q, k_cache, v_cache, tables, lens, plan.w.scale,
                               partition_tokens=pt)
    return out


def ulp(x: torch.Tensor, dtype: torch.dtype) -> torch.Tensor:
    """Spacing of `dtype` at |x| (x float64)."""
    mant = {torch.bfloat16: 7, torch.float16: 10, torch.float32: 23}[dtype]
    e = torch.floor(torch.log2(x.abs().clamp(min=2.0 ** -14)))
    return torch.pow(2.0, e - mant)


def assert_close_to_oracle(gpu_out: torch.Tensor, ref64: torch.Tensor, atol=2e-3):
    """fp32 outputs: max |gpu - oracle| <= atol.  16-bit outputs: compared with
    the oracle rounded once to that dtype, allowing max(atol, 1 ulp)."""
    g = gpu_out.detach().to("cpu").to(torch.float64)
    assert torch.isfinite(g).all(), "non-finite output"
    if gpu_out.dtype == torch.float32:
        err = (g - ref64).abs().max().item() if g.numel() else 0.0
        assert err <= atol, f"max abs err {err:.3e} > {atol}"
        return err
    r = ref64.to(gpu_out.dtype).to(torch.float64)
    err = (g - r).abs()
    bound = torch.maximum(torch.full_like(err, atol), ulp(r, gpu_out.dtype))
    bad = (err > bound)
    assert not bad.any(), f"{int(bad.sum())} elements beyond max(atol, 1 ulp); max err {err.max():.3e}"
    return err.max().item() if err.numel() else 0.0


# ---- beam search -------------------------------------------------------------

@dataclass
class BeamHistory:
    w: wl.Workload
    steps: list            # per step: (pairs, slots, order)
    lens: List[int]        # final beams (in final order), after the last step
    tables: List[List[int]]
    width: int


def plan_beam(w: wl.Workload, steps: Optional[int] = None, width: Optional[int] = None) -> BeamHistory:
    """Beam-search history on the oracle's block manager: prompts, then for
    every step the survivors' forks, the pruned beams' frees and one token per
    surviving beam (with the copy-on-write pairs it causes)."""
    plan = wl.beam_plan(w, steps)
    bm = BlockManager(w.num_blocks, w.block_size, wl.free_block_order(w))
    R, W = plan.requests, plan.width
    for r in range(R):
        root = r * W
        bm.add_sequence(root)
        bm.append_tokens(root, plan.prompt_len)
        for i in range(1, W):
            bm.fork(root, r * W + i)
    hist = []
    for st in wl.beam_schedule(plan):
        for parent, child in st.forks:
            bm.fork(parent, child)
        for sq in st.frees:
            bm.free_sequence(sq)
        slots, pairs = [], []
        for sq in st.order:
            slot, cow = bm.append(sq)
            slots.append(slot)
            if cow is not None:
                pairs.append(cow)
        hist.append((pairs, slots, st.order))
        bm.check_invariants()
    order = hist[-1][2]
    tables = [list(bm.tables[sq]) for sq in order]
    lens = [bm.lens[sq] for sq in order]
    need = max(len(t) for t in tables)
    return BeamHistory(w, hist, lens, tables, width or need)


# ---- chunked prefill ---------------------------------------------------------

@dataclass
class ChunkStep:
    w: wl.Workload
    prior: List[int]          # tokens in the cache before the step
    counts: List[int]         # this step's query tokens per sequence
    lens: List[int]           # after the step
    tables: List[List[int]]
    width: int
    slots: List[int]          # one per query row, packed by sequence
    query_start: List[int]


def plan_chunked(w: wl.Workload, prior: Sequence[int], counts: Sequence[int],
                 width: Optional[int] = None) -> ChunkStep:
    """Sequences that already hold ``prior`` tokens receive ``counts`` new
    tokens each (a prompt chunk, a decode token, or nothing), through the
    oracle's block manager."""
    bm = BlockManager(w.num_blocks, w.block_size, wl.free_block_order(w))
    slots = []
    for s, (c0, n) in enumerate(zip(prior, counts)):
        bm.add_sequence(s)
        bm.append_tokens(s, c0)
    for s, n in enumerate(counts):
        new, _ = bm.append_tokens(s, n)
        slots += list(new)
    S = len(prior)
    lens = [bm.lens[s] for s in range(S)]
    tables = [list(bm.tables[s]) for s in range(S)]
    need = max(1, max(len(t) for t in tables))
    qs = [0]
    for n in counts:
        qs.append(qs[-1] + n)
    return ChunkStep(w, list(prior), list(counts), lens, tables, width or need, slots, qs)


def unused_slots(step: ChunkStep) -> List[tuple]:
    """(block, offset) of every pool slot that no sequence's first L_s tokens
    occupy."""
    B = step.w.block_size
    used = set()
    for t, L in zip(step.tables, step.lens):
        for pos in range(L):
            used.add((t[pos // B], pos % B))
    return [(b, o) for b in range(step.w.num_blocks) for o in range(B) if (b, o) not in used]
