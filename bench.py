#!/usr/bin/env python3
"""Benchmark of the paged KV cache decode hot path on GB300.

One step = one pass of the whole path over one batch: the batched
copy-on-write block copy (when the workload has copies), the KV write of every
sequence's new token, and decode attention (partitioned pass + merge) -- all
through the library's C ABI; by default the write happens inside the
attention call (paged_attention_decode_append; --kv-write separate runs
paged_kv_write then paged_attention_decode).  Inputs are resident in HBM when
timing starts.  Before each timed loop the GPU spins ~50 ms (outside every
timed span, inside wall_s_timed) so that the host queues steps ahead of it.
L2 is flushed before every timed step, outside the timed span: a 256 MiB
buffer is written (evicting what the last step left in L2), then another
256 MiB buffer is read, so that the flush's own dirty lines are written back
before the timed span starts rather than inside it (a write-only flush adds
~15 us of write-back to a ~230 us decode call).

Prints one JSON line (rank 0).  ``--impl reference`` times the fp64 CPU oracle
on a bounded sample of the same workload instead.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl native|reference]
                    [--workload llama8b]
"""
import argparse
import dataclasses
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import torch  # noqa: E402

from paged_kv_cache_117_gb300 import workloads as wl  # noqa: E402

METRIC = "paged decode attn: achieved HBM GB/s (% of GB300 peak); seq-steps/s"
UNIT = "GB/s"
FLUSH_BYTES = 256 << 20
TABLE_WIDTH_TOKENS = {"tiny": 32, "opt13b": 2048, "llama8b": 8192, "qwen72b": 8192,
                      "shared": 2048, "beam": 2048, "prefill": 8192, "prefix": 4096,
                      "mixed": 8192}
MULTIQUERY = ("chunked", "prefix", "mixed")   # workloads of several query rows per sequence
SHARING = ("shared", "beam")   # workloads whose sequences share blocks


L2_NOTE = ("flushed before every step, outside the timed span: 256 MiB written, then another "
           "256 MiB read so the flush's dirty lines are written back before the span")


class L2Flush:
    """Evicts L2 between timed iterations: writes one buffer larger than L2,
    then reads a second one, leaving L2 full of clean lines that no kernel of
    the step reads."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 8, dtype=torch.int64, device=dev)
        self.sink = torch.zeros(1, dtype=torch.int64, device=dev)

    def __call__(self):
        self.w.zero_()
        self.sink.add_(self.r.sum())


def host_head_start():
    """Gives the host a head start before a timed loop: the GPU first spins
    for ~50 ms (a fixed cycle count), outside every timed span, while the
    host queues the steps, so that a pause of the host (a page fault, a
    collector pass) does not leave the GPU idle inside a step's span."""
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(100_000_000)


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=300)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="llama8b", choices=sorted(TABLE_WIDTH_TOKENS))
    ap.add_argument("--partition", type=int, default=None,
                    help="partition_tokens (default: the workload's, 512)")
    ap.add_argument("--cpu-workers", type=int, default=0,
                    help="oracle worker processes for the CPU baseline (default: all cores)")
    ap.add_argument("--no-other-configs", action="store_true",
                    help="default run: time only the headline workload, not the other "
                         "decode configurations")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--layers", type=int, default=1,
                    help="layers per step: one K/V pool per layer, shared block tables")
    ap.add_argument("--kv-write", choices=["append", "separate"], default="append",
                    help="decode workloads: the step's KV write inside the attention call "
                         "(paged_attention_decode_append) or as its own kernel (paged_kv_write "
                         "then paged_attention_decode)")
    ap.add_argument("--p-format", choices=["hilo", "f16"], default="hilo",
                    help="chunked workloads: P as hi + lo 16-bit operands, or as one f16 operand")
    ap.add_argument("--graph", action="store_true",
                    help="capture the whole step (all layers) in one CUDA graph and replay it")
    ap.add_argument("--seqs", type=int, default=None,
                    help="decode workloads of independent sequences: this many sequences "
                         "(the workload's length distribution unless --context is given)")
    ap.add_argument("--context", type=int, default=None,
                    help="decode workloads of independent sequences: every sequence this "
                         "long (tokens, counting this step's)")
    return ap.parse_args()


def select_workload(a):
    """The named workload, or (--seqs / --context) a copy of a decode
    workload of independent sequences with another batch or length: the same
    heads, dims, dtype, block size and partition, a pool large enough for
    every sequence, and a name that says so (no committed profile applies)."""
    w = wl.WORKLOADS[a.workload]
    if a.seqs is None and a.context is None:
        return w
    if w.lens_kind not in ("fixed", "uniform", "lognormal"):
        raise SystemExit("--seqs / --context apply to the decode workloads of independent "
                         "sequences (tiny, opt13b, llama8b, qwen72b)")
    S = a.seqs if a.seqs is not None else w.num_seqs
    if S <= 0 or (a.context is not None and a.context <= 0):
        raise SystemExit("--seqs and --context must be positive")
    if a.context is not None:
        lk, args, name = "fixed", (a.context,) * S, f"{w.name}-{S}x{a.context}"
    else:
        lk, args, name = w.lens_kind, w.lens_args, f"{w.name}-{S}seqs"
    hi = max(args) if lk == "fixed" else (args[1] if lk == "uniform" else args[3])
    blocks = S * -(-hi // w.block_size)
    return dataclasses.replace(w, name=name, num_seqs=S, lens_kind=lk, lens_args=args,
                               num_blocks=max(w.num_blocks if lk != "fixed" else 0,
                                              blocks + blocks // 8 + 64))


def width_tokens(w):
    """Block-table row width in tokens: the workload's, or the longest
    possible sequence of a resized one."""
    if w.name in TABLE_WIDTH_TOKENS:
        return TABLE_WIDTH_TOKENS[w.name]
    return max(w.lens_args) if w.lens_kind == "fixed" else (
        w.lens_args[1] if w.lens_kind == "uniform" else w.lens_args[3])


# ---------------------------------------------------------------------------
# workload and its algorithmic bytes

def build_metadata(w, manager="native"):
    """Decode state of independent sequences, built by a block manager whose
    free queue is the workload's seeded permutation (so each sequence's
    blocks are scattered over the pool): every sequence's earlier tokens,
    then this step's token of every sequence.  ``manager``: "native" (the
    library's pkv_bm_*) or "oracle" (the reference arm's, no library call).
    Returns lens, tables, width and the step's slot per sequence (int64,
    CPU), as the manager assigned them."""
    lens0 = wl.context_lens(w)
    S = len(lens0)
    if manager == "native":
        import paged_kv_cache_117_gb300 as pkv
        bm = pkv.BlockManager(w.num_blocks, w.block_size, wl.free_block_order(w))
        for s, L in enumerate(lens0):
            bm.add_sequence(s)
            if L > 1:
                bm.append_tokens(s, L - 1)
        slots, pairs = bm.append(range(S))
        assert pairs.shape[0] == 0
        tables, lens = zip(*(bm.table(s) for s in range(S)))
    else:
        from oracle.block_manager import BlockManager
        bm = BlockManager(w.num_blocks, w.block_size, wl.free_block_order(w))
        for s, L in enumerate(lens0):
            bm.add_sequence(s)
            bm.append_tokens(s, max(0, L - 1))
        slots = torch.tensor([bm.append(s)[0] for s in range(S)], dtype=torch.int64)
        tables, lens = [bm.tables[s] for s in range(S)], [bm.lens[s] for s in range(S)]
    assert list(lens) == lens0
    width = -(-width_tokens(w) // w.block_size)
    return lens0, [list(t) for t in tables], width, slots


def _manager(manager):
    """The block-manager class: the library's (default) or the one given."""
    if manager is not None:
        return manager
    import paged_kv_cache_117_gb300 as pkv
    return pkv.BlockManager


def build_shared_step(w, manager=None):
    """Parallel-sampling state built by the library's block manager: prompts,
    forks, each sample's own tokens (with the copies they caused), then this
    step's token of every sample.  Returns lens, tables, width, the step's
    slots and copy pairs, and the copies made while building the state."""
    plan = wl.shared_prefix_plan(w)
    bm = _manager(manager)(w.num_blocks, w.block_size, wl.free_block_order(w))
    S = plan.prompts * plan.samples
    setup = []
    for p in range(plan.prompts):
        root = p * plan.samples
        bm.add_sequence(root)
        bm.append_tokens(root, plan.prompt_len)
        for i in range(1, plan.samples):
            bm.fork(root, root + i)
    for s in range(S):
        _, pairs = bm.append_tokens(s, plan.own[s])
        setup += pairs.tolist()
    slots, pairs = bm.append(range(S))
    tables, lens = zip(*(bm.table(s) for s in range(S)))
    width = -(-TABLE_WIDTH_TOKENS[w.name] // w.block_size)
    return list(lens), [list(t) for t in tables], width, slots, pairs, setup


def build_beam_step(w, manager=None):
    """Beam-search state built by the library's block manager: prompts, beam
    forks, then every history step's forks, frees and one token per surviving
    beam.  Returns lens, tables, width, the measured step's slots and copy
    pairs, and the history as (pairs, slots) per step (to replay on a pool)."""
    plan = wl.beam_plan(w)
    bm = _manager(manager)(w.num_blocks, w.block_size, wl.free_block_order(w))
    R, W = plan.requests, plan.width
    for r in range(R):
        bm.add_sequence(r * W)
        bm.append_tokens(r * W, plan.prompt_len)
        for i in range(1, W):
            bm.fork(r * W, r * W + i)
    hist = []
    for st in wl.beam_schedule(plan):
        for parent, child in st.forks:
            bm.fork(parent, child)
        for sq in st.frees:
            bm.free_sequence(sq)
        slots, pairs = bm.append(st.order)
        hist.append((pairs, slots))
    tables, lens = zip(*(bm.table(sq) for sq in st.order))
    width = -(-TABLE_WIDTH_TOKENS[w.name] // w.block_size)
    pairs, slots = hist.pop()
    return list(lens), [list(t) for t in tables], width, slots, pairs, hist


def build_chunked_step(w, manager=None):
    """Chunked-prefill state built by the library's block manager: every
    sequence's earlier chunks, then this step's chunk.  Returns lens, tables,
    width, the chunk rows' slots, the per-sequence query counts and
    query_start."""
    prior, counts = wl.chunk_plan(w)
    bm = _manager(manager)(w.num_blocks, w.block_size, wl.free_block_order(w))
    for s, c0 in enumerate(prior):
        bm.add_sequence(s)
        if c0:
            bm.append_tokens(s, c0)
    slots = torch.cat([bm.append_tokens(s, n)[0] for s, n in enumerate(counts)])
    tables, lens = zip(*(bm.table(s) for s in range(len(prior))))
    width = -(-TABLE_WIDTH_TOKENS[w.name] // w.block_size)
    qs = [0]
    for n in counts:
        qs.append(qs[-1] + n)
    return list(lens), [list(t) for t in tables], width, slots, counts, qs


def build_prefix_step(w, manager=None):
    """Prefix-caching state built by the library's prefix-cache manager: one
    earlier request per system prompt prefilled it (its full blocks stay
    cached after it finished), then every request looks its prompt up and
    prefills only the rest.  Returns lens, tables, width, slots, counts,
    query_start and the prompt tokens the cache saved."""
    plan = wl.prefix_plan(w)
    if manager is None:
        import paged_kv_cache_117_gb300 as pkv
        cache_cls = pkv.PrefixCache
    else:   # the reference arm: the oracle's prefix cache
        from oracle.prefix_cache import PrefixCache as cache_cls
    pc = cache_cls(w.num_blocks, w.block_size, wl.free_block_order(w))
    for i, sysp in enumerate(plan.systems):
        sid = len(plan.prompts) + i
        warm = sysp + [0]
        c = pc.add_sequence(sid, warm)
        pc.append(sid, warm[c:])
        pc.free_sequence(sid)
    slots, counts, saved = [], [], 0
    for r, prompt in enumerate(plan.prompts):
        c = pc.add_sequence(r, prompt)
        slots.append(torch.as_tensor(pc.append(r, prompt[c:]), dtype=torch.int64))
        counts.append(len(prompt) - c)
        saved += c
    tables, lens = zip(*(pc.table(r) for r in range(len(plan.prompts))))
    width = -(-TABLE_WIDTH_TOKENS[w.name] // w.block_size)
    qs = [0]
    for n in counts:
        qs.append(qs[-1] + n)
    return list(lens), [list(t) for t in tables], width, torch.cat(slots), counts, qs, saved


def build_multiquery_step(w, manager=None):
    """(lens, tables, width, slots, counts, query_start, description) of a
    multi-query workload."""
    if w.lens_kind == "prefix":
        lens, tables, width, slots, counts, qs, saved = build_prefix_step(w, manager)
        n_sys, sys_len, q_len = w.lens_args
        desc = (f"{w.name}: {w.num_seqs} requests, each one of {n_sys} system prompts of "
                f"{sys_len} tokens + its own {q_len}-token question (seeded token ids); the system "
                f"prompts' full blocks are in the prefix cache (chained SHA-256 keys), so "
                f"{saved} of {saved + sum(counts)} prompt tokens are taken over and each request "
                f"prefills {counts[0]} tokens attending over {lens[0]}; "
                f"{w.num_q_heads} q / {w.num_kv_heads} kv heads, head_dim {w.head_dim}, "
                f"{str(w.dtype).replace('torch.', '')}, block {w.block_size}, {w.num_blocks}-block pool")
        return lens, tables, width, slots, counts, qs, desc
    prior, _ = wl.chunk_plan(w)
    lens, tables, width, slots, counts, qs = build_chunked_step(w, manager)
    if w.lens_kind == "mixed":
        n_dec, median, sigma, lo, hi, n_chunk, chunk, mx = w.lens_args
        dec_tokens = sum(lens[:n_dec])
        desc = (f"{w.name}: a continuous-batching step of {n_dec} decode sequences (lognormal "
                f"lengths, median {median:g}, sigma {sigma:g}, clipped to [{lo}, {hi}]; "
                f"{dec_tokens} tokens) and {n_chunk} prompt chunks of {chunk} tokens after "
                f"0..{mx} cached chunks each (cached tokens {min(prior[n_dec:])}.."
                f"{max(prior[n_dec:])}), {w.num_q_heads} q / {w.num_kv_heads} kv heads, head_dim "
                f"{w.head_dim}, {str(w.dtype).replace('torch.', '')}, block {w.block_size}, "
                f"{w.num_blocks}-block pool, blocks scattered by a seeded permutation, table "
                f"width {width}, q/K/V ~ N(0,1)")
        return lens, tables, width, slots, counts, qs, desc
    return lens, tables, width, slots, counts, qs, chunked_desc(w, width, prior, counts)


def chunked_flops(w, lens, counts):
    """Multiply-adds x 2 of QK^T and PV over the visible (causal) pairs: query
    i of a chunk of n in a sequence of L tokens sees L - n + i + 1 keys."""
    pairs = sum(n * (L - n) + n * (n + 1) // 2 for L, n in zip(lens, counts))
    return 4 * w.head_dim * w.num_q_heads * pairs


def replay_beam_history(w, k, v, hist, dev):
    """Runs the history's copies and writes on one pool through the library."""
    import paged_kv_cache_117_gb300 as pkv
    for t, (pairs, slots) in enumerate(hist):
        key, val = wl.make_rows(w, t, slots.numel(), dev)
        if pairs.shape[0]:
            pkv.paged_block_copy(k, v, pairs.to(dev))
        pkv.paged_kv_write(key, val, k, v, slots.to(dev))


def algorithmic_bytes(w, lens, width, pt, out_es, n_pairs=0, tables=None):
    """Bytes the step must move at minimum: every valid K/V row of every
    (sequence, KV head) once, q, the used block-table entries, lengths, the
    output, the split-context records (written once and read back once), the
    new K/V rows in and out, and the copied blocks."""
    es = w.elem_bytes
    S, Hq, Hkv, D, B = len(lens), w.num_q_heads, w.num_kv_heads, w.head_dim, w.block_size
    part_blocks = width if pt == 0 else pt // B
    nb = [-(-L // B) for L in lens]
    nparts = [-(-n // part_blocks) if n else 0 for n in nb]
    kv = sum(lens) * Hkv * D * es * 2
    rec = sum(p for p in nparts if p > 1) * Hq * (D + 2) * 4
    attention = kv + S * Hq * D * es + sum(nb) * 4 + S * 4 + S * Hq * D * out_es + 2 * rec
    write = S * Hkv * D * es * 2 * 2 + S * 8
    block_bytes = B * Hkv * D * es
    copy = n_pairs * block_bytes * 2 * 2 + n_pairs * 16
    res = {"kv": kv, "attention": attention, "records": 2 * rec, "write": write,
           "copy": copy, "step": attention + write + copy}
    if tables is not None:   # distinct (block, KV head, valid slot) rows, for shared blocks
        seen = {}
        for t, L in zip(tables, lens):
            for j, b in enumerate(t[: -(-L // B)]):
                seen[b] = max(seen.get(b, 0), min(B, L - j * B))
        res["kv_unique"] = sum(seen.values()) * Hkv * D * es * 2
    return res


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


DECODE_SOURCES = ("paged_kv_cache_117_gb300/csrc/decode_kernel.cuh",
                  "paged_kv_cache_117_gb300/csrc/pkv_device.cuh",
                  "paged_kv_cache_117_gb300/csrc/pkv_launch.h",
                  "paged_kv_cache_117_gb300/csrc/capi.cu")


CHUNKED_SOURCES = ("paged_kv_cache_117_gb300/csrc/chunked_kernel.cuh",
                   "paged_kv_cache_117_gb300/csrc/pkv_device.cuh",
                   "paged_kv_cache_117_gb300/csrc/pkv_tcgen05.cuh",
                   "paged_kv_cache_117_gb300/csrc/pkv_launch.h",
                   "paged_kv_cache_117_gb300/csrc/capi.cu")


def sources_sha256(sources):
    """Hash of the kernel's sources with comments and whitespace removed, so
    that a comment edit does not invalidate a profile of unchanged code."""
    import hashlib
    import re
    h = hashlib.sha256()
    for f in sources:
        with open(os.path.join(ROOT, f)) as fh:
            text = fh.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()


def measured_traffic(workload, partition_tokens, profile=None, sources=DECODE_SOURCES,
                     kv_write=None):
    """DRAM bytes per launch from a committed ncu summary (by default the
    decode kernel's on this workload, profiles/decode_kernel_<workload>.md),
    or None when there is none, it was taken on another workload or partition
    size, or the kernel's sources changed since."""
    profile = profile or f"decode_kernel_{workload}.md"
    try:
        text = open(os.path.join(ROOT, "profiles", profile)).read()
        kv = dict(line.split(": ", 1) for line in text.splitlines()
                  if line.startswith(("traffic_", "source_sha256")))
        if (kv.get("source_sha256") == sources_sha256(sources)
                and kv.get("traffic_kv_write", "separate") == (kv_write or "separate")
                and kv.get("traffic_workload") == workload
                and int(kv.get("traffic_partition_tokens", -1)) == partition_tokens):
            return int(kv["traffic_bytes_per_launch"])
    except Exception:
        pass
    return None


def workload_desc(w, width):
    if w.lens_kind == "shared":
        pr, plen, n, lo, hi = w.lens_args
        lk = (f"{pr} prompts of {plen} tokens x {n} samples sharing the prompt blocks, "
              f"{lo}-{hi} own tokens per sample (samples 0 and 1 of each prompt: 0), "
              f"copy-on-write of the shared partial block in the step; shared blocks are "
              f"read once per sharer (L2 reuse across sharers, not graded)")
    elif w.lens_kind == "beam":
        rq, plen, n, c, steps = w.lens_args
        lk = (f"beam search: {rq} prompts of {plen} tokens x {n} beams, {c} seeded-score "
              f"candidates per beam, top {n} survive; {steps} steps of forks, frees, "
              f"copy-on-write copies and writes replayed on the pool before the measured "
              f"step (copies + write + attention)")
    elif w.lens_kind == "fixed":
        lk = f"fixed lengths {sorted(set(w.lens_args))}"
    else:
        lk = {"lognormal": "lognormal lengths (median %g, sigma %g, clipped to [%d, %d])",
              "uniform": "uniform lengths in [%d, %d]"}[w.lens_kind] % w.lens_args
    return (f"{w.name}: {w.num_seqs} seqs, {w.num_q_heads} q / {w.num_kv_heads} kv heads, "
            f"head_dim {w.head_dim}, {str(w.dtype).replace('torch.', '')}, block {w.block_size}, "
            f"{lk}, {w.num_blocks}-block pool, blocks scattered by a seeded permutation, "
            f"table width {width}, q/K/V ~ N(0,1), one new token per seq")


# ---------------------------------------------------------------------------
# clocks

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


class ClockSampler:
    def __init__(self, device_index):
        self.proc = None
        self.path = None
        self.dev = device_index

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--query-gpu={CLOCK_FIELDS}", "--format=csv,noheader,nounits",
                 "-i", str(self.dev), "-lms", "50"], stdout=self.f, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.f.close()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 10:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return None
        sm = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        mx = [float(r[3]) for r in rows if r[3].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[6 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(world, x, device):
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# CPU oracle timing (the only place bench.py touches oracle/)

def cpu_model():
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if line.lower().startswith(("model name", "cpu part", "hardware")):
                    return line.split(":", 1)[1].strip()
    except Exception:
        pass
    import platform
    return platform.processor() or platform.machine()


def _oracle_worker(conn):
    """One oracle worker process.  It receives its share of a sample once
    ("load"), then runs the fp64 oracle on it each time it is told to ("go"),
    on a fresh copy of its compact pool, with one torch thread, and reports
    its own busy seconds."""
    import pickle
    torch.set_num_threads(1)
    import oracle.paged_ops as ops
    job = None
    while True:
        msg = pickle.loads(conn.recv_bytes())
        if msg[0] == "stop":
            break
        if msg[0] == "load":
            job = msg[1]
            conn.send_bytes(pickle.dumps("ready"))
            continue
        kc, vc = job["k"].clone(), job["v"].clone()
        t0 = time.perf_counter()
        oracle_step(ops, job, kc, vc)
        conn.send_bytes(pickle.dumps(("done", time.perf_counter() - t0)))


def oracle_step(ops, job, kc, vc):
    """The oracle's step on one job, in place on the pool copy kc/vc: the
    copies, the write of the new rows, then attention.  Returns the output."""
    ops.copy_blocks(kc, vc, job["pairs"])
    ops.write_kv(kc, vc, job["key"], job["value"], job["slots"])
    if job["kind"] == "decode":
        return ops.attend(job["q"], kc, vc, job["tables"], job["lens"], job["scale"])
    return ops.attend_chunked(job["q"], kc, vc, job["tables"], job["lens"], job["qs"],
                              job["scale"])


class OraclePool:
    """Worker processes for timing the fp64 oracle across the host's cores.

    Started with the spawn method (safe whatever CUDA state the parent is
    in).  A sample is split by sequence into one job per worker; the jobs are
    sent and loaded first, then all workers are started together and the
    wall time from the start signal to the last worker's reply is the
    sample's time.  Each worker runs torch with one thread, so the number of
    workers that received a job is the number of cores used."""

    def __init__(self, workers):
        import multiprocessing as mp
        ctx = mp.get_context("spawn")
        self.workers = []
        for _ in range(max(1, workers)):
            parent, child = ctx.Pipe()
            proc = ctx.Process(target=_oracle_worker, args=(child,), daemon=True)
            proc.start()
            child.close()
            self.workers.append((proc, parent))
        self.active = []

    def __len__(self):
        return len(self.workers)

    def load(self, jobs):
        import pickle
        assert len(jobs) <= len(self.workers)
        self.active = [c for (_, c), _ in zip(self.workers, jobs)]
        for c, job in zip(self.active, jobs):
            c.send_bytes(pickle.dumps(("load", job)))
        for c in self.active:
            assert pickle.loads(c.recv_bytes()) == "ready"

    def run(self):
        """(wall seconds, per-worker busy seconds) of one pass over the
        loaded sample."""
        import pickle
        go = pickle.dumps(("go",))
        t0 = time.perf_counter()
        for c in self.active:
            c.send_bytes(go)
        busy = [pickle.loads(c.recv_bytes())[1] for c in self.active]
        return time.perf_counter() - t0, busy

    def close(self):
        import pickle
        for proc, c in self.workers:
            try:
                c.send_bytes(pickle.dumps(("stop",)))
            except Exception:
                pass
        for proc, c in self.workers:
            proc.join(timeout=10)
            if proc.is_alive():
                proc.kill()
        self.workers = []


def split_by_work(seqs, work, n):
    """Sequences spread over at most n workers, longest first to the least
    loaded (each part kept in sequence order)."""
    parts, loads = [[] for _ in range(n)], [0] * n
    for s in sorted(seqs, key=lambda s: -work[s]):
        i = loads.index(min(loads))
        parts[i].append(s)
        loads[i] += work[s]
    return [sorted(p) for p in parts if p]


def oracle_jobs(w, kind, seqs_parts, tables, lens, pairs, fetch, q_rows, key_rows, value_rows,
                slots, row_start=None):
    """One oracle job per part: a compact pool holding the part's blocks (and
    the sources of the step's copies into them), its copy pairs, new rows and
    slots, queries, tables and lengths, all renumbered into that pool.
    ``fetch(ids)`` returns the pool blocks ``ids`` as CPU tensors.  Decode:
    row s of q/key/value/slots belongs to sequence s.  Chunked: sequence s
    owns rows row_start[s] .. row_start[s+1]-1."""
    B = w.block_size
    jobs = []
    for part in seqs_parts:
        ids = {b for s in part for b in tables[s]}
        step_pairs = [(int(a), int(b)) for a, b in pairs if int(b) in ids]
        ids |= {a for a, _ in step_pairs}
        ids = sorted(ids)
        remap = {b: i for i, b in enumerate(ids)}
        kc, vc = fetch(ids)
        rows = ([s for s in part] if row_start is None else
                [r for s in part for r in range(row_start[s], row_start[s + 1])])
        loc = [remap[int(slots[r]) // B] * B + int(slots[r]) % B for r in rows]
        job = {"kind": kind, "k": kc, "v": vc, "scale": w.scale,
               "pairs": [(remap[a], remap[b]) for a, b in step_pairs],
               "key": key_rows[rows].cpu(), "value": value_rows[rows].cpu(), "slots": loc,
               "q": q_rows[rows].cpu(), "tables": [[remap[b] for b in tables[s]] for s in part],
               "lens": [lens[s] for s in part]}
        if row_start is not None:
            qs = [0]
            for s in part:
                qs.append(qs[-1] + row_start[s + 1] - row_start[s])
            job["qs"] = qs
        jobs.append(job)
    return jobs


def device_fetch(k, v):
    def fetch(ids):
        idx = torch.tensor(ids, dtype=torch.int64, device=k.device)
        return k[idx].cpu(), v[idx].cpu()
    return fetch


def cpu_baseline_decode(pool, w, lens, tables, width, pairs, fetch, q, key, value, slots):
    """The fp64 oracle's step (copies, KV write, attention) over the whole
    batch, split by sequence over the pool's workers."""
    S = len(lens)
    parts = split_by_work(range(S), lens, len(pool))
    pairs = [tuple(p) for p in (pairs.tolist() if torch.is_tensor(pairs) else pairs)]
    pool.load(oracle_jobs(w, "decode", parts, tables, lens, pairs, fetch, q, key, value,
                          slots.tolist() if torch.is_tensor(slots) else slots))
    wall, busy = pool.run()
    b = algorithmic_bytes(w, lens, width, 0, w.elem_bytes, len(pairs))["step"]
    return {"value": b / wall / 1e9, "unit": UNIT, "cores": len(parts), "kind": "oracle",
            "cpu": f"{cpu_model()}, {os.cpu_count()} logical cores",
            "sample": f"fp64 oracle (torch CPU ops) step of all {S} sequences: "
                      f"{len(pairs)} block copies, KV write, attention; split by sequence over "
                      f"{len(parts)} worker processes with one torch thread each, {wall:.2f} s "
                      f"wall ({sum(busy):.1f} s busy); bytes = the step's algorithmic bytes "
                      f"without split-context records"}


# Decode configurations measured after the headline one in a default run
# (each under "other_configs" of the one JSON line).
OTHER_DECODE_CONFIGS = ("opt13b", "qwen72b", "shared")


def run_native(a, world, rank, local):
    import paged_kv_cache_117_gb300 as pkv
    from paged_kv_cache_117_gb300 import build as pbuild
    if rank == 0:
        pbuild.build()
    barrier(world)
    pkv.load()
    assert torch.cuda.is_available(), "the native benchmark needs a GPU"
    w = select_workload(a)
    others = []
    if (not a.no_other_configs and w is wl.LLAMA8B and a.layers == 1 and not a.graph
            and a.partition is None):
        others = [wl.WORKLOADS[n] for n in OTHER_DECODE_CONFIGS]
    pool = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        pool = OraclePool(a.cpu_workers or os.cpu_count() or 1)
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    try:
        res = measure_decode(a, w, world, rank, dev, pool)
        if others:
            sub = argparse.Namespace(**{**vars(a), "partition": None, "layers": 1,
                                        "graph": False})
            res["other_configs"] = []
            for wo in others:
                r = measure_decode(sub, wo, world, rank, dev, pool)
                for key_ in ("metric", "unit", "n_gpus", "steps", "warmup", "higher_is_better",
                             "scaling", "vs_baseline", "data"):
                    r.pop(key_, None)
                res["other_configs"].append(r)
        if others:
            res["block_copy"] = measure_block_copy(wl.LLAMA8B, dev, a.steps, a.warmup)
    finally:
        if pool is not None:
            pool.close()
    return res


def measure_block_copy(w, dev, steps, warmup, sizes=(16, 256, 4096)):
    """paged_block_copy alone on a pool of the workload's shape: P disjoint
    (src, dst) pairs drawn from a seeded permutation, for each P with the scan
    check (no workspace) and with the counter workspace.  GB/s counts every
    copied block read once and written once in both pools."""
    import paged_kv_cache_117_gb300 as pkv
    k, v = wl.make_pool_chunked(w, dev)
    ws = pkv.block_copy_workspace(k)
    perm = torch.randperm(w.num_blocks, generator=torch.Generator().manual_seed(w.seed + 6000))
    block_bytes = w.block_size * w.num_kv_heads * w.head_dim * w.elem_bytes
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    peak, kind = peak_hbm()
    rows = []
    for P in sizes:
        pairs = torch.stack([perm[:P], perm[P:2 * P]], 1).to(dev)
        for wsp in (None, ws):
            for _ in range(max(3, warmup)):
                flush()
                pkv.paged_block_copy(k, v, pairs, workspace=wsp)
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]
            torch.cuda.synchronize()
            host_head_start()
            for e0, e1 in evs:
                flush()
                e0.record(stream)
                pkv.paged_block_copy(k, v, pairs, workspace=wsp)
                e1.record(stream)
            torch.cuda.synchronize()
            us = 1e3 * sum(e0.elapsed_time(e1) for e0, e1 in evs) / steps
            nbytes = P * block_bytes * 2 * 2 + P * 16
            gbs = nbytes / (us * 1e-6) / 1e9
            rows.append({"pairs": P, "check": "scan" if wsp is None else "counters",
                         "us": round(us, 2), "gbs": round(gbs, 1),
                         "frac": round(gbs / peak, 4), "launches": 1 if wsp is None else 3})
    assert pkv.read_device_flags(clear=True) == 0
    return {"workload": f"{w.name}-shaped pool ({w.num_blocks} blocks of {block_bytes} B per "
                        f"pool), disjoint pairs from a seeded permutation; L2 flushed before "
                        f"each call; bytes = each copied block read and written in K and V",
            "peak": peak, "peak_kind": f"{kind} hbm_gbs", "rows": rows}


def measure_decode(a, w, world, rank, dev, pool):
    """One decode workload: build its state, time the step and the attention
    call, the end-to-end step through host buffers, and (with a pool) the
    fp64 oracle's step on the host cores.  Returns the bench line's fields."""
    import paged_kv_cache_117_gb300 as pkv
    pt = w.partition_tokens if a.partition is None else a.partition
    k, v = wl.make_pool_chunked(w, dev)
    hist = None
    if w.lens_kind == "shared":
        lens, tables, width, slots_cpu, pairs_cpu, setup = build_shared_step(w)
        if setup:   # copies made while the samples added their own tokens
            pkv.paged_block_copy(k, v, torch.tensor(setup, dtype=torch.int64, device=dev))
    elif w.lens_kind == "beam":
        lens, tables, width, slots_cpu, pairs_cpu, hist = build_beam_step(w)
        replay_beam_history(w, k, v, hist, dev)
    else:
        lens, tables, width, slots_cpu = build_metadata(w)
        pairs_cpu = torch.zeros((0, 2), dtype=torch.int64)
    tab_cpu = wl.pad_tables(tables, width)
    lens_cpu = torch.tensor(lens, dtype=torch.int32)
    q, key, value = wl.make_step_inputs(w, dev)
    tab, lens_t, slots = tab_cpu.to(dev), lens_cpu.to(dev), slots_cpu.to(dev)
    pairs = pairs_cpu.to(dev)
    layers = [(k, v, q, key, value)]
    for li in range(1, a.layers):   # one pool per layer; one block id = one slot range in all
        wl_l = dataclasses.replace(w, seed=w.seed + 10 * li)
        kl, vl = wl.make_pool_chunked(wl_l, dev)
        if w.lens_kind == "shared" and setup:
            pkv.paged_block_copy(kl, vl, torch.tensor(setup, dtype=torch.int64, device=dev))
        if hist is not None:
            replay_beam_history(wl_l, kl, vl, hist, dev)
        layers.append((kl, vl) + tuple(wl.make_step_inputs(wl_l, dev)))
    outs = [torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=w.dtype, device=dev)
            for _ in range(a.layers)]
    out = torch.empty((w.num_seqs, w.num_q_heads, w.head_dim), dtype=w.dtype, device=dev)
    nws = pkv.paged_attention_workspace_bytes(w.num_seqs, w.num_q_heads, w.head_dim,
                                              width * w.block_size, pt)
    ws = torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
    wss = [ws] + [torch.empty(max(nws, 16), dtype=torch.uint8, device=dev)
                  for _ in range(1, a.layers)]
    flush = L2Flush(dev)
    nbytes = algorithmic_bytes(w, lens, width, pt, out.element_size(), pairs.shape[0],
                               tables if w.lens_kind in SHARING else None)
    # block copy (when there are pairs) + KV write (its own kernel unless
    # appended by the attention call) + work list + attention, per layer
    fused = a.kv_write == "append"
    launches_per_step = a.layers * ((1 if pairs.shape[0] else 0) + (0 if fused else 1) + 2)

    # CPU-oracle step over the whole batch: the pool's blocks are fetched
    # before any kernel of the step runs on them
    cpu = None
    if pool is not None:
        cpu = cpu_baseline_decode(pool, w, lens, tables, width, pairs_cpu, device_fetch(k, v),
                                  q, key, value, slots_cpu)

    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def attend(o, ql, keyl, vall, kl, vl, tb, ln, wsl):
        if fused:
            pkv.paged_attention_decode_append(o, ql, keyl, vall, kl, vl, tb, ln, w.scale,
                                              partition_tokens=pt, workspace=wsl)
        else:
            pkv.paged_attention_decode(o, ql, kl, vl, tb, ln, w.scale, partition_tokens=pt,
                                       workspace=wsl)

    def step(d0=None, d1=None):
        for li, (kl, vl, ql, keyl, vall) in enumerate(layers):
            if pairs.shape[0]:
                pkv.paged_block_copy(kl, vl, pairs)
            if not fused:
                pkv.paged_kv_write(keyl, vall, kl, vl, slots)
            if li == 0 and d0 is not None:
                d0.record(stream)
            attend(outs[li] if li else out, ql, keyl, vall, kl, vl, tab, lens_t, wss[li])
            if li == 0 and d1 is not None:
                d1.record(stream)

    for _ in range(max(3, a.warmup)):
        flush()
        step()
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0

    K = a.steps
    graph = None
    if a.graph:
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph):
            step()
        torch.cuda.synchronize()
    evs = [(ev(), ev(), ev(), ev()) for _ in range(K)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    host_head_start()
    for s0, s1, d0, d1 in evs:
        flush()
        s0.record(stream)
        if graph is not None:
            graph.replay()
        else:
            step(d0, d1)
        s1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    clocks = sampler.stop()
    step_ms = sum(s0.elapsed_time(s1) for s0, s1, _, _ in evs) / K
    if graph is not None:   # layer 0's attention call, timed eagerly for the roofline
        host_head_start()
        for _, _, d0, d1 in evs:
            flush()
            d0.record(stream)
            attend(out, q, key, value, k, v, tab, lens_t, ws)
            d1.record(stream)
        torch.cuda.synchronize()
    dec_ms = sum(d0.elapsed_time(d1) for _, _, d0, d1 in evs) / K
    step_ms = max_over_ranks(world, step_ms, dev)
    dec_ms = max_over_ranks(world, dec_ms, dev)

    # end to end: each step's inputs (q, new K/V rows, block tables, lengths,
    # slot mapping -- not needed when the attention call appends -- and copy
    # pairs) arrive in one pinned host staging buffer and go to the device in
    # one copy; the result comes back in one copy
    slots_e, slots_cpu_e = (slots[:0], slots_cpu[:0]) if fused else (slots, slots_cpu)
    parts = [q, key, value, tab, lens_t, slots_e, pairs]
    sizes = [t.numel() * t.element_size() for t in parts]
    offs = [0]
    for n in sizes:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    h_in = torch.empty(offs[-1], dtype=torch.uint8).pin_memory()
    d_in = torch.empty(offs[-1], dtype=torch.uint8, device=dev)
    for t, o, n in zip((q, key, value, tab_cpu, lens_cpu, slots_cpu_e, pairs_cpu), offs, sizes):
        if n:
            h_in[o:o + n].copy_(t.cpu().contiguous().view(torch.uint8).view(-1))
    views = [d_in[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts, offs, sizes)]
    e_q, e_key, e_val, e_tab, e_lens, e_slots, e_pairs = views
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()
    h2d = sum(sizes)
    d2h = h_out.numel() * h_out.element_size()

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        if pairs.shape[0]:
            pkv.paged_block_copy(k, v, e_pairs)
        if not fused:
            pkv.paged_kv_write(e_key, e_val, k, v, e_slots)
        attend(out, e_q, e_key, e_val, k, v, e_tab, e_lens, ws)
        h_out.copy_(out, non_blocking=True)

    if a.layers != 1:   # the end-to-end leg times the single-layer step only
        e2e_step = None
    for _ in range(3 if e2e_step else 0):
        e2e_step()
    e2e_evs = [(ev(), ev()) for _ in range(K if e2e_step else 0)]
    barrier(world)
    torch.cuda.synchronize()
    host_head_start()
    for e0, e1 in e2e_evs:
        flush()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = (max_over_ranks(world, sum(e0.elapsed_time(e1) for e0, e1 in e2e_evs) / K, dev)
              if e2e_evs else None)
    assert pkv.read_device_flags(clear=True) == 0

    peak, peak_kind = peak_hbm()
    # the timed call's algorithmic bytes: the attention's, plus the new rows
    # read and stored when it appends them
    call_bytes = nbytes["attention"] + (nbytes["write"] if fused else 0)
    achieved = call_bytes / (dec_ms * 1e-3) / 1e9
    value_gbs = world * a.layers * nbytes["step"] / (step_ms * 1e-3) / 1e9
    res = {
        "metric": METRIC, "value": round(value_gbs, 1), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": max(3, a.warmup), "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": str(w.dtype).replace("torch.", "").replace("bfloat16", "bf16").replace("float16", "f16"),
        "data": "synthetic",
        "config": {"workload": workload_desc(w, width), "partition_tokens": pt,
                   "out_dtype": str(out.dtype).replace("torch.", ""),
                   "l2": L2_NOTE, "kv_write": a.kv_write,
                   "layers": a.layers, "cuda_graph": bool(a.graph),
                   "parallelism": f"replicas x{world} (independent batches, no collective)"},
        "pct_of_peak": round(100 * value_gbs / world / peak, 1),
        "seq_steps_per_s": round(world * w.num_seqs / (step_ms * 1e-3), 1),
        "attention_ms": round(dec_ms, 4),
        "bytes_per_step": nbytes,
        **({"unique_kv_gbs": round(world * a.layers * (nbytes["step"] - nbytes["kv"] + nbytes["kv_unique"])
                                   / (step_ms * 1e-3) / 1e9, 1)} if "kv_unique" in nbytes else {}),
        "roofline": {"kernel": ("paged_attention_decode_append (work list + KV write, attention "
                                "and merge in one pass)" if fused else
                                "paged_attention_decode (work list + attention with fused merge)"),
                     "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} hbm_gbs", "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "traffic": measured_traffic(w.name, pt, kv_write=a.kv_write)},
        "e2e": ({"value": round(world * nbytes["step"] / (e2e_ms * 1e-3) / 1e9, 1), "unit": UNIT,
                 "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": h2d,
                 "d2h_bytes_per_step": d2h} if e2e_ms else None),
        "gpu_launches": launches_per_step * K,
        "clocks": clocks,
        "wall_s_timed": round(wall, 4),
        "cpu_baseline": cpu,
    }
    return res


CHUNK_METRIC = "paged chunked-prefill attn: achieved TFLOP/s (% of GB300 bf16 dense peak)"


def peak_bf16():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    except Exception:
        return 1900.0, "fallback"


def chunked_desc(w, width, prior, counts):
    chunk, mx = w.lens_args
    return (f"{w.name}: {w.num_seqs} prompt chunks of {chunk} tokens after 0..{mx} cached "
            f"chunks each (seeded; cached tokens {min(prior)}..{max(prior)}), "
            f"{w.num_q_heads} q / {w.num_kv_heads} kv heads, head_dim {w.head_dim}, "
            f"{str(w.dtype).replace('torch.', '')}, block {w.block_size}, {w.num_blocks}-block "
            f"pool, blocks scattered by a seeded permutation, table width {width}, "
            f"causal within each chunk, q/K/V ~ N(0,1)")


def cpu_baseline_chunked(pool, w, lens, tables, counts, qs, fetch, q, key, value, slots,
                         seqs=None):
    """The fp64 oracle's chunked step (write of the chunk rows, multi-query
    attention) over ``seqs`` (default: the whole batch), split by sequence
    over the pool's workers."""
    seqs = list(range(len(lens))) if seqs is None else list(seqs)
    work = {s: counts[s] * lens[s] for s in seqs}
    parts = split_by_work(seqs, work, len(pool))
    pool.load(oracle_jobs(w, "chunked", parts, tables, lens, [], fetch, q, key, value,
                          slots.tolist() if torch.is_tensor(slots) else slots, row_start=qs))
    wall, busy = pool.run()
    fl = chunked_flops(w, [lens[s] for s in seqs], [counts[s] for s in seqs])
    return {"value": fl / wall / 1e12, "unit": "TFLOP/s", "cores": len(parts), "kind": "oracle",
            "cpu": f"{cpu_model()}, {os.cpu_count()} logical cores",
            "sample": f"fp64 oracle (torch CPU ops) write + chunked attention of {len(seqs)} of "
                      f"{len(lens)} sequences ({sum(counts[s] for s in seqs)} query rows), split "
                      f"by sequence over {len(parts)} worker processes with one torch thread "
                      f"each, {wall:.2f} s wall ({sum(busy):.1f} s busy)"}


def run_native_chunked(a, world, rank, local):
    import paged_kv_cache_117_gb300 as pkv
    from paged_kv_cache_117_gb300 import build as pbuild
    if rank == 0:
        pbuild.build()
    barrier(world)
    pkv.load()
    assert torch.cuda.is_available(), "the native benchmark needs a GPU"
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = wl.WORKLOADS[a.workload]
    lens, tables, width, slots_cpu, counts, qs, desc = build_multiquery_step(w)
    T = qs[-1]
    k, v = wl.make_pool_chunked(w, dev)
    g = torch.Generator(device=dev)
    g.manual_seed(w.seed + 3000)
    q = torch.randn((T, w.num_q_heads, w.head_dim), generator=g, device=dev).to(w.dtype)
    key, value = wl.make_rows(w, 0, T, dev)
    tab_cpu = wl.pad_tables(tables, width)
    lens_cpu = torch.tensor(lens, dtype=torch.int32)
    qs_cpu = torch.tensor(qs, dtype=torch.int32)
    tab, lens_t, qs_t, slots = (x.to(dev) for x in (tab_cpu, lens_cpu, qs_cpu, slots_cpu))
    maxq = max(counts)
    out = torch.empty((T, w.num_q_heads, w.head_dim), dtype=w.dtype, device=dev)
    flush = L2Flush(dev)
    flops = chunked_flops(w, lens, counts)
    # a mixed batch goes through paged_attention_mixed: decode rows on the
    # decode kernel, chunks on the tensor cores
    mixed = w.lens_kind == "mixed"
    ws = None
    if mixed:
        ws = torch.empty(max(16, pkv.paged_attention_workspace_bytes(
            len(lens), w.num_q_heads, w.head_dim, width * w.block_size, w.partition_tokens)),
            dtype=torch.uint8, device=dev)

    def attend(o, qq, tb, ln, qsx, single=False):
        if mixed and not single:
            pkv.paged_attention_mixed(o, qq, k, v, tb, ln, qsx, w.scale, max_query_len=maxq,
                                      p_format=a.p_format, partition_tokens=w.partition_tokens,
                                      workspace=ws)
        else:
            pkv.paged_attention_chunked(o, qq, k, v, tb, ln, qsx, w.scale, max_query_len=maxq,
                                        p_format=a.p_format)

    cpu = None
    if rank == 0 and world == 1 and not a.no_cpu_baseline:
        pool = OraclePool(min(len(lens), a.cpu_workers or os.cpu_count() or 1))
        try:
            cpu = cpu_baseline_chunked(pool, w, lens, tables, counts, qs, device_fetch(k, v),
                                       q, key, value, slots_cpu)
        finally:
            pool.close()

    stream = torch.cuda.current_stream(dev)
    ev = lambda: torch.cuda.Event(enable_timing=True)

    def step(d0=None, d1=None):
        pkv.paged_kv_write(key, value, k, v, slots)
        if d0 is not None:
            d0.record(stream)
        attend(out, q, tab, lens_t, qs_t)
        if d1 is not None:
            d1.record(stream)

    for _ in range(max(3, a.warmup)):
        flush()
        step()
    torch.cuda.synchronize()
    assert pkv.read_device_flags(clear=True) == 0
    K = a.steps
    evs = [(ev(), ev(), ev(), ev()) for _ in range(K)]
    sampler = ClockSampler(torch.cuda.current_device())
    sampler.start()
    time.sleep(0.3)
    barrier(world)
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    host_head_start()
    for s0, s1, d0, d1 in evs:
        flush()
        s0.record(stream)
        step(d0, d1)
        s1.record(stream)
    torch.cuda.synchronize()
    barrier(world)
    wall = time.perf_counter() - t0
    clocks = sampler.stop()
    step_ms = max_over_ranks(world, sum(s0.elapsed_time(s1) for s0, s1, _, _ in evs) / K, dev)
    dec_ms = max_over_ranks(world, sum(d0.elapsed_time(d1) for _, _, d0, d1 in evs) / K, dev)

    # end to end: q, the chunk's K/V rows, tables, lengths, query_start and
    # slots in one pinned host buffer -> one H2D copy; the output back in one
    parts_cpu = [q.cpu(), key.cpu(), value.cpu(), tab_cpu, lens_cpu, qs_cpu, slots_cpu]
    sizes = [t.numel() * t.element_size() for t in parts_cpu]
    offs = [0]
    for n in sizes:
        offs.append(offs[-1] + (n + 255) // 256 * 256)
    h_in = torch.empty(offs[-1], dtype=torch.uint8).pin_memory()
    d_in = torch.empty(offs[-1], dtype=torch.uint8, device=dev)
    for t, o, n in zip(parts_cpu, offs, sizes):
        h_in[o:o + n].copy_(t.contiguous().view(torch.uint8).view(-1))
    e_q, e_key, e_val, e_tab, e_lens, e_qs, e_slots = (
        d_in[o:o + n].view(t.dtype).view(t.shape) for t, o, n in zip(parts_cpu, offs, sizes))
    h_out = torch.empty(out.shape, dtype=out.dtype).pin_memory()

    def e2e_step():
        d_in.copy_(h_in, non_blocking=True)
        pkv.paged_kv_write(e_key, e_val, k, v, e_slots)
        attend(out, e_q, e_tab, e_lens, e_qs)
        h_out.copy_(out, non_blocking=True)

    for _ in range(3):
        e2e_step()
    e2e_evs = [(ev(), ev()) for _ in range(K)]
    barrier(world)
    torch.cuda.synchronize()
    host_head_start()
    for e0, e1 in e2e_evs:
        flush()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_ms = max_over_ranks(world, sum(e0.elapsed_time(e1) for e0, e1 in e2e_evs) / K, dev)
    assert pkv.read_device_flags(clear=True) == 0

    peak, kind = peak_bf16()
    achieved = flops / (dec_ms * 1e-3) / 1e12
    value_tf = world * flops / (step_ms * 1e-3) / 1e12
    roof = {"kernel": "paged_attention_chunked (tcgen05)", "bound": "tensor",
            "achieved": round(achieved, 1), "peak": peak,
            "peak_kind": f"{kind} bf16_tflops (burst)", "unit": "TFLOP/s",
            "frac": round(achieved / peak, 4),
            "traffic": measured_traffic(w.name, 0, "chunked_kernel_prefill.md", CHUNKED_SOURCES)}
    extra = {}
    if mixed:
        # the share of the SMs the work list gave the decode rows in the last
        # call (word 2 of the workspace's control block: decoders that ran,
        # three to an SM when the passes run side by side)
        torch.cuda.synchronize()
        ctrl = ws[:16].view(torch.int32).cpu().tolist()
        side_by_side = w.num_q_heads // w.num_kv_heads <= 8 and maxq >= 2
        decode_sms = ctrl[2] // 3 if side_by_side else None
        # the same batch in one paged_attention_chunked launch, for comparison
        sev = [(ev(), ev()) for _ in range(K)]
        host_head_start()
        for e0, e1 in sev:
            flush()
            e0.record(stream)
            attend(out, q, tab, lens_t, qs_t, single=True)
            e1.record(stream)
        torch.cuda.synchronize()
        single_ms = sum(e0.elapsed_time(e1) for e0, e1 in sev) / K
        # the call's floor: the decode rows' bytes at the HBM peak plus the
        # chunks' flops at the bf16 peak
        n_dec = w.lens_args[0]
        hbm, hkind = peak_hbm()
        dec_bytes = algorithmic_bytes(w, lens[:n_dec], width, w.partition_tokens,
                                      out.element_size())["attention"]
        ch_flops = chunked_flops(w, lens[n_dec:], counts[n_dec:])
        floor_ms = 1e3 * (dec_bytes / (hbm * 1e9) + ch_flops / (peak * 1e12))
        roof = {"kernel": "paged_attention_mixed (decode rows: decode kernel, HBM; chunks: "
                          "tcgen05 kernel, tensor)", "bound": "hbm+tensor",
                "achieved": round(floor_ms / dec_ms, 4), "peak": 1.0,
                "peak_kind": f"time floor {floor_ms * 1e3:.1f} us = decode rows' "
                             f"{dec_bytes} B at the {hkind} {hbm} GB/s + chunks' {ch_flops} "
                             f"FLOP at the {kind} {peak} TFLOP/s", "unit": "floor / time",
                "frac": round(floor_ms / dec_ms, 4), "traffic": None}
        extra = {"decode_sms": decode_sms,
                 "sms": torch.cuda.get_device_properties(dev).multi_processor_count,
                 "single_chunked_call_ms": round(single_ms, 4),
                 "speedup_vs_single_chunked_call": round(single_ms / dec_ms, 3),
                 "decode_rows": n_dec, "decode_bytes": dec_bytes, "chunk_flops": ch_flops}
    return {
        "metric": CHUNK_METRIC, "value": round(value_tf, 2), "unit": "TFLOP/s", "n_gpus": world,
        "steps": K, "warmup": max(3, a.warmup), "ms_per_step": round(step_ms, 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": desc, "out_dtype": "bfloat16", "p_format": a.p_format,
                   "l2": L2_NOTE,
                   "parallelism": f"replicas x{world} (independent batches, no collective)"},
        "tokens_per_s": round(world * T / (step_ms * 1e-3), 1),
        "attention_ms": round(dec_ms, 4),
        "flops_per_step": flops,
        "roofline": roof,
        **extra,
        "e2e": {"value": round(world * flops / (e2e_ms * 1e-3) / 1e12, 2), "unit": "TFLOP/s",
                "ms_per_step": round(e2e_ms, 4), "h2d_bytes_per_step": sum(sizes),
                "d2h_bytes_per_step": h_out.numel() * h_out.element_size()},
        "gpu_launches": (4 if mixed else 2) * K,
        "clocks": clocks,
        "wall_s_timed": round(wall, 4),
        "cpu_baseline": cpu,
        **({"host_manager": prefix_manager_cost(w)} if w.lens_kind == "prefix" else {}),
    }


def prefix_manager_cost(w, rounds=20):
    """Host time of the library's prefix-cache manager per request of the
    prefix workload: the prompt's lookup (the chained SHA-256 key of each full
    block, then the key map), the append of its own tokens and its release,
    through the Python binding, on a cache that holds the system prompts.

    Two costs are reported.  ``miss``: every round brings requests with fresh
    (seeded) questions, so each request finds only its system prompt cached
    and allocates blocks for its own tokens, evicting cached blocks of earlier
    rounds from the free queue.  ``hit``: the same requests again right after,
    when their question blocks are cached too.  ``us_per_request`` is the miss
    cost (a new request's)."""
    import paged_kv_cache_117_gb300 as pkv
    plan = wl.prefix_plan(w)
    n_sys, _, q_len = w.lens_args
    pc = pkv.PrefixCache(w.num_blocks, w.block_size, wl.free_block_order(w))
    for i, sysp in enumerate(plan.systems):
        sid = len(plan.prompts) + i
        warm = sysp + [0]
        c = pc.add_sequence(sid, warm)
        pc.append(sid, warm[c:])
        pc.free_sequence(sid)
    systems = [torch.tensor(sp, dtype=torch.int32) for sp in plan.systems]
    g = torch.Generator().manual_seed(w.seed + 7000)
    R = len(plan.prompts)

    def admit(prompts):
        t0 = time.perf_counter()
        cached = 0
        for r, p_ in enumerate(prompts):
            c = pc.add_sequence(r, p_)
            pc.append(r, p_[c:])
            cached += c
        for r in range(R):
            pc.free_sequence(r)
        return time.perf_counter() - t0, cached

    t_miss = t_hit = 0.0
    c_miss = c_hit = 0
    for _ in range(rounds):
        qs = torch.randint(0, 32000, (R, q_len), generator=g, dtype=torch.int32)
        prompts = [torch.cat([systems[r % n_sys], qs[r]]) for r in range(R)]
        dt, c = admit(prompts)
        t_miss, c_miss = t_miss + dt, c_miss + c
        dt, c = admit(prompts)
        t_hit, c_hit = t_hit + dt, c_hit + c
    miss = t_miss / (rounds * R) * 1e6
    hit = t_hit / (rounds * R) * 1e6
    return {"us_per_request": round(miss, 1), "us_per_request_miss": round(miss, 1),
            "us_per_request_hit": round(hit, 1), "requests": R,
            "prompt_tokens": len(plan.prompts[0]),
            "cached_tokens_per_request_miss": c_miss // (rounds * R),
            "cached_tokens_per_request_hit": c_hit // (rounds * R), "cpu": cpu_model(),
            "what": "lookup + append + free per request, host C++ through the binding; miss: "
                    "fresh questions (only the system prompt cached; blocks allocated and "
                    "older cached blocks evicted), hit: the same requests again (all full "
                    "blocks cached); us_per_request is the miss cost"}


class OracleManager:
    """The oracle's block manager behind the library manager's calls
    (append of several sequences, tables as lists), for the reference arm,
    which runs no library code."""

    def __init__(self, num_blocks, block_size, free_order=None):
        from oracle.block_manager import BlockManager
        self.bm = BlockManager(num_blocks, block_size, free_order)

    def add_sequence(self, seq):
        self.bm.add_sequence(seq)

    def fork(self, parent, child):
        self.bm.fork(parent, child)

    def free_sequence(self, seq):
        self.bm.free_sequence(seq)

    def append(self, seqs):
        slots, pairs = [], []
        for s in seqs:
            slot, cow = self.bm.append(int(s))
            slots.append(slot)
            if cow is not None:
                pairs.append(list(cow))
        return (torch.tensor(slots, dtype=torch.int64),
                torch.tensor(pairs, dtype=torch.int64).reshape(-1, 2))

    def append_tokens(self, seq, count):
        return self.append([seq] * int(count))

    def table(self, seq):
        return list(self.bm.tables[seq]), self.bm.lens[seq]


def host_pool_fetch(w, ids, seed):
    """K/V values for the pool blocks ``ids`` only, N(0,1) on the host (the
    reference arm touches no GPU); returns a fetch(ids) over them."""
    g = torch.Generator().manual_seed(seed)
    shape = (len(ids), w.block_size, w.num_kv_heads, w.head_dim)
    kc = torch.randn(shape, generator=g).to(w.dtype)
    vc = torch.randn(shape, generator=g).to(w.dtype)
    pos = {b: i for i, b in enumerate(ids)}

    def fetch(sub):
        idx = torch.tensor([pos[b] for b in sub], dtype=torch.int64)
        return kc[idx], vc[idx]
    return fetch


def reference_line(metric, unit, val, ms, a, world, desc, cores, sample, digits):
    return {"impl": "reference", "metric": metric, "value": round(val, digits), "unit": unit,
            "n_gpus": world, "steps": a.steps, "warmup": max(3, a.warmup),
            "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": desc},
            "cpu_baseline": {"value": round(val, digits), "unit": unit, "cores": cores,
                             "kind": "oracle", "sample": sample},
            "e2e": {"value": round(val, digits), "unit": unit, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}


def run_reference(a, world, rank, local):
    """The fp64 CPU oracle as it stands: each step is the oracle's decode step
    (copies, KV write, attention) of the whole batch, split by sequence over
    worker processes on the host's cores."""
    if rank != 0:
        return None
    w = select_workload(a)
    if w.lens_kind == "shared":
        lens, tables, width, slots, pairs, _ = build_shared_step(w, OracleManager)
    elif w.lens_kind == "beam":
        lens, tables, width, slots, pairs, _ = build_beam_step(w, OracleManager)
    else:
        lens, tables, width, slots = build_metadata(w, manager="oracle")
        pairs = torch.zeros((0, 2), dtype=torch.int64)
    pairs = [tuple(p) for p in pairs.tolist()]
    ids = sorted({b for t in tables for b in t} | {p[0] for p in pairs})
    fetch = host_pool_fetch(w, ids, w.seed + 2000)
    q, key, value = wl.make_step_inputs(w, "cpu")
    pool = OraclePool(a.cpu_workers or os.cpu_count() or 1)
    try:
        parts = split_by_work(range(len(lens)), lens, len(pool))
        pool.load(oracle_jobs(w, "decode", parts, tables, lens, pairs, fetch, q, key, value,
                              slots.tolist()))
        times = []
        for i in range(max(3, a.warmup) + a.steps):
            wall, _ = pool.run()
            if i >= max(3, a.warmup):
                times.append(wall)
    finally:
        pool.close()
    nbytes = algorithmic_bytes(w, lens, width, 0, w.elem_bytes, len(pairs))["step"]
    ms = 1e3 * sum(times) / len(times)
    val = nbytes / (ms * 1e-3) / 1e9
    sample = (f"fp64 oracle step of all {len(lens)} sequences ({len(pairs)} block copies, KV "
              f"write, attention; {nbytes / 1e6:.1f} MB algorithmic) per step, split by sequence "
              f"over {len(parts)} worker processes with one torch thread each")
    return reference_line(METRIC, UNIT, val, ms, a, world, workload_desc(w, width), len(parts),
                          sample, 4)


def subchunk_jobs(w, seq, lens, tables, counts, qs, fetch, q, key, value, slots, n):
    """One sequence's chunk split by query rows into about n jobs of equal
    work: rows a..b-1 of a chunk of c rows in a sequence of L tokens are the
    last b - a rows of a sequence of L - c + b tokens, so each job is the
    oracle's chunked call on that shorter sequence (its write covers rows
    0..b-1 of the chunk, which those queries see)."""
    L, c, r0 = lens[seq], counts[seq], qs[seq]
    first = L - c                      # position of chunk row 0
    total = sum(first + i + 1 for i in range(c))
    bounds, acc, a0 = [], 0, 0
    for i in range(c):
        acc += first + i + 1
        if acc >= total * (len(bounds) + 1) / n or i == c - 1:
            bounds.append((a0, i + 1))
            a0 = i + 1
    ids = sorted(set(tables[seq]))
    remap = {b: i for i, b in enumerate(ids)}
    kc, vc = fetch(ids)
    B = w.block_size
    jobs = []
    for a_, b_ in bounds:
        rows = list(range(r0, r0 + b_))
        jobs.append({"kind": "chunked", "k": kc, "v": vc, "scale": w.scale, "pairs": [],
                     "key": key[rows].cpu(), "value": value[rows].cpu(),
                     "slots": [remap[int(slots[r]) // B] * B + int(slots[r]) % B for r in rows],
                     "q": q[r0 + a_:r0 + b_].cpu(), "tables": [[remap[x] for x in tables[seq]]],
                     "lens": [first + b_], "qs": [0, b_ - a_]})
    return jobs


def run_reference_chunked(a, world, rank, local):
    """The fp64 CPU oracle on a chunked workload: each step is the shortest
    sequence's chunk (write + multi-query attention), split by query rows
    over worker processes on the host's cores (the whole batch would take
    the oracle tens of seconds per step)."""
    if rank != 0:
        return None
    w = wl.WORKLOADS[a.workload]
    lens, tables, width, slots, counts, qs, desc = build_multiquery_step(w, OracleManager)
    multi = [s for s in range(len(lens)) if counts[s] > 1] or list(range(len(lens)))
    seq = min(multi, key=lambda s: lens[s])
    fetch = host_pool_fetch(w, sorted(set(tables[seq])), w.seed + 2000)
    T = qs[-1]
    g = torch.Generator().manual_seed(w.seed + 3000)
    q = torch.randn((T, w.num_q_heads, w.head_dim), generator=g).to(w.dtype)
    key, value = wl.make_rows(w, 0, T)
    pool = OraclePool(a.cpu_workers or os.cpu_count() or 1)
    try:
        jobs = subchunk_jobs(w, seq, lens, tables, counts, qs, fetch, q, key, value,
                             slots.tolist(), len(pool))
        pool.load(jobs)
        times = []
        for i in range(max(3, a.warmup) + a.steps):
            wall, _ = pool.run()
            if i >= max(3, a.warmup):
                times.append(wall)
    finally:
        pool.close()
    fl = chunked_flops(w, [lens[seq]], [counts[seq]])
    ms = 1e3 * sum(times) / len(times)
    val = fl / (ms * 1e-3) / 1e12
    sample = (f"fp64 oracle write + chunked attention of sequence {seq} per step "
              f"({counts[seq]} queries over {lens[seq]} tokens), split by query rows over "
              f"{len(jobs)} worker processes with one torch thread each")
    return reference_line(CHUNK_METRIC, "TFLOP/s", val, ms, a, world, desc, len(jobs), sample, 6)


def main():
    a = parse_args()
    world, rank, local = dist_init()
    chunked = wl.WORKLOADS[a.workload].lens_kind in MULTIQUERY
    if chunked and (a.seqs is not None or a.context is not None):
        raise SystemExit("--seqs / --context apply to the decode workloads of independent "
                         "sequences (tiny, opt13b, llama8b, qwen72b)")
    if a.impl == "reference":
        res = (run_reference_chunked if chunked else run_reference)(a, world, rank, local)
    else:
        res = (run_native_chunked if chunked else run_native)(a, world, rank, local)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
