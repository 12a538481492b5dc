"""Seeded synthetic inputs for the paged decode path.

This module is the one place both sides draw their inputs from: the parity
tests feed what it makes to the fp64 oracle and to the CUDA library alike, and
the benchmark uses it to build its batches.  It holds shapes, seeds and value
distributions only -- none of the method's arithmetic (no attention, no block
table walk, no reference counting).

The five workloads follow the shapes the pages use for their examples:

* ``tiny``     -- 4-token blocks as in "PagedAttention" (tensortonic), section 3
                  "Dividing the Cache into Small Blocks"; lengths 1, 6, 9, 17 so
                  that 9 and 17 open a fresh block.
* ``opt13b``   -- OPT-13B, 40 heads x 128 (5120 hidden), fp16, as sized in
                  "PagedAttention: Virtual Memory for the KV Cache", section
                  "The problem: serving throughput is memory-bound".
* ``llama8b``  -- Llama 3.1 8B, 32 query / 8 KV heads x 128, bf16, 16-token
                  blocks ("PagedAttention and vLLM: Paging the KV Cache Like an
                  OS", Step 3).
* ``qwen72b``  -- Qwen2.5-72B, 64 query / 8 KV heads x 128, 8k context
                  ("vLLM's PagedAttention: How Memory Management Supports Large
                  Model Inference", section 2.1).
* ``shared``   -- parallel sampling from shared prompts ("PagedAttention and
                  vLLM ...", Step 4): 16 prompts of 1,000 tokens, 8 samples each.
* ``beam``     -- beam search over shared prompts (same Step 4): 32 prompts of
                  1,000 tokens, 8 beams each, seeded scores in place of a model.
* ``prefill``  -- chunked prefill ("Paging the KV Cache Like an OS", continuous
                  batching): 16 prompt chunks of 512 tokens after 0..15 cached
                  chunks each.
* ``prefix``   -- prefix caching (same page, section 2.4): 32 requests over 2
                  cached 2,048-token system prompts, each prefilling its own
                  256-token question.
* ``mixed``    -- a continuous-batching step (same page, continuous batching):
                  the ``llama8b`` decode batch plus 8 prompt chunks of 512
                  tokens.

The pages measure on ShareGPT/Alpaca traces; none is used or reproduced here.
Lengths come from the seeded distributions below instead.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field, replace
from typing import List, Optional, Sequence, Tuple

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    num_seqs: int
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    dtype: torch.dtype
    partition_tokens: int          # 0 = one partition per sequence
    seed: int
    lens_kind: str                 # "fixed" | "uniform" | "lognormal" | "shared" | "beam" | "chunked" | "prefix" | "mixed"
    lens_args: tuple = field(default_factory=tuple)

    @property
    def group(self) -> int:
        return self.num_q_heads // self.num_kv_heads

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.head_dim)

    @property
    def elem_bytes(self) -> int:
        return torch.tensor([], dtype=self.dtype).element_size()


# seed = 117 + the workload's position in the list below (1-based)
TINY = Workload("tiny", 4, 4, 4, 64, 4, 64, torch.bfloat16, 0, 118,
                "fixed", (1, 6, 9, 17))
OPT13B = Workload("opt13b", 64, 40, 40, 128, 16, 10_000, torch.float16, 1024, 119,
                  "uniform", (128, 2048))
LLAMA8B = Workload("llama8b", 256, 32, 8, 128, 16, 40_000, torch.bfloat16, 768, 120,
                   "lognormal", (1024.0, 0.8, 16, 8192))
QWEN72B = Workload("qwen72b", 32, 64, 8, 128, 16, 20_480, torch.bfloat16, 512, 121,
                   "fixed", (8192,) * 32)
SHARED = Workload("shared", 128, 32, 8, 128, 16, 4_096, torch.bfloat16, 512, 122,
                  "shared", (16, 1000, 8, 0, 200))

# Beam search over shared prompts ("PagedAttention and vLLM ...", Step 4, beam
# search): 32 prompts of 1,000 tokens, 8 beams each, 20 decode steps before the
# measured one (so that the measured token lands in a partly filled block and
# copy-on-write copies happen in it).  Scores come from a seeded generator
# (there is no model): every beam proposes 2 continuations and the 8
# best-scoring ones survive.
BEAM = Workload("beam", 256, 32, 8, 128, 16, 8_192, torch.bfloat16, 512, 123,
                "beam", (32, 1000, 8, 2, 20))

# Chunked prefill ("Paging the KV Cache Like an OS", continuous batching): a
# step's budget of 8,192 tokens filled with 512-token prompt chunks of 16
# sequences, each of which already holds 0..15 earlier chunks of its prompt
# (seeded), Llama-3.1-8B heads.
PREFILL = Workload("prefill", 16, 32, 8, 128, 16, 16_384, torch.bfloat16, 0, 124,
                   "chunked", (512, 15))

# Prefix caching ("Paging the KV Cache Like an OS", section 2.4 and summary
# point 5): 32 requests share one of 2 system prompts of 2,048 tokens and add a
# 256-token question of their own; the system prompts were prefilled (and
# their blocks cached) by earlier requests, so each request prefills only its
# question, attending over 2,304 tokens.  Token ids are seeded.
PREFIX = Workload("prefix", 32, 32, 8, 128, 16, 16_384, torch.bfloat16, 0, 125,
                  "prefix", (2, 2048, 256))

# A continuous-batching step ("Paging the KV Cache Like an OS", continuous
# batching: every waiting decode goes into the step, prefill chunks fill the
# rest of the token budget): the Llama-3.1-8B decode batch (256 sequences,
# lognormal lengths as in ``llama8b``) plus 8 prompt chunks of 512 tokens
# after 0..7 cached chunks each.
MIXED = Workload("mixed", 264, 32, 8, 128, 16, 40_000, torch.bfloat16, 768, 126,
                 "mixed", (256, 1024.0, 0.8, 16, 8192, 8, 512, 7))

WORKLOADS = {w.name: w for w in (TINY, OPT13B, LLAMA8B, QWEN72B, SHARED, BEAM, PREFILL, PREFIX,
                                 MIXED)}


def scaled(w: Workload, num_seqs: int, max_len: Optional[int] = None,
           num_blocks: Optional[int] = None) -> Workload:
    """A smaller copy of a workload (same heads, dims, dtype, distribution)."""
    args = w.lens_args
    if max_len is not None and w.lens_kind == "uniform":
        args = (min(args[0], max_len), min(args[1], max_len))
    elif max_len is not None and w.lens_kind == "lognormal":
        args = (min(args[0], max_len / 2), args[1], min(args[2], max_len), max_len)
    elif max_len is not None and w.lens_kind == "fixed":
        args = tuple(min(a, max_len) for a in args[:num_seqs])
    return replace(w, num_seqs=num_seqs, lens_args=args,
                   num_blocks=num_blocks if num_blocks is not None else w.num_blocks)


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def context_lens(w: Workload) -> List[int]:
    """Per-sequence context length L_s, counting the token written this step."""
    g = _gen(w.seed)
    if w.lens_kind == "fixed":
        lens = list(w.lens_args)[: w.num_seqs]
        assert len(lens) == w.num_seqs
        return [int(x) for x in lens]
    if w.lens_kind == "uniform":
        lo, hi = w.lens_args
        return [int(x) for x in torch.randint(lo, hi + 1, (w.num_seqs,), generator=g)]
    if w.lens_kind == "lognormal":
        median, sigma, lo, hi = w.lens_args
        z = torch.randn(w.num_seqs, generator=g, dtype=torch.float64)
        raw = torch.exp(math.log(median) + sigma * z)
        return [int(min(max(round(float(x)), lo), hi)) for x in raw]
    raise ValueError(f"{w.name}: lengths come from shared_prefix_plan()")


@dataclass(frozen=True)
class SharedPlan:
    """Parallel-sampling layout: ``n`` samples fork from each prompt and then
    append ``own[i]`` tokens of their own before the timed step."""
    prompts: int
    prompt_len: int
    samples: int
    own: List[int]           # own-token count per sequence (prompt-major order)


def shared_prefix_plan(w: Workload) -> SharedPlan:
    prompts, prompt_len, n, lo, hi = w.lens_args
    g = _gen(w.seed)
    own = [int(x) for x in torch.randint(lo, hi + 1, (prompts * n,), generator=g)]
    # Samples 0 and 1 of every prompt keep zero own tokens so that the timed
    # step's write lands in the still-shared partial prompt block (copy by the
    # first writer, in-place write by the last remaining sharer).
    for p in range(prompts):
        own[p * n + 0] = 0
        own[p * n + 1] = 0
    return SharedPlan(prompts, prompt_len, n, own)


def free_block_order(w: Workload) -> List[int]:
    """Order in which free physical blocks are handed out: a seeded random
    permutation of the pool, so logically adjacent blocks land far apart."""
    g = _gen(w.seed + 1000)
    return [int(x) for x in torch.randperm(w.num_blocks, generator=g)]


def make_pool(w: Workload, device="cpu"):
    """k_cache, v_cache of shape [num_blocks, block_size, num_kv_heads, head_dim],
    every slot filled with seeded N(0,1) values (no slot is left undefined)."""
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 2000)
    k = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(w.dtype)
    v = torch.randn(shape, generator=g, device=device, dtype=torch.float32).to(w.dtype)
    return k, v


def make_pool_chunked(w: Workload, device):
    """Same distribution as make_pool, generated in slabs so that the fp32
    temporaries stay small for multi-GB pools (values differ from make_pool)."""
    shape = (w.num_blocks, w.block_size, w.num_kv_heads, w.head_dim)
    k = torch.empty(shape, dtype=w.dtype, device=device)
    v = torch.empty(shape, dtype=w.dtype, device=device)
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 2000)
    step = max(1, (64 << 20) // (w.block_size * w.num_kv_heads * w.head_dim * 4))
    for t in (k, v):
        for i in range(0, w.num_blocks, step):
            j = min(w.num_blocks, i + step)
            t[i:j] = torch.randn((j - i,) + shape[1:], generator=g, device=device,
                                 dtype=torch.float32).to(w.dtype)
    return k, v


def make_step_inputs(w: Workload, device="cpu"):
    """This step's query q[S, Hq, D] and new key/value [S, Hkv, D], N(0,1)."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 3000)
    q = torch.randn((w.num_seqs, w.num_q_heads, w.head_dim), generator=g,
                    device=device, dtype=torch.float32).to(w.dtype)
    key = torch.randn((w.num_seqs, w.num_kv_heads, w.head_dim), generator=g,
                      device=device, dtype=torch.float32).to(w.dtype)
    value = torch.randn((w.num_seqs, w.num_kv_heads, w.head_dim), generator=g,
                        device=device, dtype=torch.float32).to(w.dtype)
    return q, key, value


def pad_tables(tables: Sequence[Sequence[int]], width: Optional[int] = None,
               fill: int = 0) -> torch.Tensor:
    """Pack per-sequence block lists into an int32 [S, width] tensor."""
    width = width if width is not None else max(1, max((len(t) for t in tables), default=1))
    out = torch.full((len(tables), width), fill, dtype=torch.int32)
    for i, t in enumerate(tables):
        if len(t):
            out[i, : len(t)] = torch.tensor(list(t), dtype=torch.int32)
    return out


def chunk_plan(w: Workload):
    """(prior tokens, this step's query tokens) per sequence of a chunked
    prefill workload, or of a mixed one (decode sequences first: L_s - 1
    earlier tokens and one new token each; then the prompt chunks)."""
    if w.lens_kind == "mixed":
        n_dec, median, sigma, lo, hi, n_chunk, chunk, max_prior = w.lens_args
        g = _gen(w.seed)
        z = torch.randn(n_dec, generator=g, dtype=torch.float64)
        lens = [int(min(max(round(float(x)), lo), hi)) for x in torch.exp(math.log(median) + sigma * z)]
        prior = (torch.randint(0, max_prior + 1, (n_chunk,), generator=g) * chunk).tolist()
        return [L - 1 for L in lens] + [int(x) for x in prior], [1] * n_dec + [chunk] * n_chunk
    chunk, max_prior = w.lens_args
    g = _gen(w.seed)
    prior = (torch.randint(0, max_prior + 1, (w.num_seqs,), generator=g) * chunk).tolist()
    return [int(x) for x in prior], [chunk] * w.num_seqs


@dataclass(frozen=True)
class PrefixPlan:
    systems: List[List[int]]        # token ids of each system prompt
    prompts: List[List[int]]        # each request's prompt (system + question)


def prefix_plan(w: Workload) -> PrefixPlan:
    n_sys, sys_len, q_len = w.lens_args
    g = _gen(w.seed)
    systems = torch.randint(0, 32000, (n_sys, sys_len), generator=g).tolist()
    questions = torch.randint(0, 32000, (w.num_seqs, q_len), generator=g).tolist()
    return PrefixPlan(systems, [systems[r % n_sys] + questions[r] for r in range(w.num_seqs)])


@dataclass(frozen=True)
class BeamPlan:
    requests: int
    prompt_len: int
    width: int
    cands: int
    # parents[t][r] = for step t and request r, the parent beam index (0..width-1)
    # of each of the `width` survivors, in survivor order
    parents: List[List[List[int]]]


def beam_plan(w: Workload, steps: Optional[int] = None) -> BeamPlan:
    requests, prompt_len, width, cands, n_steps = w.lens_args
    if steps is not None:
        n_steps = steps
    g = _gen(w.seed)
    parents = []
    for _ in range(n_steps + 1):            # history steps + the measured step
        per_req = []
        for _ in range(requests):
            scores = torch.rand(width * cands, generator=g, dtype=torch.float64)
            best = torch.topk(scores, width).indices.tolist()
            per_req.append([b // cands for b in best])
        parents.append(per_req)
    return BeamPlan(requests, prompt_len, width, cands, parents)


@dataclass(frozen=True)
class BeamStep:
    forks: List[Tuple[int, int]]    # (parent sequence, child sequence), in order
    frees: List[int]                # pruned sequences, freed after the forks
    order: List[int]                # surviving sequences, request-major; one token each


def beam_schedule(plan: BeamPlan) -> List[BeamStep]:
    """Sequence-level bookkeeping of a beam plan.  Request r starts as beam
    sequences r*width .. r*width+width-1, all forked from r*width after its
    prompt.  In a step, a parent's first surviving child keeps the parent's
    sequence id, every further child is a fork with a fresh id, and parents
    with no surviving child are freed."""
    R, W = plan.requests, plan.width
    beams = [[r * W + i for i in range(W)] for r in range(R)]
    next_id = R * W
    out = []
    for par_t in plan.parents:
        forks, frees = [], []
        for r in range(R):
            old, new, used = beams[r], [], set()
            for p in par_t[r]:
                if p in used:
                    forks.append((old[p], next_id))
                    new.append(next_id)
                    next_id += 1
                else:
                    used.add(p)
                    new.append(old[p])
            frees += [sq for p, sq in enumerate(old) if p not in used]
            beams[r] = new
        out.append(BeamStep(forks, frees, [sq for b in beams for sq in b]))
    return out


def make_rows(w: Workload, step: int, n: int, device="cpu"):
    """New key/value rows [n, Hkv, D] of history step `step`, N(0,1)."""
    g = torch.Generator(device=device)
    g.manual_seed(w.seed + 5000 + step)
    key = torch.randn((n, w.num_kv_heads, w.head_dim), generator=g, device=device,
                      dtype=torch.float32).to(w.dtype)
    value = torch.randn((n, w.num_kv_heads, w.head_dim), generator=g, device=device,
                        dtype=torch.float32).to(w.dtype)
    return key, value
