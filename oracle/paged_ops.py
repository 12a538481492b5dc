"""Write, copy and decode attention over a paged KV pool, in plain PyTorch CPU
ops (oracle; test infrastructure only).

Layout, as the library uses it:
  k_cache, v_cache : [num_blocks, block_size, num_kv_heads, head_dim]
  block_tables     : int32 [num_seqs, max_blocks]; row s lists the physical
                     block of each logical block of sequence s
  context_lens     : int32 [num_seqs]; L_s, counting this step's token
  q                : [num_seqs, num_q_heads, head_dim]
  key, value       : [num_tokens, num_kv_heads, head_dim]
  slot_mapping     : int64 [num_tokens]; slot = block * block_size + offset,
                     a negative slot means "skip this token"

Attention is the plain definition, computed in float64: the method reaches
ordinary attention exactly and only the addresses differ ("PagedAttention and
vLLM: Paging the KV Cache Like an OS", Step 5).  Softmax runs over all L_s
valid positions of the sequence at once, never per block ("PagedAttention"
(tensortonic), section 5), and the slots of the last block past L_s are not
read.  Query head hq uses KV head hq // (num_q_heads / num_kv_heads).
"""
from __future__ import annotations

from typing import Iterable, List, Sequence, Tuple

import torch


def write_kv(k_cache: torch.Tensor, v_cache: torch.Tensor, key: torch.Tensor,
             value: torch.Tensor, slot_mapping: Sequence[int]) -> None:
    """Store token t's key/value rows at (slot // B, slot % B), in place:
    the block and offset the token's slot names ("PagedAttention"
    (tensortonic), section 5).
    """
    B = k_cache.shape[1]
    for t, slot in enumerate(int(x) for x in slot_mapping):
        if slot < 0:
            continue
        blk, off = divmod(slot, B)
        k_cache[blk, off] = key[t]
        v_cache[blk, off] = value[t]


def copy_blocks(k_cache: torch.Tensor, v_cache: torch.Tensor,
                pairs: Iterable[Tuple[int, int]]) -> None:
    """Copy every slot of block src to block dst, keys and values, in place.

    The copy-on-write copy: the writer takes a fresh block and the tokens
    held so far are copied into it ("PagedAttention and vLLM ...", Step 4).
    The whole block is copied (all block_size slots).
    """
    for src, dst in pairs:
        k_cache[int(dst)] = k_cache[int(src)].clone()
        v_cache[int(dst)] = v_cache[int(src)].clone()


def gather_logical(cache: torch.Tensor, table: Sequence[int], length: int) -> torch.Tensor:
    """The sequence's first ``length`` tokens in logical order, [length, H, D],
    found by walking its block table ("PagedAttention" (tensortonic),
    section 4: logical block j lives in physical block table[j])."""
    B = cache.shape[1]
    rows = []
    for pos in range(length):
        rows.append(cache[int(table[pos // B]), pos % B])
    if not rows:
        return cache.new_zeros((0,) + tuple(cache.shape[2:]))
    return torch.stack(rows, 0)


def attend_one(q_heads: torch.Tensor, keys: torch.Tensor, values: torch.Tensor,
               scale: float) -> torch.Tensor:
    """Softmax attention of the query rows q_heads [G, D] over keys/values
    [L, D], float64.  L = 0 gives zeros (nothing to attend to)."""
    q64 = q_heads.to(torch.float64)
    if keys.shape[0] == 0:
        return torch.zeros_like(q64)
    k64 = keys.to(torch.float64)
    v64 = values.to(torch.float64)
    z = (q64 @ k64.T) * scale                       # [G, L]
    m = z.max(dim=1, keepdim=True).values
    w = torch.exp(z - m)
    return (w @ v64) / w.sum(dim=1, keepdim=True)


def attend(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
           block_tables, context_lens, scale: float) -> torch.Tensor:
    """Decode attention of every sequence over its paged context, float64
    [num_seqs, num_q_heads, head_dim]."""
    S, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    scale = float(torch.tensor(scale, dtype=torch.float32))   # the fp32 value
    out = torch.zeros((S, Hq, D), dtype=torch.float64)
    tables = block_tables.tolist() if torch.is_tensor(block_tables) else block_tables
    lens = context_lens.tolist() if torch.is_tensor(context_lens) else context_lens
    for s in range(S):
        L = int(lens[s])
        keys = gather_logical(k_cache, tables[s], L)
        vals = gather_logical(v_cache, tables[s], L)
        for h in range(Hkv):
            out[s, h * G:(h + 1) * G] = attend_one(q[s, h * G:(h + 1) * G],
                                                   keys[:, h], vals[:, h], scale)
    return out


def attend_contiguous(q: torch.Tensor, keys: List[torch.Tensor],
                      values: List[torch.Tensor], scale: float) -> torch.Tensor:
    """The same attention over per-sequence contiguous [L_s, Hkv, D] arrays."""
    S, Hq, D = q.shape
    Hkv = keys[0].shape[1]
    G = Hq // Hkv
    scale = float(torch.tensor(scale, dtype=torch.float32))
    out = torch.zeros((S, Hq, D), dtype=torch.float64)
    for s in range(S):
        for h in range(Hkv):
            out[s, h * G:(h + 1) * G] = attend_one(q[s, h * G:(h + 1) * G],
                                                   keys[s][:, h], values[s][:, h], scale)
    return out


def query_positions(context_len: int, num_queries: int) -> List[int]:
    """Positions of a chunk's queries: the sequence's last ``num_queries``
    tokens, so query i sits at context_len - num_queries + i."""
    if num_queries < 0 or num_queries > context_len:
        raise ValueError("a chunk cannot hold more queries than the sequence has tokens")
    return [context_len - num_queries + i for i in range(num_queries)]


def attend_chunked(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                   block_tables, context_lens, query_start, scale: float) -> torch.Tensor:
    """Multi-query attention over a paged context: chunked prefill, and decode
    as its one-query case ("Paging the KV Cache Like an OS", continuous
    batching: a long prompt is processed in chunks over several passes, each
    filling a few blocks, interleaved with other sequences' decode steps).

    q holds num_tokens query rows [num_tokens, Hq, D], packed by sequence:
    sequence s owns rows query_start[s] .. query_start[s+1]-1, its last n_s
    positions (their keys and values are already in the cache, so
    context_lens[s] = L_s counts them).  The query at position p attends to
    positions 0..p of its own sequence -- ordinary causal attention, which is
    what processing a prompt in pieces must reproduce.  float64
    [num_tokens, Hq, D]."""
    T, Hq, D = q.shape
    Hkv = k_cache.shape[2]
    assert Hq % Hkv == 0
    G = Hq // Hkv
    scale = float(torch.tensor(scale, dtype=torch.float32))   # the fp32 value
    tables = block_tables.tolist() if torch.is_tensor(block_tables) else block_tables
    lens = context_lens.tolist() if torch.is_tensor(context_lens) else context_lens
    starts = query_start.tolist() if torch.is_tensor(query_start) else query_start
    assert starts[0] == 0 and starts[-1] == T and len(starts) == len(lens) + 1
    out = torch.zeros((T, Hq, D), dtype=torch.float64)
    for s in range(len(lens)):
        L = int(lens[s])
        r0, n = int(starts[s]), int(starts[s + 1]) - int(starts[s])
        pos = query_positions(L, n)
        keys = gather_logical(k_cache, tables[s], L)
        vals = gather_logical(v_cache, tables[s], L)
        for i, p in enumerate(pos):
            for h in range(Hkv):
                out[r0 + i, h * G:(h + 1) * G] = attend_one(
                    q[r0 + i, h * G:(h + 1) * G], keys[: p + 1, h], vals[: p + 1, h], scale)
    return out
