"""KV-cache sizing arithmetic (oracle; test infrastructure only).

* Bytes per token: one key and one value vector per layer and KV head --
  "PagedAttention: Virtual Memory for the KV Cache", section "The problem:
  serving throughput is memory-bound" (OPT-13B: 800 KB per token), and
  "vLLM's PagedAttention: How Memory Management Supports Large Model
  Inference", section 2.1 (Qwen2.5-72B: 327,680 bytes per token).
* Bytes per block: block_size times the per-token figure -- "Batching and
  PagedAttention", section "How PagedAttention virtualizes the KV cache" and
  its Quick Reference table.
* Blocks for n tokens: ceil(n / block_size), since a block is taken only when
  the previous one is full -- "PagedAttention and vLLM: Paging the KV Cache
  Like an OS", section "How much can still be wasted".
"""
from __future__ import annotations


def kv_bytes_per_token(num_layers: int, num_kv_heads: int, head_dim: int,
                       bytes_per_elem: int) -> int:
    return 2 * num_layers * num_kv_heads * head_dim * bytes_per_elem


def kv_bytes_per_block(block_size: int, num_layers: int, num_kv_heads: int,
                       head_dim: int, bytes_per_elem: int) -> int:
    return block_size * kv_bytes_per_token(num_layers, num_kv_heads, head_dim,
                                           bytes_per_elem)


def blocks_for_tokens(num_tokens: int, block_size: int) -> int:
    return -(-num_tokens // block_size)


def max_waste_slots(block_size: int) -> int:
    """Only the last block of an unshared, append-only sequence can be partly
    empty, and it holds at least one token."""
    return block_size - 1
