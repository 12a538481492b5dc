"""Plain, slow CPU oracle for the paged KV cache decode path.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports this
directory; only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline
leg of ``bench.py`` may use it.  It shares no code with the CUDA library:
the two meet only in the seeded input generators
(``paged_kv_cache_117_gb300.workloads``), which hold no arithmetic of the
method.

Contents, each written from the pages' description:

* ``block_manager`` -- on-demand block allocation, reference counts and
  copy-on-write ("PagedAttention and vLLM: Paging the KV Cache Like an OS",
  Steps 3 and 4; "PagedAttention" (tensortonic), sections 3, 6 and 7).
* ``paged_ops`` -- the per-step K/V slot write, the block copy, and decode
  attention over the block table in fp64 ("PagedAttention and vLLM ...",
  Step 5; "PagedAttention" (tensortonic), section 5; the block-wise attention
  equation in "PagedAttention: Virtual Memory for the KV Cache"), and
  multi-query attention for chunked prefill mixed with decode
  (``attend_chunked``: each query attends causally to its own sequence's
  positions up to its own; "Paging the KV Cache Like an OS", continuous
  batching and chunked prefill).
* ``prefix_cache`` -- block pool with a prefix cache: chained SHA-256 block
  keys, a hash -> block map of full blocks, a free queue whose order is the
  eviction order ("PagedAttention and vLLM ...", section 2.4 and summary
  point 5).
* ``sizing`` -- KV bytes per token and per block ("PagedAttention: Virtual
  Memory for the KV Cache", memory-bound section; "Batching and
  PagedAttention", bytes-per-block formula).

Every function is pinned by ``tests/test_oracle_*.py`` against facts the pages
print, closed forms, a library attention routine and brute force on tiny
inputs.
"""
