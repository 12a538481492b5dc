"""GB300-native paged KV cache decode path (sm_103a CUDA library + binding).

The compute lives in ``libpaged_kv.so`` (built from ``csrc/`` by
``paged_kv_cache_117_gb300.build``); ``binding`` marshals torch tensors into
its C ABI.  ``workloads`` holds the seeded synthetic inputs.
"""
from .binding import (  # noqa: F401
    FLAG_BLOCK_RANGE, FLAG_LEN_RANGE, FLAG_PAIR_CONFLICT, FLAG_PAIR_RANGE, FLAG_SLOT_RANGE, FLAG_TIMEOUT, FLAG_V_RANGE,
    BlockManager, PrefixCache, chain_keys, sha256, EXPORTED_SYMBOLS, NOALLOC_SCRATCH_BYTES, PkvError, load,
    paged_attention_decode, paged_attention_decode_noalloc, paged_attention_decode_append,
    paged_attention_chunked, paged_attention_mixed,
    paged_attention_workspace_bytes, paged_block_copy, paged_kv_write, read_device_flags,
    block_copy_workspace, paged_block_copy_workspace_bytes,
)
