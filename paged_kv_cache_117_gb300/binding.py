"""Thin ctypes binding over the C ABI in ``include/paged_kv.h``.

Argument marshalling only: every step of the path runs in the CUDA library.
There is no fallback: if ``libpaged_kv.so`` is missing or fails to load, every
call raises.  Functions take CUDA tensors laid out as the header describes and
launch on the current torch stream (or the ``stream`` given).
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

_PKG_DIR = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG_DIR, "libpaged_kv.so")

PKV_F16, PKV_BF16, PKV_F32 = 0, 1, 2
_DTYPE_CODE = {torch.float16: PKV_F16, torch.bfloat16: PKV_BF16, torch.float32: PKV_F32}

FLAG_BLOCK_RANGE = 0x1
FLAG_SLOT_RANGE = 0x2
FLAG_PAIR_RANGE = 0x4
FLAG_LEN_RANGE = 0x8
FLAG_TIMEOUT = 0x10
FLAG_V_RANGE = 0x20
FLAG_PAIR_CONFLICT = 0x40

EXPORTED_SYMBOLS = (
    "paged_kv_write",
    "paged_block_copy",
    "paged_block_copy_ws",
    "paged_block_copy_workspace_bytes",
    "paged_attention_decode",
    "paged_attention_workspace_bytes",
    "pkv_status_string",
    "pkv_read_device_flags",
    "pkv_last_error_string",
    "paged_attention_decode_noalloc",
    "paged_attention_decode_append",
    "paged_attention_chunked",
    "paged_attention_mixed",
    "pkv_pc_create",
    "pkv_pc_add_sequence",
    "pkv_pc_append",
    "pkv_pc_free_sequence",
    "pkv_sha256",
    "pkv_bm_create", "pkv_bm_destroy", "pkv_bm_add_sequence", "pkv_bm_fork",
    "pkv_bm_free_sequence", "pkv_bm_append", "pkv_bm_table", "pkv_bm_num_free",
    "pkv_bm_refcount",
)

# Fixed scratch size of paged_attention_decode_noalloc (PKV_NOALLOC_SCRATCH_BYTES).
NOALLOC_SCRATCH_BYTES = 64 << 20


class PkvError(RuntimeError):
    def __init__(self, func: str, status: int, text: str):
        super().__init__(f"{func}: status {status} ({text})")
        self.status = status


_lib = None


def load(path: Optional[str] = None) -> ctypes.CDLL:
    """Load the CUDA library (once).  Raises if it is missing: there is no
    fallback path."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"CUDA library not found at {p}; build it with "
            "`python -m paged_kv_cache_117_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(p)
    vp, ci, cf, cs = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    lib.paged_kv_write.argtypes = [vp, vp, vp, vp, vp, ci, ci, ci, ci, ci, ci, vp]
    lib.paged_kv_write.restype = ci
    lib.paged_block_copy.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ci, vp]
    lib.paged_block_copy.restype = ci
    lib.paged_block_copy_ws.argtypes = [vp, vp, vp, ci, ci, ci, ci, ci, ci, vp, cs, vp]
    lib.paged_block_copy_ws.restype = ci
    lib.paged_block_copy_workspace_bytes.argtypes = [ci]
    lib.paged_block_copy_workspace_bytes.restype = cs
    lib.paged_attention_decode.argtypes = [vp, ci, vp, vp, vp, ci, vp, ci, vp, ci, ci, ci,
                                           ci, ci, ci, cf, ci, vp, cs, vp]
    lib.paged_attention_decode.restype = ci
    lib.paged_attention_decode_append.argtypes = [vp, ci, vp, vp, vp, vp, vp, ci, vp, ci, vp,
                                                  ci, ci, ci, ci, ci, ci, cf, ci, vp, cs, vp]
    lib.paged_attention_decode_append.restype = ci
    lib.paged_attention_workspace_bytes.argtypes = [ci, ci, ci, ci, ci]
    lib.paged_attention_workspace_bytes.restype = cs
    lib.pkv_status_string.argtypes = [ci]
    lib.pkv_status_string.restype = ctypes.c_char_p
    lib.pkv_read_device_flags.argtypes = [ctypes.POINTER(ctypes.c_uint32), ci, vp]
    lib.pkv_read_device_flags.restype = ci
    lib.pkv_last_error_string.argtypes = []
    lib.pkv_last_error_string.restype = ctypes.c_char_p
    lib.paged_attention_decode_noalloc.argtypes = [vp, ci, vp, vp, vp, ci, vp, ci, vp, ci, ci,
                                                   ci, ci, ci, ci, cf, ci, vp]
    lib.paged_attention_decode_noalloc.restype = ci
    i64, i32p, i64p = ctypes.c_int64, ctypes.POINTER(ctypes.c_int32), ctypes.POINTER(ctypes.c_int64)
    lib.paged_attention_chunked.argtypes = [vp, ci, vp, vp, vp, ci, vp, ci, vp, vp, ci, ci, ci,
                                            ci, ci, ci, ci, ci, ctypes.c_float, ci, vp]
    lib.paged_attention_chunked.restype = ci
    lib.paged_attention_mixed.argtypes = [vp, ci, vp, vp, vp, ci, vp, ci, vp, vp, ci, ci, ci,
                                          ci, ci, ci, ci, ci, ctypes.c_float, ci, ci, vp, cs, vp]
    lib.paged_attention_mixed.restype = ci
    lib.pkv_bm_create.argtypes = [ci, ci, vp]
    lib.pkv_bm_create.restype = vp
    lib.pkv_bm_destroy.argtypes = [vp]
    lib.pkv_bm_destroy.restype = None
    lib.pkv_bm_add_sequence.argtypes = [vp, i64]
    lib.pkv_bm_add_sequence.restype = ci
    lib.pkv_bm_fork.argtypes = [vp, i64, i64]
    lib.pkv_bm_fork.restype = ci
    lib.pkv_bm_free_sequence.argtypes = [vp, i64]
    lib.pkv_bm_free_sequence.restype = ci
    lib.pkv_bm_append.argtypes = [vp, vp, ci, vp, vp, ctypes.POINTER(ci)]
    lib.pkv_bm_append.restype = ci
    lib.pkv_bm_table.argtypes = [vp, i64, vp, ci, ctypes.POINTER(ci), i64p]
    lib.pkv_bm_table.restype = ci
    lib.pkv_bm_num_free.argtypes = [vp]
    lib.pkv_bm_num_free.restype = ci
    lib.pkv_bm_refcount.argtypes = [vp, ci]
    lib.pkv_bm_refcount.restype = ci
    u64, u8p = ctypes.c_uint64, ctypes.POINTER(ctypes.c_uint8)
    lib.pkv_pc_create.argtypes = [ci, ci, vp]
    lib.pkv_pc_create.restype = vp
    lib.pkv_pc_destroy.argtypes = [vp]
    lib.pkv_pc_destroy.restype = None
    lib.pkv_pc_add_sequence.argtypes = [vp, i64, vp, ci, u64, ctypes.POINTER(ci)]
    lib.pkv_pc_add_sequence.restype = ci
    lib.pkv_pc_append.argtypes = [vp, i64, vp, ci, vp]
    lib.pkv_pc_append.restype = ci
    lib.pkv_pc_free_sequence.argtypes = [vp, i64]
    lib.pkv_pc_free_sequence.restype = ci
    lib.pkv_pc_table.argtypes = [vp, i64, vp, ci, ctypes.POINTER(ci), i64p]
    lib.pkv_pc_table.restype = ci
    lib.pkv_pc_num_free.argtypes = [vp]
    lib.pkv_pc_num_free.restype = ci
    lib.pkv_pc_num_cached.argtypes = [vp]
    lib.pkv_pc_num_cached.restype = ci
    lib.pkv_pc_refcount.argtypes = [vp, ci]
    lib.pkv_pc_refcount.restype = ci
    lib.pkv_pc_block_key.argtypes = [vp, ci, vp, ctypes.POINTER(ci)]
    lib.pkv_pc_block_key.restype = ci
    lib.pkv_pc_free_queue.argtypes = [vp, vp, ci, ctypes.POINTER(ci)]
    lib.pkv_pc_free_queue.restype = ci
    lib.pkv_pc_chain_keys.argtypes = [vp, ci, ci, u64, vp]
    lib.pkv_pc_chain_keys.restype = ci
    lib.pkv_sha256.argtypes = [vp, ctypes.c_size_t, vp]
    lib.pkv_sha256.restype = ci
    if path is None:
        _lib = lib
    return lib


def _check(func: str, status: int) -> None:
    if status != 0:
        text = load().pkv_status_string(status).decode()
        if status == 6:
            text += ": " + load().pkv_last_error_string().decode()
        raise PkvError(func, status, text)


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _need_cuda(name: str, *ts: torch.Tensor) -> None:
    for t in ts:
        if not t.is_cuda:
            raise ValueError(f"{name}: tensors must be on a CUDA device")
        if not t.is_contiguous():
            raise ValueError(f"{name}: tensors must be contiguous")


def _cache_dims(k_cache: torch.Tensor):
    if k_cache.dim() != 4:
        raise ValueError("k_cache must be [num_blocks, block_size, num_kv_heads, head_dim]")
    return tuple(int(x) for x in k_cache.shape)


def paged_kv_write(key, value, k_cache, v_cache, slot_mapping, stream=None) -> None:
    """Store key/value [T, Hkv, D] into the pool slots slot_mapping (int64 [T])."""
    _need_cuda("paged_kv_write", key, value, k_cache, v_cache, slot_mapping)
    N, B, H, D = _cache_dims(k_cache)
    if slot_mapping.dtype != torch.int64:
        raise ValueError("slot_mapping must be int64")
    st = load().paged_kv_write(_ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
                               _ptr(slot_mapping), int(key.shape[0]), N, B, H, D,
                               _DTYPE_CODE.get(k_cache.dtype, -1), _stream(stream))
    _check("paged_kv_write", st)


def paged_block_copy_workspace_bytes(num_blocks: int) -> int:
    n = load().paged_block_copy_workspace_bytes(int(num_blocks))
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid block copy workspace query")
    return int(n)


def block_copy_workspace(k_cache) -> torch.Tensor:
    """A zeroed counter workspace for paged_block_copy(..., workspace=) on
    k_cache's pool: allocate once, reuse for every call on that pool (each
    call leaves it zeroed)."""
    n = paged_block_copy_workspace_bytes(int(k_cache.shape[0]))
    return torch.zeros(n, dtype=torch.uint8, device=k_cache.device)


def paged_block_copy(k_cache, v_cache, block_pairs, workspace=None, stream=None) -> None:
    """Copy whole blocks src -> dst for every row (src, dst) of int64 [P, 2].
    With ``workspace`` (from block_copy_workspace) the pair check costs O(1)
    per CTA (paged_block_copy_ws); without, each CTA scans the pair list
    (paged_block_copy), which suits the few pairs of a decode step."""
    _need_cuda("paged_block_copy", k_cache, v_cache, block_pairs)
    N, B, H, D = _cache_dims(k_cache)
    if block_pairs.dtype != torch.int64:
        raise ValueError("block_pairs must be int64")
    P = int(block_pairs.shape[0]) if block_pairs.numel() else 0
    code = _DTYPE_CODE.get(k_cache.dtype, -1)
    if workspace is None:
        st = load().paged_block_copy(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), P, N, B,
                                     H, D, code, _stream(stream))
        _check("paged_block_copy", st)
        return
    _need_cuda("paged_block_copy", workspace)
    st = load().paged_block_copy_ws(_ptr(k_cache), _ptr(v_cache), _ptr(block_pairs), P, N, B,
                                    H, D, code, _ptr(workspace),
                                    workspace.numel() * workspace.element_size(),
                                    _stream(stream))
    _check("paged_block_copy_ws", st)


def paged_attention_workspace_bytes(num_seqs: int, num_q_heads: int, head_dim: int,
                                    max_context: int, partition_tokens: int) -> int:
    n = load().paged_attention_workspace_bytes(num_seqs, num_q_heads, head_dim,
                                               max_context, partition_tokens)
    if n == ctypes.c_size_t(-1).value:
        raise ValueError("invalid workspace query")
    return int(n)


def paged_attention_decode(out, q, k_cache, v_cache, block_tables, context_lens, scale,
                           partition_tokens=512, workspace=None, stream=None):
    """Decode attention: out [S, Hq, D] (f32, f16 or bf16) from q [S, Hq, D]
    over the paged pool.  A workspace tensor is allocated by torch when none is
    given and the partitioned pass needs one."""
    _need_cuda("paged_attention_decode", out, q, k_cache, v_cache, block_tables, context_lens)
    N, B, Hkv, D = _cache_dims(k_cache)
    S, Hq, _ = (int(x) for x in q.shape)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    max_blocks = int(block_tables.shape[1])
    need = paged_attention_workspace_bytes(S, Hq, D, max_blocks * B, partition_tokens)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().paged_attention_decode(
        _ptr(out), _DTYPE_CODE.get(out.dtype, -1), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _DTYPE_CODE.get(k_cache.dtype, -1), _ptr(block_tables), max_blocks, _ptr(context_lens),
        S, Hq, Hkv, D, B, N, float(scale), int(partition_tokens), _ptr(workspace), ws_bytes,
        _stream(stream))
    _check("paged_attention_decode", st)
    return out


def paged_attention_decode_append(out, q, key, value, k_cache, v_cache, block_tables,
                                  context_lens, scale, partition_tokens=512, workspace=None,
                                  stream=None):
    """The decode step's KV write and decode attention in one call: the rows
    key/value [S, Hkv, D] go to each sequence's position context_lens[s] - 1
    (the slot its block table gives) in both pools, and out [S, Hq, D] is the
    attention over all context_lens[s] positions, that one included."""
    _need_cuda("paged_attention_decode_append", out, q, key, value, k_cache, v_cache,
               block_tables, context_lens)
    N, B, Hkv, D = _cache_dims(k_cache)
    S, Hq, _ = (int(x) for x in q.shape)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    for t in (key, value):
        if tuple(t.shape) != (S, Hkv, D) or t.dtype != k_cache.dtype or not t.is_contiguous():
            raise ValueError("key/value must be contiguous [num_seqs, num_kv_heads, head_dim] "
                             "of the cache dtype")
    max_blocks = int(block_tables.shape[1])
    need = paged_attention_workspace_bytes(S, Hq, D, max_blocks * B, partition_tokens)
    if workspace is None and need > 0:
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().paged_attention_decode_append(
        _ptr(out), _DTYPE_CODE.get(out.dtype, -1), _ptr(q), _ptr(key), _ptr(value),
        _ptr(k_cache), _ptr(v_cache), _DTYPE_CODE.get(k_cache.dtype, -1), _ptr(block_tables),
        max_blocks, _ptr(context_lens), S, Hq, Hkv, D, B, N, float(scale),
        int(partition_tokens), _ptr(workspace), ws_bytes, _stream(stream))
    _check("paged_attention_decode_append", st)
    return out


def paged_attention_decode_noalloc(out, q, k_cache, v_cache, block_tables, context_lens,
                                   scale, partition_tokens=512, stream=None):
    """paged_attention_decode for callers that cannot allocate a workspace:
    the library's own fixed scratch (NOALLOC_SCRATCH_BYTES per device) is
    used instead.  Calls that overlap in time on one device must not be
    issued (they share that scratch)."""
    _need_cuda("paged_attention_decode_noalloc", out, q, k_cache, v_cache, block_tables,
               context_lens)
    N, B, Hkv, D = _cache_dims(k_cache)
    S, Hq, _ = (int(x) for x in q.shape)
    if block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32:
        raise ValueError("block_tables and context_lens must be int32")
    st = load().paged_attention_decode_noalloc(
        _ptr(out), _DTYPE_CODE.get(out.dtype, -1), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _DTYPE_CODE.get(k_cache.dtype, -1), _ptr(block_tables), int(block_tables.shape[1]),
        _ptr(context_lens), S, Hq, Hkv, D, B, N, float(scale), int(partition_tokens),
        _stream(stream))
    _check("paged_attention_decode_noalloc", st)
    return out


P_FORMATS = {"hilo": 0, "f16": 1}


def paged_attention_chunked(out, q, k_cache, v_cache, block_tables, context_lens, query_start,
                            scale, max_query_len=None, p_format="hilo", stream=None):
    """Multi-query attention (chunked prefill and decode in one batch): out
    [T, Hq, D] from q [T, Hq, D], rows packed by sequence as query_start
    (int32 [S + 1]) says, each sequence's rows being its last positions.
    ``max_query_len`` bounds every sequence's row count; when omitted it is
    read from query_start (a device-to-host copy).  ``p_format``: "hilo" (P as
    hi + lo 16-bit operands, ~1e-5) or "f16" (P and V as f16, half the P.V
    work)."""
    _need_cuda("paged_attention_chunked", out, q, k_cache, v_cache, block_tables, context_lens,
               query_start)
    N, B, Hkv, D = _cache_dims(k_cache)
    T, Hq, _ = (int(x) for x in q.shape)
    if (block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32
            or query_start.dtype != torch.int32):
        raise ValueError("block_tables, context_lens and query_start must be int32")
    S = int(context_lens.shape[0])
    if int(query_start.shape[0]) != S + 1:
        raise ValueError("query_start must have num_seqs + 1 entries")
    if max_query_len is None:
        max_query_len = int((query_start[1:] - query_start[:-1]).max().item()) if S else 0
    st = load().paged_attention_chunked(
        _ptr(out), _DTYPE_CODE.get(out.dtype, -1), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _DTYPE_CODE.get(k_cache.dtype, -1), _ptr(block_tables), int(block_tables.shape[1]),
        _ptr(context_lens), _ptr(query_start), S, T, int(max_query_len), Hq, Hkv, D, B, N,
        float(scale), P_FORMATS.get(p_format, -1), _stream(stream))
    _check("paged_attention_chunked", st)
    return out


def paged_attention_mixed(out, q, k_cache, v_cache, block_tables, context_lens, query_start,
                          scale, max_query_len=None, p_format="hilo", partition_tokens=512,
                          workspace=None, stream=None):
    """paged_attention_chunked for a batch that mixes decode tokens with
    prompt chunks: the sequences with one query row run on the decode kernel
    (rows found through query_start), the others on the tensor-core kernel;
    with at most 8 query heads per KV head the two run side by side on
    disjoint SMs.  A workspace tensor is allocated by torch when none is
    given."""
    _need_cuda("paged_attention_mixed", out, q, k_cache, v_cache, block_tables, context_lens,
               query_start)
    N, B, Hkv, D = _cache_dims(k_cache)
    T, Hq, _ = (int(x) for x in q.shape)
    if (block_tables.dtype != torch.int32 or context_lens.dtype != torch.int32
            or query_start.dtype != torch.int32):
        raise ValueError("block_tables, context_lens and query_start must be int32")
    S = int(context_lens.shape[0])
    if int(query_start.shape[0]) != S + 1:
        raise ValueError("query_start must have num_seqs + 1 entries")
    if max_query_len is None:
        max_query_len = int((query_start[1:] - query_start[:-1]).max().item()) if S else 0
    max_blocks = int(block_tables.shape[1])
    if workspace is None and S:
        need = paged_attention_workspace_bytes(S, Hq, D, max_blocks * B, partition_tokens)
        workspace = torch.empty(need, dtype=torch.uint8, device=q.device)
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    st = load().paged_attention_mixed(
        _ptr(out), _DTYPE_CODE.get(out.dtype, -1), _ptr(q), _ptr(k_cache), _ptr(v_cache),
        _DTYPE_CODE.get(k_cache.dtype, -1), _ptr(block_tables), max_blocks, _ptr(context_lens),
        _ptr(query_start), S, T, int(max_query_len), Hq, Hkv, D, B, N, float(scale),
        P_FORMATS.get(p_format, -1), int(partition_tokens), _ptr(workspace), ws_bytes,
        _stream(stream))
    _check("paged_attention_mixed", st)
    return out


def read_device_flags(clear: bool = True, stream=None) -> int:
    v = ctypes.c_uint32(0)
    st = load().pkv_read_device_flags(ctypes.byref(v), 1 if clear else 0, _stream(stream))
    _check("pkv_read_device_flags", st)
    return int(v.value)


class BlockManager:
    """The library's host-side block manager (pkv_bm_* in the C ABI): block
    allocation, reference counts and copy-on-write for one pool."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self._lib = load()
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        order = None
        if free_order is not None:
            order = _host(free_order, torch.int32)
            if order.numel() != num_blocks:
                raise ValueError("free_order must list every block once")
        self._order = order
        h = self._lib.pkv_bm_create(int(num_blocks), int(block_size),
                                    None if order is None else order.data_ptr())
        if not h:
            raise ValueError("invalid block manager arguments")
        self._h = h

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.pkv_bm_destroy(h)

    def add_sequence(self, seq: int) -> None:
        _check("pkv_bm_add_sequence", self._lib.pkv_bm_add_sequence(self._h, int(seq)))

    def fork(self, parent: int, child: int) -> None:
        _check("pkv_bm_fork", self._lib.pkv_bm_fork(self._h, int(parent), int(child)))

    def free_sequence(self, seq: int) -> None:
        _check("pkv_bm_free_sequence", self._lib.pkv_bm_free_sequence(self._h, int(seq)))

    def append(self, seqs):
        """Next-token slots of ``seqs`` (in order) and the copy-on-write pairs
        that must run first: (int64 [n] slots, int64 [P, 2] pairs), CPU."""
        ids = _host(seqs, torch.int64)
        n = ids.numel()
        slots = torch.empty(n, dtype=torch.int64)
        pairs = torch.empty((max(n, 1), 2), dtype=torch.int64)
        npairs = ctypes.c_int(0)
        st = self._lib.pkv_bm_append(self._h, ids.data_ptr() if n else None, n,
                                     slots.data_ptr() if n else None, pairs.data_ptr(),
                                     ctypes.byref(npairs))
        _check("pkv_bm_append", st)
        return slots, pairs[: npairs.value].clone()

    def append_tokens(self, seq: int, count: int):
        """`count` tokens to one sequence: (slots, pairs)."""
        return self.append([seq] * int(count))

    def table(self, seq: int):
        """(block table as a list, number of tokens) of one sequence."""
        nb, nt = ctypes.c_int(0), ctypes.c_int64(0)
        _check("pkv_bm_table", self._lib.pkv_bm_table(self._h, int(seq), None, 0,
                                                      ctypes.byref(nb), ctypes.byref(nt)))
        out = torch.empty(max(nb.value, 1), dtype=torch.int32)
        _check("pkv_bm_table", self._lib.pkv_bm_table(self._h, int(seq), out.data_ptr(),
                                                      nb.value, ctypes.byref(nb),
                                                      ctypes.byref(nt)))
        return out[: nb.value].tolist(), int(nt.value)

    def num_free(self) -> int:
        return int(self._lib.pkv_bm_num_free(self._h))

    def num_used_blocks(self) -> int:
        return self.num_blocks - self.num_free()

    def refcount(self, block: int) -> int:
        return int(self._lib.pkv_bm_refcount(self._h, int(block)))


def _host(xs, dtype) -> torch.Tensor:
    """A contiguous host copy of a tensor or a sequence of ints, in `dtype`
    (for the host managers' C calls).  A tensor must hold integers that fit
    `dtype`: a float, complex or bool tensor, or a value out of range, raises
    ValueError, as the sequence path does (a value that wrapped would, for
    example, give two different token streams the same block key)."""
    if isinstance(xs, torch.Tensor):
        t = xs.detach().to(device="cpu")
        if t.dtype.is_floating_point or t.dtype.is_complex or t.dtype == torch.bool:
            raise ValueError(f"integer tensor expected, got {t.dtype}")
        if t.numel():
            info = torch.iinfo(dtype)
            lo, hi = int(t.min()), int(t.max())
            if lo < info.min or hi > info.max:
                raise ValueError(f"value out of range for {dtype}: [{lo}, {hi}]")
        return t.to(dtype=dtype).contiguous()
    try:
        return torch.as_tensor(list(xs), dtype=dtype).contiguous()
    except (RuntimeError, TypeError) as e:
        raise ValueError(f"integers that fit {dtype} expected: {e}") from None


def _i32(xs) -> torch.Tensor:
    return _host(xs, torch.int32)


def sha256(data: bytes) -> bytes:
    """SHA-256 digest computed by the library."""
    buf = ctypes.create_string_buffer(bytes(data), max(1, len(data)))
    out = (ctypes.c_uint8 * 32)()
    _check("pkv_sha256", load().pkv_sha256(ctypes.cast(buf, ctypes.c_void_p), len(data),
                                           ctypes.cast(out, ctypes.c_void_p)))
    return bytes(out)


def chain_keys(tokens, block_size: int, extra_key: int = 0):
    """Chained keys (32 bytes each) of every full block of a token stream."""
    t = _i32(tokens)
    nb = t.numel() // int(block_size)
    out = (ctypes.c_uint8 * max(1, 32 * nb))()
    _check("pkv_pc_chain_keys", load().pkv_pc_chain_keys(
        t.data_ptr() if t.numel() else None, t.numel(), int(block_size), int(extra_key),
        ctypes.cast(out, ctypes.c_void_p)))
    raw = bytes(out)
    return [raw[32 * i:32 * (i + 1)] for i in range(nb)]


class PrefixCache:
    """The library's block manager with a prefix cache (pkv_pc_* in the C
    ABI): chained block keys, a key -> block map of full blocks, and a free
    queue whose order is the eviction order."""

    def __init__(self, num_blocks: int, block_size: int, free_order=None):
        self._lib = load()
        self.num_blocks, self.block_size = int(num_blocks), int(block_size)
        order = None if free_order is None else _i32(free_order)
        if order is not None and order.numel() != num_blocks:
            raise ValueError("free_order must list every block once")
        self._order = order
        h = self._lib.pkv_pc_create(int(num_blocks), int(block_size),
                                    None if order is None else order.data_ptr())
        if not h:
            raise ValueError("invalid prefix cache arguments")
        self._h = h

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            self._lib.pkv_pc_destroy(h)

    def add_sequence(self, seq: int, prompt, extra_key: int = 0) -> int:
        """Start a request; returns the number of prompt tokens already cached."""
        t = _i32(prompt)
        n = ctypes.c_int(0)
        _check("pkv_pc_add_sequence", self._lib.pkv_pc_add_sequence(
            self._h, int(seq), t.data_ptr() if t.numel() else None, t.numel(), int(extra_key),
            ctypes.byref(n)))
        return int(n.value)

    def append(self, seq: int, tokens) -> torch.Tensor:
        """Slots (int64, CPU) of the sequence's next tokens."""
        t = _i32(tokens)
        slots = torch.empty(max(t.numel(), 1), dtype=torch.int64)
        _check("pkv_pc_append", self._lib.pkv_pc_append(
            self._h, int(seq), t.data_ptr() if t.numel() else None, t.numel(), slots.data_ptr()))
        return slots[: t.numel()]

    def free_sequence(self, seq: int) -> None:
        _check("pkv_pc_free_sequence", self._lib.pkv_pc_free_sequence(self._h, int(seq)))

    def table(self, seq: int):
        nb, nt = ctypes.c_int(0), ctypes.c_int64(0)
        _check("pkv_pc_table", self._lib.pkv_pc_table(self._h, int(seq), None, 0,
                                                      ctypes.byref(nb), ctypes.byref(nt)))
        out = torch.empty(max(nb.value, 1), dtype=torch.int32)
        _check("pkv_pc_table", self._lib.pkv_pc_table(self._h, int(seq), out.data_ptr(), nb.value,
                                                      ctypes.byref(nb), ctypes.byref(nt)))
        return out[: nb.value].tolist(), int(nt.value)

    def num_free(self) -> int:
        return int(self._lib.pkv_pc_num_free(self._h))

    def num_cached(self) -> int:
        return int(self._lib.pkv_pc_num_cached(self._h))

    def refcount(self, block: int) -> int:
        return int(self._lib.pkv_pc_refcount(self._h, int(block)))

    def block_key(self, block: int):
        """The block's cached key (bytes), or None."""
        out = (ctypes.c_uint8 * 32)()
        cached = ctypes.c_int(0)
        _check("pkv_pc_block_key", self._lib.pkv_pc_block_key(
            self._h, int(block), ctypes.cast(out, ctypes.c_void_p), ctypes.byref(cached)))
        return bytes(out) if cached.value else None

    def free_queue(self):
        """The free queue from front (next to allocate / evict) to back."""
        out = torch.empty(max(self.num_blocks, 1), dtype=torch.int32)
        n = ctypes.c_int(0)
        _check("pkv_pc_free_queue", self._lib.pkv_pc_free_queue(
            self._h, out.data_ptr(), self.num_blocks, ctypes.byref(n)))
        return out[: n.value].tolist()
