// The library's C ABI (declared in include/paged_kv.h): host-side argument
// checks, TMA descriptor encoding for the pool, and the kernel launches.
#include <limits.h>
#include <stdio.h>
#include <string.h>

#include <mutex>

#include "pkv_device.cuh"
#include "pkv_launch.h"

// OR of PKV_FLAG_* bits raised by the kernels on this device.
__device__ unsigned int g_pkv_flags;

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                   const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                   const cuuint32_t *, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

constexpr int MAX_DEVICES = 64;

unsigned *device_flags() {
  static unsigned *ptrs[MAX_DEVICES] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= MAX_DEVICES) return nullptr;
  if (!ptrs[dev]) {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_pkv_flags) != cudaSuccess) return nullptr;
    ptrs[dev] = static_cast<unsigned *>(p);
  }
  return ptrs[dev];
}

// TMA descriptor over one pool [N, B, Hkv, D] whose box is a [min(B, 16), 64]
// slab of one KV head of one block, 128B-swizzled in shared memory (the
// layout the decode kernel's ldmatrix reads assume).  A few recent
// descriptors are cached per thread.
struct MapKey {
  const void *base;
  int dt, n, b, h, d, rows;
  bool operator==(const MapKey &o) const {
    return base == o.base && dt == o.dt && n == o.n && b == o.b && h == o.h && d == o.d &&
           rows == o.rows;
  }
};

// Tensor map of a K or V pool: one box = 64 dims (128 bytes, 128B-swizzled) x
// box_rows tokens of one KV head of one block.
bool pool_map(CUtensorMap *out, const void *base, pkv_dtype dt, int N, int B, int Hkv, int D,
              int box_rows) {
  struct Entry {
    MapKey key;
    CUtensorMap map;
    bool used;
  };
  thread_local Entry cache[4] = {};
  thread_local int next = 0;
  const MapKey key{base, (int)dt, N, B, Hkv, D, box_rows};
  for (auto &e : cache)
    if (e.used && e.key == key) {
      *out = e.map;
      return true;
    }
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t es = 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)Hkv, (cuuint64_t)B, (cuuint64_t)N};
  cuuint64_t strides[3] = {D * es, (cuuint64_t)Hkv * D * es, (cuuint64_t)B * Hkv * D * es};
  cuuint32_t box[4] = {64u, 1u, (cuuint32_t)box_rows, 1u};
  cuuint32_t estr[4] = {1u, 1u, 1u, 1u};
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  const CUtensorMapDataType t =
      dt == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
  const CUresult r = fn(&map, t, 4, const_cast<void *>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  cache[next] = Entry{key, map, true};
  next = (next + 1) & 3;
  *out = map;
  return true;
}

// Text of the CUDA error behind the last PKV_ERR_CUDA returned on this thread.
thread_local char g_last_error[256] = "no error";

pkv_status cuda_fail(cudaError_t e, const char *where) {
  snprintf(g_last_error, sizeof(g_last_error), "%s: %s (%s)", where, cudaGetErrorName(e),
           cudaGetErrorString(e));
  return PKV_ERR_CUDA;
}

pkv_status cuda_fail_msg(const char *msg) {
  snprintf(g_last_error, sizeof(g_last_error), "%s", msg);
  return PKV_ERR_CUDA;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

bool overlap(const void *a, size_t na, const void *b, size_t nb) {
  if (!a || !b || na == 0 || nb == 0) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

bool supported_cache_dtype(pkv_dtype d) { return d == PKV_F16 || d == PKV_BF16; }
bool supported_head_dim(int d) { return d == 64 || d == 128; }
bool supported_block(int b) { return b == 4 || b == 8 || b == 16 || b == 32; }

size_t dtype_bytes(pkv_dtype d) { return d == PKV_F32 ? 4 : 2; }

long long ceil_div_ll(long long a, long long b) { return (a + b - 1) / b; }

}  // namespace

extern "C" {

const char *pkv_status_string(pkv_status s) {
  switch (s) {
    case PKV_OK: return "ok";
    case PKV_ERR_NULL: return "null pointer";
    case PKV_ERR_SHAPE: return "unsupported or inconsistent shape";
    case PKV_ERR_DTYPE: return "unsupported dtype";
    case PKV_ERR_RANGE: return "size out of range";
    case PKV_ERR_ALIAS: return "buffers overlap";
    case PKV_ERR_CUDA: return "CUDA error";
    case PKV_ERR_WORKSPACE: return "workspace missing or too small";
    case PKV_ERR_ALIGN: return "pointer not aligned as required";
    case PKV_ERR_NO_BLOCKS: return "too few free blocks";
  }
  return "unknown status";
}

size_t paged_attention_workspace_bytes(int num_seqs, int num_q_heads, int head_dim,
                                       int max_context, int partition_tokens) {
  if (num_seqs < 0 || num_q_heads < 0 || head_dim <= 0 || max_context < 0 ||
      partition_tokens < 0)
    return (size_t)-1;
  return pkv::workspace_layout(num_seqs, num_q_heads, head_dim, max_context, partition_tokens)
      .total;
}

pkv_status paged_kv_write(const void *key, const void *value, void *k_cache, void *v_cache,
                          const int64_t *slot_mapping, int num_tokens, int num_blocks,
                          int block_size, int num_kv_heads, int head_dim, pkv_dtype dtype,
                          pkv_stream_t stream) {
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0) return PKV_ERR_RANGE;
  if (!supported_cache_dtype(dtype)) return PKV_ERR_DTYPE;
  if (!supported_head_dim(head_dim) || !supported_block(block_size)) return PKV_ERR_SHAPE;
  if (num_tokens == 0) return PKV_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PKV_ERR_NULL;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) ||
      !aligned(v_cache, 16) || !aligned(slot_mapping, 8))
    return PKV_ERR_ALIGN;
  const size_t row = (size_t)num_kv_heads * head_dim * 2;
  const size_t pool = (size_t)num_blocks * block_size * row;
  const size_t in = (size_t)num_tokens * row;
  if (overlap(k_cache, pool, v_cache, pool) || overlap(key, in, k_cache, pool) ||
      overlap(key, in, v_cache, pool) || overlap(value, in, k_cache, pool) ||
      overlap(value, in, v_cache, pool))
    return PKV_ERR_ALIAS;
  if (row > (size_t)INT_MAX) return PKV_ERR_RANGE;
  unsigned *flags = device_flags();
  if (!flags) return cuda_fail_msg("device flag word unavailable");
  const cudaError_t e = pkv::launch_kv_write(key, value, k_cache, v_cache, slot_mapping,
                                             num_tokens, (int)row,
                                             (long long)num_blocks * block_size, flags,
                                             reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, "paged_kv_write launch");
}

}  // extern "C"

namespace {
pkv_status block_copy_impl(void *k_cache, void *v_cache, const int64_t *block_pairs,
                           int num_pairs, int num_blocks, int block_size, int num_kv_heads,
                           int head_dim, pkv_dtype dtype, void *workspace,
                           size_t workspace_bytes, pkv_stream_t stream, const char *what) {
  if (num_pairs < 0 || num_blocks <= 0 || num_kv_heads <= 0) return PKV_ERR_RANGE;
  if (!supported_cache_dtype(dtype)) return PKV_ERR_DTYPE;
  if (!supported_head_dim(head_dim) || !supported_block(block_size)) return PKV_ERR_SHAPE;
  if (num_pairs == 0) return PKV_OK;
  if (!k_cache || !v_cache || !block_pairs) return PKV_ERR_NULL;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 8))
    return PKV_ERR_ALIGN;
  const size_t block_bytes = (size_t)block_size * num_kv_heads * head_dim * 2;
  const size_t pool = block_bytes * num_blocks;
  const size_t pairs_sz = (size_t)num_pairs * 16;
  if (overlap(k_cache, pool, v_cache, pool) || overlap(block_pairs, pairs_sz, k_cache, pool) ||
      overlap(block_pairs, pairs_sz, v_cache, pool))
    return PKV_ERR_ALIAS;
  if (workspace != nullptr) {
    if (workspace_bytes < paged_block_copy_workspace_bytes(num_blocks)) return PKV_ERR_WORKSPACE;
    if (!aligned(workspace, 256)) return PKV_ERR_ALIGN;
    const size_t ws = (size_t)num_blocks * 8;
    if (overlap(workspace, ws, k_cache, pool) || overlap(workspace, ws, v_cache, pool) ||
        overlap(workspace, ws, block_pairs, pairs_sz))
      return PKV_ERR_ALIAS;
  }
  unsigned *flags = device_flags();
  if (!flags) return cuda_fail_msg("device flag word unavailable");
  const cudaError_t e = pkv::launch_block_copy(
      k_cache, v_cache, block_pairs, num_pairs, (long long)block_bytes, num_blocks,
      static_cast<unsigned *>(workspace), flags, reinterpret_cast<cudaStream_t>(stream));
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, what);
}
}  // namespace

extern "C" {

pkv_status paged_block_copy(void *k_cache, void *v_cache, const int64_t *block_pairs,
                            int num_pairs, int num_blocks, int block_size, int num_kv_heads,
                            int head_dim, pkv_dtype dtype, pkv_stream_t stream) {
  return block_copy_impl(k_cache, v_cache, block_pairs, num_pairs, num_blocks, block_size,
                         num_kv_heads, head_dim, dtype, nullptr, 0, stream,
                         "paged_block_copy launch");
}

size_t paged_block_copy_workspace_bytes(int num_blocks) {
  if (num_blocks <= 0) return (size_t)-1;
  return pkv::round256((size_t)num_blocks * 8);
}

pkv_status paged_block_copy_ws(void *k_cache, void *v_cache, const int64_t *block_pairs,
                               int num_pairs, int num_blocks, int block_size, int num_kv_heads,
                               int head_dim, pkv_dtype dtype, void *workspace,
                               size_t workspace_bytes, pkv_stream_t stream) {
  if (!workspace) return PKV_ERR_WORKSPACE;
  return block_copy_impl(k_cache, v_cache, block_pairs, num_pairs, num_blocks, block_size,
                         num_kv_heads, head_dim, dtype, workspace, workspace_bytes, stream,
                         "paged_block_copy_ws launch");
}

}  // extern "C"

namespace {
// Decode attention, optionally appending this step's token first (key_new /
// value_new non-null).
pkv_status decode_impl(void *out, pkv_dtype out_dtype, const void *q, const void *key_new,
                       const void *value_new, void *k_cache, void *v_cache, pkv_dtype dtype,
                       const int32_t *block_tables, int max_blocks, const int32_t *context_lens,
                       int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, float scale, int partition_tokens,
                       void *workspace, size_t workspace_bytes, pkv_stream_t stream,
                       const char *what, const int32_t *query_start = nullptr,
                       int num_tokens = 0, int beside_chunked = 0) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      max_blocks <= 0 || partition_tokens < 0)
    return PKV_ERR_RANGE;
  if (!supported_cache_dtype(dtype)) return PKV_ERR_DTYPE;
  if (out_dtype != PKV_F32 && out_dtype != PKV_F16 && out_dtype != PKV_BF16)
    return PKV_ERR_DTYPE;
  if (!supported_head_dim(head_dim) || !supported_block(block_size)) return PKV_ERR_SHAPE;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_SHAPE;
  if (partition_tokens % block_size != 0) return PKV_ERR_SHAPE;
  if ((long long)max_blocks * block_size > INT_MAX) return PKV_ERR_RANGE;
  if (num_seqs == 0) return PKV_OK;
  if (num_seqs > 65535) return PKV_ERR_RANGE;
  const int group = num_q_heads / num_kv_heads;
  const int gchunks = group <= 16 ? 1 : (group + 15) / 16;
  if ((long long)num_kv_heads * gchunks > 65535) return PKV_ERR_RANGE;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PKV_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(out, dtype_bytes(out_dtype)) || !aligned(block_tables, 4) ||
      !aligned(context_lens, 4))
    return PKV_ERR_ALIGN;

  const int part_blocks = partition_tokens == 0 ? max_blocks : partition_tokens / block_size;
  const pkv::WorkspaceLayout lay = pkv::workspace_layout(
      num_seqs, num_q_heads, head_dim, (long long)max_blocks * block_size, partition_tokens);
  const int max_parts = lay.max_parts;
  if (max_parts != (int)ceil_div_ll(max_blocks, part_blocks)) return PKV_ERR_RANGE;
  const size_t need = lay.total;
  if (!workspace || workspace_bytes < need) return PKV_ERR_WORKSPACE;
  if (!aligned(workspace, 256)) return PKV_ERR_ALIGN;

  const size_t pool = (size_t)num_blocks * block_size * num_kv_heads * head_dim * 2;
  // q and out rows: one per sequence, or (a mixed batch) num_tokens
  const size_t nrows = query_start ? (size_t)num_tokens : (size_t)num_seqs;
  const size_t out_sz = nrows * num_q_heads * head_dim * dtype_bytes(out_dtype);
  const size_t q_sz = nrows * num_q_heads * head_dim * 2;
  const size_t tab_sz = (size_t)num_seqs * max_blocks * 4;
  if (query_start && (overlap(workspace, need, query_start, (size_t)(num_seqs + 1) * 4) ||
                      overlap(out, out_sz, query_start, (size_t)(num_seqs + 1) * 4)))
    return PKV_ERR_ALIAS;
  if (overlap(k_cache, pool, v_cache, pool) || overlap(out, out_sz, q, q_sz) ||
      overlap(out, out_sz, k_cache, pool) || overlap(out, out_sz, v_cache, pool) ||
      overlap(out, out_sz, block_tables, tab_sz) ||
      overlap(out, out_sz, context_lens, (size_t)num_seqs * 4) ||
      overlap(workspace, need, out, out_sz) || overlap(workspace, need, q, q_sz) ||
      overlap(workspace, need, k_cache, pool) || overlap(workspace, need, v_cache, pool) ||
      overlap(workspace, need, block_tables, tab_sz) ||
      overlap(workspace, need, context_lens, (size_t)num_seqs * 4))
    return PKV_ERR_ALIAS;
  if (key_new || value_new) {
    if (!key_new || !value_new) return PKV_ERR_NULL;
    if (!aligned(key_new, 16) || !aligned(value_new, 16)) return PKV_ERR_ALIGN;
    // the new rows are read while the pools are written: no overlap with
    // anything the call writes
    const size_t row_sz = (size_t)num_seqs * num_kv_heads * head_dim * 2;
    for (const void *r : {key_new, value_new})
      if (overlap(r, row_sz, k_cache, pool) || overlap(r, row_sz, v_cache, pool) ||
          overlap(r, row_sz, out, out_sz) || overlap(r, row_sz, workspace, need))
        return PKV_ERR_ALIAS;
  }

  CUtensorMap kmap, vmap;
  const int rows16 = block_size < 16 ? block_size : 16;   // decode: up to 16 tokens a box
  if (!pool_map(&kmap, k_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, rows16) ||
      !pool_map(&vmap, v_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim, rows16))
    return cuda_fail_msg("cuTensorMapEncodeTiled failed for the KV pool");
  unsigned *flags = device_flags();
  if (!flags) return cuda_fail_msg("device flag word unavailable");

  pkv::DecodeParams p;
  p.out = out;
  p.out_dtype = (int)out_dtype;
  p.q = q;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.max_blocks = max_blocks;
  p.num_seqs = num_seqs;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.num_gchunks = gchunks;
  p.num_hc = num_kv_heads * gchunks;
  p.head_dim = head_dim;
  p.block_size = block_size;
  p.num_blocks = num_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.part_blocks = part_blocks;
  p.max_parts = max_parts;
  unsigned char *ws = static_cast<unsigned char *>(workspace);
  p.ctrl = reinterpret_cast<unsigned *>(ws + lay.ctrl);
  p.seq_done = reinterpret_cast<unsigned *>(ws + lay.seq_done);
  p.items = reinterpret_cast<int2 *>(ws + lay.items);
  p.part_o = max_parts > 1 ? reinterpret_cast<float *>(ws + lay.part_o) : nullptr;
  p.part_ml = max_parts > 1 ? reinterpret_cast<float *>(ws + lay.part_ml) : nullptr;
  p.flags = flags;
  p.key_new = key_new;
  p.value_new = value_new;
  p.k_pool = key_new ? k_cache : nullptr;
  p.v_pool = key_new ? v_cache : nullptr;
  p.query_start = query_start;
  p.num_tokens = num_tokens;
  if (beside_chunked && query_start && group <= 8) {
    // The SM split between this pass and the chunked pass beside it, from
    // measurements of the two kernels on a 152-SM GB300.  The decode pass
    // in its grouped form, confined to x SMs of the Llama-shaped batch,
    // streams 71.5-73.2 GB/s per SM up to 56 SMs (0.88 TB/s on 12, 4.01 on
    // 56), then 5.00, 5.61, 5.94, 6.25 and 6.39 TB/s on 76, 100, 120, 136 and
    // 152: min(73 GB/s * x, 9.15 TB/s * x / (x + 63)) within 3 %.  The
    // chunked pass's rate per SM, 5.5 TFLOP/s, lies between its rate on
    // 512-token chunks run alone (4.8: waves of a 512-CTA grid) and on long
    // chunks (6.5); it is the value at which the split lands where sweeps of
    // a 256-row + 8-chunk batch found the call fastest (~75 of 152 SMs for
    // the decode rows; 66, 70 and 80+ slower).  Side by side only when the
    // model puts it 5 % ahead of the passes in turn: at the extremes (few
    // decode SMs) it is least accurate.
    p.overlap = 1;
    p.ovl_sm_bps = 73e9f;
    p.ovl_peak_bps = 9.15e12f;
    p.ovl_half_sms = 63.f;
    p.ovl_flops_sm = 5.5e12f;
    p.ovl_margin = 0.05f;
  }

  int launches = 0;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      dtype == PKV_BF16
          ? pkv::launch_decode_bf16(kmap, vmap, p, head_dim, block_size, st, &launches)
          : pkv::launch_decode_f16(kmap, vmap, p, head_dim, block_size, st, &launches);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, what);
}
}  // namespace

extern "C" {

pkv_status paged_attention_decode(void *out, pkv_dtype out_dtype, const void *q,
                                  const void *k_cache, const void *v_cache, pkv_dtype dtype,
                                  const int32_t *block_tables, int max_blocks,
                                  const int32_t *context_lens, int num_seqs, int num_q_heads,
                                  int num_kv_heads, int head_dim, int block_size,
                                  int num_blocks, float scale, int partition_tokens,
                                  void *workspace, size_t workspace_bytes,
                                  pkv_stream_t stream) {
  // the pools are only read when nothing is appended
  return decode_impl(out, out_dtype, q, nullptr, nullptr, const_cast<void *>(k_cache),
                     const_cast<void *>(v_cache), dtype, block_tables, max_blocks,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                     num_blocks, scale, partition_tokens, workspace, workspace_bytes, stream,
                     "paged_attention_decode launch");
}

pkv_status paged_attention_decode_append(void *out, pkv_dtype out_dtype, const void *q,
                                         const void *key, const void *value, void *k_cache,
                                         void *v_cache, pkv_dtype dtype,
                                         const int32_t *block_tables, int max_blocks,
                                         const int32_t *context_lens, int num_seqs,
                                         int num_q_heads, int num_kv_heads, int head_dim,
                                         int block_size, int num_blocks, float scale,
                                         int partition_tokens, void *workspace,
                                         size_t workspace_bytes, pkv_stream_t stream) {
  if (num_seqs > 0 && (!key || !value)) return PKV_ERR_NULL;
  return decode_impl(out, out_dtype, q, key, value, k_cache, v_cache, dtype, block_tables,
                     max_blocks, context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, scale, partition_tokens, workspace, workspace_bytes,
                     stream, "paged_attention_decode_append launch");
}

}  // extern "C"

namespace {
// Multi-query attention.  skip_single: the sequences with one query row are
// left out (a mixed batch whose decode rows go to the decode kernel).
pkv_status chunked_impl(void *out, pkv_dtype out_dtype, const void *q, const void *k_cache,
                        const void *v_cache, pkv_dtype dtype, const int32_t *block_tables,
                        int max_blocks, const int32_t *context_lens,
                        const int32_t *query_start, int num_seqs, int num_tokens,
                        int max_query_len, int num_q_heads, int num_kv_heads, int head_dim,
                        int block_size, int num_blocks, float scale, pkv_p_format p_format,
                        pkv_stream_t stream, int skip_single, bool validate_only,
                        const char *what, unsigned *ovl_done = nullptr) {
  if (p_format != PKV_P_HILO && p_format != PKV_P_F16) return PKV_ERR_DTYPE;
  if (num_seqs < 0 || num_tokens < 0 || max_query_len < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || num_blocks <= 0 || max_blocks <= 0)
    return PKV_ERR_RANGE;
  if (!supported_cache_dtype(dtype)) return PKV_ERR_DTYPE;
  if (out_dtype != PKV_F32 && out_dtype != PKV_F16 && out_dtype != PKV_BF16)
    return PKV_ERR_DTYPE;
  if (!supported_head_dim(head_dim) || !supported_block(block_size)) return PKV_ERR_SHAPE;
  if (num_q_heads % num_kv_heads != 0) return PKV_ERR_SHAPE;
  const int group = num_q_heads / num_kv_heads;
  if (group > 128) return PKV_ERR_SHAPE;
  if (block_size < 8) return PKV_ERR_SHAPE;   // a block's box must fill whole swizzle atoms
  if ((long long)max_blocks * block_size > INT_MAX) return PKV_ERR_RANGE;
  if (num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return PKV_OK;
  if (max_query_len > num_tokens) return PKV_ERR_RANGE;
  const int tile_tokens = 128 / group;
  const long long qtiles = ceil_div_ll(max_query_len, tile_tokens);
  if (qtiles * num_seqs * num_kv_heads > INT_MAX) return PKV_ERR_RANGE;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens || !query_start)
    return PKV_ERR_NULL;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
      !aligned(block_tables, 4) || !aligned(context_lens, 4) || !aligned(query_start, 4))
    return PKV_ERR_ALIGN;
  const size_t pool = (size_t)num_blocks * block_size * num_kv_heads * head_dim * 2;
  const size_t rows = (size_t)num_tokens * num_q_heads * head_dim;
  const size_t out_sz = rows * dtype_bytes(out_dtype), q_sz = rows * 2;
  if (overlap(k_cache, pool, v_cache, pool) || overlap(out, out_sz, q, q_sz) ||
      overlap(out, out_sz, k_cache, pool) || overlap(out, out_sz, v_cache, pool) ||
      overlap(out, out_sz, block_tables, (size_t)num_seqs * max_blocks * 4) ||
      overlap(out, out_sz, context_lens, (size_t)num_seqs * 4) ||
      overlap(out, out_sz, query_start, (size_t)(num_seqs + 1) * 4))
    return PKV_ERR_ALIAS;
  if (validate_only) return PKV_OK;

  CUtensorMap kmap, vmap, qmap;
  // chunked: a whole block (up to 32 tokens) a box -- fewer, larger TMA boxes
  if (!pool_map(&kmap, k_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim,
                block_size) ||
      !pool_map(&vmap, v_cache, dtype, num_blocks, block_size, num_kv_heads, head_dim,
                block_size))
    return cuda_fail_msg("cuTensorMapEncodeTiled failed for the KV pool");
  {
    EncodeTiledFn fn = encode_fn();
    if (!fn) return cuda_fail_msg("cuTensorMapEncodeTiled unavailable");
    // q as [tokens][heads][dims]; one box = 64 dims x the group's heads x
    // 128 / group tokens (128 rows of 128 bytes, 128B-swizzled)
    cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_q_heads, (cuuint64_t)num_tokens};
    cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)num_q_heads * head_dim * 2};
    cuuint32_t box[3] = {64u, (cuuint32_t)group, (cuuint32_t)tile_tokens};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    memset(&qmap, 0, sizeof(qmap));
    const CUtensorMapDataType t =
        dtype == PKV_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    if (fn(&qmap, t, 3, const_cast<void *>(q), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
      return cuda_fail_msg("cuTensorMapEncodeTiled failed for q");
  }
  unsigned *flags = device_flags();
  if (!flags) return cuda_fail_msg("device flag word unavailable");

  pkv::ChunkedParams p;
  p.out = out;
  p.out_dtype = (int)out_dtype;
  p.block_tables = block_tables;
  p.context_lens = context_lens;
  p.query_start = query_start;
  p.max_blocks = max_blocks;
  p.num_seqs = num_seqs;
  p.num_tokens = num_tokens;
  p.num_q_heads = num_q_heads;
  p.num_kv_heads = num_kv_heads;
  p.group = group;
  p.tile_tokens = tile_tokens;
  p.num_qtiles = (int)qtiles;
  p.num_qpairs = (int)((qtiles + 1) / 2);
  p.p_format = (int)p_format;
  p.skip_single = skip_single;
  p.max_query_len = max_query_len;
  p.num_blocks = num_blocks;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.flags = flags;
  p.ovl_done = ovl_done;
  const cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const cudaError_t e =
      dtype == PKV_BF16 ? pkv::launch_chunked_bf16(qmap, kmap, vmap, p, head_dim, block_size, st)
                        : pkv::launch_chunked_f16(qmap, kmap, vmap, p, head_dim, block_size, st);
  return e == cudaSuccess ? PKV_OK : cuda_fail(e, what);
}
}  // namespace

extern "C" {

pkv_status paged_attention_chunked(void *out, pkv_dtype out_dtype, const void *q,
                                   const void *k_cache, const void *v_cache, pkv_dtype dtype,
                                   const int32_t *block_tables, int max_blocks,
                                   const int32_t *context_lens, const int32_t *query_start,
                                   int num_seqs, int num_tokens, int max_query_len,
                                   int num_q_heads, int num_kv_heads, int head_dim,
                                   int block_size, int num_blocks, float scale,
                                   pkv_p_format p_format, pkv_stream_t stream) {
  return chunked_impl(out, out_dtype, q, k_cache, v_cache, dtype, block_tables, max_blocks,
                      context_lens, query_start, num_seqs, num_tokens, max_query_len,
                      num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                      p_format, stream, 0, false, "paged_attention_chunked launch");
}

pkv_status paged_attention_mixed(void *out, pkv_dtype out_dtype, const void *q,
                                 const void *k_cache, const void *v_cache, pkv_dtype dtype,
                                 const int32_t *block_tables, int max_blocks,
                                 const int32_t *context_lens, const int32_t *query_start,
                                 int num_seqs, int num_tokens, int max_query_len,
                                 int num_q_heads, int num_kv_heads, int head_dim,
                                 int block_size, int num_blocks, float scale,
                                 pkv_p_format p_format, int partition_tokens, void *workspace,
                                 size_t workspace_bytes, pkv_stream_t stream) {
  // every argument of both halves is checked before anything is launched
  pkv_status st = chunked_impl(out, out_dtype, q, k_cache, v_cache, dtype, block_tables,
                               max_blocks, context_lens, query_start, num_seqs, num_tokens,
                               max_query_len, num_q_heads, num_kv_heads, head_dim, block_size,
                               num_blocks, scale, p_format, stream, 1, true,
                               "paged_attention_mixed launch");
  if (st != PKV_OK || num_seqs == 0 || num_tokens == 0 || max_query_len == 0) return st;
  if (num_seqs > 65535) return PKV_ERR_RANGE;
  if (!workspace) return PKV_ERR_WORKSPACE;
  // The decode rows (sequences with one query row), then the chunks; the two
  // kernels write disjoint rows of out and only read the pool.  With chunks
  // in the batch and a group of at most 8 heads, the two passes run at the
  // same time on disjoint SMs: the decode pass holds whole SMs (three
  // decoders per CTA) and keeps the share its work list picks, the chunked
  // pass takes the rest as they free up, and its grid ends after the decode
  // grid (its finished-CTA counter is word 3 of the workspace's control
  // block, zeroed by the decode work list).
  const bool ovl = max_query_len >= 2 && num_q_heads / num_kv_heads <= 8;
  st = decode_impl(out, out_dtype, q, nullptr, nullptr, const_cast<void *>(k_cache),
                   const_cast<void *>(v_cache), dtype, block_tables, max_blocks, context_lens,
                   num_seqs, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                   partition_tokens, workspace, workspace_bytes, stream,
                   "paged_attention_mixed decode launch", query_start, num_tokens, ovl ? 1 : 0);
  if (st != PKV_OK || max_query_len < 2) return st;
  unsigned *ovl_done =
      ovl ? reinterpret_cast<unsigned *>(static_cast<unsigned char *>(workspace) +
                                         pkv::WS_CTRL_OFFSET) +
                pkv::WS_CTRL_CHUNKED_DONE
          : nullptr;
  return chunked_impl(out, out_dtype, q, k_cache, v_cache, dtype, block_tables, max_blocks,
                      context_lens, query_start, num_seqs, num_tokens, max_query_len,
                      num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale,
                      p_format, stream, 1, false, "paged_attention_mixed chunked launch",
                      ovl_done);
}

pkv_status pkv_read_device_flags(uint32_t *flags_out, int clear, pkv_stream_t stream) {
  if (!flags_out) return PKV_ERR_NULL;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
  unsigned v = 0;
  e = cudaMemcpyFromSymbol(&v, g_pkv_flags, sizeof(v));
  if (e != cudaSuccess) return cuda_fail(e, "read flag word");
  *flags_out = v;
  if (clear) {
    const unsigned zero = 0;
    e = cudaMemcpyToSymbol(g_pkv_flags, &zero, sizeof(zero));
    if (e != cudaSuccess) return cuda_fail(e, "clear flag word");
  }
  return PKV_OK;
}

const char *pkv_last_error_string(void) { return g_last_error; }

}  // extern "C"
