// Internal host-side interface between the C ABI (capi.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

// Workspace carve-up of paged_attention_decode (offsets in bytes, each
// 256-byte aligned): control words, per-sequence completion counters, the
// work list, then the partition records when a sequence can span more than
// one partition.
struct WorkspaceLayout {
  size_t ctrl, seq_done, items, part_o, part_ml, total;
  int max_parts;
};

inline size_t round256(size_t v) { return (v + 255) / 256 * 256; }

// The control block (64 uint32 words) opens the workspace: [0] next work
// unit, [1] number of units, [2] decoders that run, [3] chunked CTAs finished.
constexpr size_t WS_CTRL_OFFSET = 0;
constexpr int WS_CTRL_CHUNKED_DONE = 3;

inline WorkspaceLayout workspace_layout(long long S, long long Hq, long long D,
                                        long long max_context, long long partition_tokens) {
  WorkspaceLayout w{};
  long long parts = 1;
  if (partition_tokens > 0) parts = (max_context + partition_tokens - 1) / partition_tokens;
  if (parts < 1) parts = 1;
  w.max_parts = (int)parts;
  w.ctrl = WS_CTRL_OFFSET;
  w.seq_done = WS_CTRL_OFFSET + 256;
  w.items = w.seq_done + round256((size_t)(S * Hq) * 4);
  w.part_o = w.items + round256((size_t)(S * parts) * 8);
  if (parts > 1) {
    w.part_ml = w.part_o + (size_t)(S * Hq * parts * D) * 4;
    w.total = w.part_ml + (size_t)(S * Hq * parts) * 8;
  } else {
    w.part_ml = w.part_o;
    w.total = w.part_o;
  }
  return w;
}

struct DecodeParams {
  void *out;
  int out_dtype;                 // pkv_dtype
  const void *q;                 // [S, Hq, D]
  const int32_t *block_tables;   // [S, max_blocks]
  const int32_t *context_lens;   // [S]
  int max_blocks;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;                     // Hq / Hkv
  int num_gchunks;               // query-head chunks (<= 16 heads each) per KV head
  int num_hc;                    // num_kv_heads * num_gchunks
  int head_dim;
  int block_size;
  int num_blocks;                // pool size, for range checks
  float scale_log2;              // scale * log2(e): scores live in the exp2 domain
  int part_blocks;               // blocks per partition
  int max_parts;                 // partitions per sequence the workspace holds
  float *part_ml;                // [S, Hq, max_parts, 2]  (running max, sum)
  float *part_o;                 // [S, Hq, max_parts, D]  unnormalised output
  unsigned *ctrl;                // [0] next work unit, [1] number of work units,
                                 // [2] decoders that run, [3] chunked CTAs finished
  int grid = 0;                  // CTAs of the attention grid (set at launch)
  unsigned *seq_done;            // [S, num_hc] partitions finished per sequence
  int2 *items;                   // [S * max_parts] (sequence, partition) work list
  unsigned *flags;               // device flag word
  // Appending this step's token (null: the pool already holds it): its K and V
  // rows [S, Hkv, D], used for position L - 1 and stored into the pools.
  const void *key_new = nullptr;
  const void *value_new = nullptr;
  void *k_pool = nullptr;
  void *v_pool = nullptr;
  // A mixed batch (null: row s of q and out is sequence s): sequence s owns
  // rows query_start[s] .. query_start[s + 1] - 1 of q and out, and only the
  // sequences with exactly one row are this kernel's (the others are left to
  // the chunked kernel).
  const int32_t *query_start = nullptr;
  int num_tokens = 0;            // rows of q and out when query_start is set
  // A mixed batch whose chunked pass runs at the same time as this decode
  // pass (overlap = 1, group <= 8): the work list picks how many SMs the
  // decode pass keeps (ctrl[2] decoders) from this model of the two passes,
  // and the decode CTAs hold whole SMs, ovl_wg decoders each.
  int overlap = 0;
  int ovl_wg = 1;                // decoders per CTA (set at launch)
  int ovl_sms = 0;               // SMs of the device (set at launch)
  float ovl_sm_bps = 0.f;        // decode bandwidth model on x SMs:
  float ovl_peak_bps = 0.f;      //   min(sm_bps * x, peak * x / (x + half))
  float ovl_half_sms = 0.f;
  float ovl_flops_sm = 0.f;      // chunked pass: flop/s per SM
  float ovl_margin = 0.f;        // side by side only when predicted this much faster
};

// Launch the work-list pass and the decode pass for one cache dtype /
// head_dim / block_size combination.  Returns a cudaError_t.
cudaError_t launch_decode_bf16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeParams &p, int head_dim, int block_size,
                               cudaStream_t stream, int *launches);
cudaError_t launch_decode_f16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const DecodeParams &p, int head_dim, int block_size,
                              cudaStream_t stream, int *launches);

// Multi-query (chunked prefill) attention: one CTA per (pair of query tiles,
// sequence, KV head).  A query tile is tile_tokens = 128 / group tokens.
struct ChunkedParams {
  void *out;                     // [num_tokens, Hq, D]
  int out_dtype;                 // pkv_dtype
  const int32_t *block_tables;   // [S, max_blocks]
  const int32_t *context_lens;   // [S], counting this chunk's tokens
  const int32_t *query_start;    // [S + 1]
  int max_blocks;
  int num_seqs;
  int num_tokens;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int tile_tokens;
  int num_qtiles;                // ceil(max_query_len / tile_tokens)
  int num_qpairs;                // ceil(num_qtiles / 2): query tiles go two to a CTA
  int compact = 0;               // the grid lists only existing units (set at launch)
  int p_format;                  // pkv_p_format
  int skip_single = 0;           // sequences with one query row are left to the decode kernel
  int max_query_len;
  int num_blocks;
  float scale_log2;
  unsigned *flags;
  // Non-null: the chunked pass of a mixed batch that runs beside the decode
  // pass launched just before it; counts this grid's finished CTAs (zeroed
  // by the decode work list), and the last one waits for the decode grid.
  unsigned *ovl_done = nullptr;
};

cudaError_t launch_chunked_bf16(const CUtensorMap &qmap, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, const ChunkedParams &p, int head_dim,
                                int block_size, cudaStream_t stream);
cudaError_t launch_chunked_f16(const CUtensorMap &qmap, const CUtensorMap &kmap,
                               const CUtensorMap &vmap, const ChunkedParams &p, int head_dim,
                               int block_size, cudaStream_t stream);

// Launches `kern` with programmatic stream serialization allowed, so that
// its launch overlaps the tail of the previous kernel on `stream`.  The
// kernels call griddepcontrol.wait before touching shared data.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

cudaError_t launch_kv_write(const void *key, const void *value, void *k_cache,
                            void *v_cache, const int64_t *slots, int num_tokens,
                            int row_bytes, long long num_slots, unsigned *flags,
                            cudaStream_t stream);

// counters: null (each copy CTA scans the pair list) or the caller's zeroed
// [2, num_blocks] counter workspace (counting pass, copy, reset pass).
cudaError_t launch_block_copy(void *k_cache, void *v_cache, const int64_t *pairs,
                              int num_pairs, long long block_bytes, int num_blocks,
                              unsigned *counters, unsigned *flags, cudaStream_t stream);

}  // namespace pkv
