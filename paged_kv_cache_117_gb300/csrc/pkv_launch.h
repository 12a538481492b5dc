// Internal host-side interface between the C ABI (capi.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace pkv {

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
  int num_gchunks;               // CTAs per KV head along the query group
  int num_blocks;                // pool size, for range checks
  float scale_log2;              // scale * log2(e): scores live in the exp2 domain
  int part_blocks;               // blocks per partition
  int max_parts;                 // partitions per sequence the workspace holds
  float *part_ml;                // [S, Hq, max_parts, 2]  (running max, sum)
  float *part_o;                 // [S, Hq, max_parts, D]  unnormalised output
  unsigned *flags;               // device flag word
};

// Launch the decode pass (and, when max_parts > 1, the merge pass) for one
// cache dtype / head_dim / block_size combination.  Returns a cudaError_t.
cudaError_t launch_decode_bf16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                               const DecodeParams &p, int head_dim, int block_size,
                               cudaStream_t stream, int *launches);
cudaError_t launch_decode_f16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const DecodeParams &p, int head_dim, int block_size,
                              cudaStream_t stream, int *launches);

cudaError_t launch_kv_write(const void *key, const void *value, void *k_cache,
                            void *v_cache, const int64_t *slots, int num_tokens,
                            int row_bytes, long long num_slots, unsigned *flags,
                            cudaStream_t stream);

cudaError_t launch_block_copy(void *k_cache, void *v_cache, const int64_t *pairs,
                              int num_pairs, long long block_bytes, int num_blocks,
                              unsigned *flags, cudaStream_t stream);

}  // namespace pkv
