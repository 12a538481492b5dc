// paged_block_copy: the batched copy-on-write copy.  Every (src, dst) pair
// copies a whole block -- block_size slots of K and of V -- and one launch
// serves every pair of the step ("PagedAttention and vLLM: Paging the KV
// Cache Like an OS", Step 5, "Copy").  A block is one contiguous run of
// block_bytes in each pool, moved in 16-byte vectors; CTA (x, y) copies chunk
// x % chunks of pair x / chunks in pool y (0 = K, 1 = V).
#include "pkv_device.cuh"
#include "pkv_launch.h"

namespace pkv {

constexpr int COPY_THREADS = 256;
constexpr int COPY_UNROLL = 4;
constexpr int COPY_CHUNK_VECS = COPY_THREADS * COPY_UNROLL;  // 16 KiB per CTA

__global__ void __launch_bounds__(COPY_THREADS)
    block_copy_kernel(uint4 *k_cache, uint4 *v_cache, const int64_t *__restrict__ pairs,
                      int num_pairs, long long block_vecs, int chunks, int num_blocks,
                      unsigned *flags) {
  pdl_launch_dependents();
  pdl_wait_predecessors();   // the pool may be written or read by earlier kernels
  const int pair = blockIdx.x / chunks;
  const int chunk = blockIdx.x - pair * chunks;
  if (pair >= num_pairs) return;
  const long long src = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * pair);
  const long long dst = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * pair + 1);
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (chunk == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(flags, PKV_FLAG_PAIR_RANGE);
    return;
  }
  // The copies of one call run in any order, so a pair whose dst is also
  // another pair's dst or src would race: such a pair is skipped and flagged
  // (the block manager never produces one).
  bool clash = false;
  for (int i = threadIdx.x; i < num_pairs; i += COPY_THREADS) {
    if (i == pair) continue;
    const long long si = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * i);
    const long long di = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * i + 1);
    clash |= si == dst || di == dst;
  }
  if (__syncthreads_or(clash)) {
    if (chunk == 0 && blockIdx.y == 0 && threadIdx.x == 0)
      atomicOr(flags, PKV_FLAG_PAIR_CONFLICT);
    return;
  }
  uint4 *pool = blockIdx.y == 0 ? k_cache : v_cache;
  const uint4 *s = pool + src * block_vecs;
  uint4 *d = pool + dst * block_vecs;
  const long long v0 = (long long)chunk * COPY_CHUNK_VECS + threadIdx.x;
  uint4 buf[COPY_UNROLL];
#pragma unroll
  for (int u = 0; u < COPY_UNROLL; ++u) {
    const long long v = v0 + u * COPY_THREADS;
    if (v < block_vecs) buf[u] = s[v];
  }
#pragma unroll
  for (int u = 0; u < COPY_UNROLL; ++u) {
    const long long v = v0 + u * COPY_THREADS;
    if (v < block_vecs) d[v] = buf[u];
  }
}

cudaError_t launch_block_copy(void *k_cache, void *v_cache, const int64_t *pairs,
                              int num_pairs, long long block_bytes, int num_blocks,
                              unsigned *flags, cudaStream_t stream) {
  const long long block_vecs = block_bytes / 16;
  const int chunks = (int)((block_vecs + COPY_CHUNK_VECS - 1) / COPY_CHUNK_VECS);
  const long long gx = (long long)num_pairs * chunks;
  if (gx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_pdl(block_copy_kernel, dim3((unsigned)gx, 2), dim3(COPY_THREADS), 0, stream,
                    static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), pairs,
                    num_pairs, block_vecs, chunks, num_blocks, flags);
}

}  // namespace pkv
