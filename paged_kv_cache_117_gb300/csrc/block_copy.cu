// paged_block_copy: the batched copy-on-write copy.  Every (src, dst) pair
// copies a whole block -- block_size slots of K and of V -- and one launch
// serves every pair of the step ("PagedAttention and vLLM: Paging the KV
// Cache Like an OS", Step 5, "Copy").  A block is one contiguous run of
// block_bytes in each pool, moved in 16-byte vectors; CTA (x, y) copies chunk
// x % chunks of pair x / chunks in pool y (0 = K, 1 = V).
//
// The copies of one call run in no particular order, so a pair whose dst is
// another pair's dst or src would race; such a pair is skipped and flagged.
// Two ways to find them:
//  * scan (no workspace): each CTA compares its pair with every other pair,
//    O(num_pairs) per CTA -- nothing for the few pairs of a decode step;
//  * counts (caller workspace of two counters per pool block, zero between
//    calls): a counting pass adds every pair's dst to cnt_dst[dst] and its src
//    to cnt_src[src]; the copy CTA of a pair then reads two counters, O(1);
//    a reset pass zeroes the counters it touched.  Three launches chained by
//    programmatic dependent launch, each waiting for its predecessor.
#include "pkv_device.cuh"
#include "pkv_launch.h"

namespace pkv {

constexpr int COPY_THREADS = 256;
constexpr int COPY_UNROLL = 4;
constexpr int COPY_CHUNK_VECS = COPY_THREADS * COPY_UNROLL;  // 16 KiB per CTA

constexpr int COUNT_THREADS = 256;

__device__ __forceinline__ bool pair_in_range(long long src, long long dst, int num_blocks) {
  return src >= 0 && src < num_blocks && dst >= 0 && dst < num_blocks;
}

// Counting pass: cnt[dst] += 1 and cnt[num_blocks + src] += 1 for every pair
// in range (out-of-range pairs are flagged by the copy pass).
__global__ void __launch_bounds__(COUNT_THREADS)
    block_copy_count_kernel(const int64_t *__restrict__ pairs, int num_pairs, int num_blocks,
                            unsigned *cnt) {
  pdl_launch_dependents();
  pdl_wait_predecessors();   // the previous call's reset pass may still own cnt
  const int i = blockIdx.x * COUNT_THREADS + threadIdx.x;
  if (i >= num_pairs) return;
  const long long src = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * i);
  const long long dst = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * i + 1);
  if (!pair_in_range(src, dst, num_blocks)) return;
  atomicAdd(cnt + dst, 1u);
  atomicAdd(cnt + num_blocks + src, 1u);
}

// Reset pass: zeroes the counters the counting pass raised, so the workspace
// is all zero again when the call's work is done.
__global__ void __launch_bounds__(COUNT_THREADS)
    block_copy_reset_kernel(const int64_t *__restrict__ pairs, int num_pairs, int num_blocks,
                            unsigned *cnt) {
  pdl_launch_dependents();
  pdl_wait_predecessors();   // every copy CTA has read its counters
  const int i = blockIdx.x * COUNT_THREADS + threadIdx.x;
  if (i >= num_pairs) return;
  const long long src = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * i);
  const long long dst = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * i + 1);
  if (!pair_in_range(src, dst, num_blocks)) return;
  cnt[dst] = 0u;
  cnt[num_blocks + src] = 0u;
}

// cnt == nullptr: the scan check; otherwise the counters of the counting pass.
__global__ void __launch_bounds__(COPY_THREADS)
    block_copy_kernel(uint4 *k_cache, uint4 *v_cache, const int64_t *__restrict__ pairs,
                      int num_pairs, long long block_vecs, int chunks, int num_blocks,
                      const unsigned *cnt, unsigned *flags) {
  pdl_launch_dependents();
  pdl_wait_predecessors();   // the pool may be written or read by earlier kernels
  const int pair = blockIdx.x / chunks;
  const int chunk = blockIdx.x - pair * chunks;
  if (pair >= num_pairs) return;
  const long long src = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * pair);
  const long long dst = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * pair + 1);
  if (!pair_in_range(src, dst, num_blocks)) {
    if (chunk == 0 && blockIdx.y == 0 && threadIdx.x == 0) atomicOr(flags, PKV_FLAG_PAIR_RANGE);
    return;
  }
  // A pair whose dst is also another pair's dst or src would race: it is
  // skipped and flagged (the block manager never produces one).  A pair that
  // copies a block onto itself clashes with no one.  Pairs outside the pool
  // copy nothing, so they clash with no one either (in both checks).
  bool clash = false;
  if (cnt != nullptr) {
    if (threadIdx.x == 0)
      clash = __ldcg(cnt + dst) > 1u || __ldcg(cnt + num_blocks + dst) > (src == dst ? 1u : 0u);
  } else {
    for (int i = threadIdx.x; i < num_pairs; i += COPY_THREADS) {
      if (i == pair) continue;
      const long long si = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * i);
      const long long di = __ldg(reinterpret_cast<const long long *>(pairs) + 2 * i + 1);
      clash |= pair_in_range(si, di, num_blocks) && (si == dst || di == dst);
    }
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
                              unsigned *counters, unsigned *flags, cudaStream_t stream) {
  const long long block_vecs = block_bytes / 16;
  const int chunks = (int)((block_vecs + COPY_CHUNK_VECS - 1) / COPY_CHUNK_VECS);
  const long long gx = (long long)num_pairs * chunks;
  if (gx > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  const unsigned gc = (unsigned)((num_pairs + COUNT_THREADS - 1) / COUNT_THREADS);
  cudaError_t e = cudaSuccess;
  if (counters != nullptr) {
    e = launch_pdl(block_copy_count_kernel, dim3(gc), dim3(COUNT_THREADS), 0, stream, pairs,
                   num_pairs, num_blocks, counters);
    if (e != cudaSuccess) return e;
  }
  e = launch_pdl(block_copy_kernel, dim3((unsigned)gx, 2), dim3(COPY_THREADS), 0, stream,
                 static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), pairs, num_pairs,
                 block_vecs, chunks, num_blocks, static_cast<const unsigned *>(counters), flags);
  if (e != cudaSuccess || counters == nullptr) return e;
  return launch_pdl(block_copy_reset_kernel, dim3(gc), dim3(COUNT_THREADS), 0, stream, pairs,
                    num_pairs, num_blocks, counters);
}

}  // namespace pkv
