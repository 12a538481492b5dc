// paged_kv_write ("reshape and cache"): token t's key and value rows go to
// pool slot slot_mapping[t].  In the [num_blocks, block_size, num_kv_heads,
// head_dim] pool, slot s starts at byte s * row_bytes with row_bytes =
// num_kv_heads * head_dim * elem_bytes, so each token's K (and V) row is one
// contiguous run: the kernel moves it in 16-byte vectors, all tokens in one
// launch ("PagedAttention and vLLM: Paging the KV Cache Like an OS", Step 5,
// "Write").
#include "pkv_device.cuh"
#include "pkv_launch.h"

namespace pkv {

__global__ void __launch_bounds__(256)
    kv_write_kernel(const uint4 *__restrict__ key, const uint4 *__restrict__ value,
                    uint4 *__restrict__ k_cache, uint4 *__restrict__ v_cache,
                    const int64_t *__restrict__ slots, int num_tokens, int row_vecs,
                    long long num_slots, unsigned *flags) {
  pdl_launch_dependents();
  pdl_wait_predecessors();   // inputs may come from, and the pool be read by, earlier kernels
  const long long total = (long long)num_tokens * row_vecs;
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < total;
       i += (long long)gridDim.x * blockDim.x) {
    const int t = (int)(i / row_vecs);
    const int c = (int)(i - (long long)t * row_vecs);
    const long long slot = __ldg(reinterpret_cast<const long long *>(slots) + t);
    if (slot < 0) continue;  // padding token
    if (slot >= num_slots) {
      if (c == 0) atomicOr(flags, PKV_FLAG_SLOT_RANGE);
      continue;
    }
    const size_t src = (size_t)t * row_vecs + c;
    const size_t dst = (size_t)slot * row_vecs + c;
    const uint4 kx = __ldg(key + src);
    const uint4 vx = __ldg(value + src);
    k_cache[dst] = kx;
    v_cache[dst] = vx;
  }
}

cudaError_t launch_kv_write(const void *key, const void *value, void *k_cache,
                            void *v_cache, const int64_t *slots, int num_tokens,
                            int row_bytes, long long num_slots, unsigned *flags,
                            cudaStream_t stream) {
  const int row_vecs = row_bytes / 16;
  const long long total = (long long)num_tokens * row_vecs;
  long long blocks = (total + 255) / 256;
  if (blocks > 152LL * 32) blocks = 152LL * 32;
  return launch_pdl(kv_write_kernel, dim3((unsigned)blocks), dim3(256), 0, stream,
                    static_cast<const uint4 *>(key), static_cast<const uint4 *>(value),
                    static_cast<uint4 *>(k_cache), static_cast<uint4 *>(v_cache), slots,
                    num_tokens, row_vecs, num_slots, flags);
}

}  // namespace pkv
