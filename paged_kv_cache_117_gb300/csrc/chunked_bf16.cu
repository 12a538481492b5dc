// Multi-query (chunked prefill) attention instantiations for a bf16 KV cache.
#include "chunked_kernel.cuh"

namespace pkv {
cudaError_t launch_chunked_bf16(const CUtensorMap &qmap, const CUtensorMap &kmap,
                                const CUtensorMap &vmap, const ChunkedParams &p, int head_dim,
                                int block_size, cudaStream_t stream) {
  return launch_chunked_t<__nv_bfloat16>(qmap, kmap, vmap, p, head_dim, block_size, stream);
}
}  // namespace pkv
