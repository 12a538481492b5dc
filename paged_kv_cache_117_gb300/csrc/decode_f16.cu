// Decode attention instantiations for an fp16 KV cache.
#include "decode_kernel.cuh"

namespace pkv {
cudaError_t launch_decode_f16(const CUtensorMap &kmap, const CUtensorMap &vmap,
                              const DecodeParams &p, int head_dim, int block_size,
                              cudaStream_t stream, int *launches) {
  return launch_decode_typed<__half>(kmap, vmap, p, head_dim, block_size, stream, launches);
}
}  // namespace pkv
