// paged_attention_decode_noalloc: decode attention that needs no workspace
// from its caller.
//
// paged_attention_decode asks the caller for a scratch buffer (work list,
// completion counters, partition records).  Some callers cannot provide one:
// a host program whose device memory is owned by another memory manager that
// hands out no extra buffers, a plugin running inside a host process with a
// fixed, pre-reserved memory budget, or a latency-critical serving loop that
// must not call cudaMalloc (which can synchronise the device).  For them this
// entry point uses a scratch array that is part of the library image itself:
// the CUDA runtime places it in device memory when the library's module is
// loaded, and every GPU that loads the library keeps it until the process
// exits.
//
// Set-up: the first call on a device, with that device current, looks up the
// array's device address with cudaGetSymbolAddress and caches it; later calls
// on that device reuse it.  Make that first call before any stream capture.
// The cached address is never refreshed, so a process that calls
// cudaDeviceReset on a device must not call this entry point on that device
// again.  Nothing here allocates memory.
//
// The array is shared by every call on a device and keeps the last call's
// contents; the attention pass resets what must start at zero itself.  Calls
// that overlap in time on one device race on the array: issue them on one
// stream, or wait for one to finish before the next starts.
#include <limits.h>

#include <mutex>

#include "pkv_device.cuh"

// Scratch of the allocation-free entry point (see above).
static __device__ __align__(256) unsigned char g_noalloc_scratch[PKV_NOALLOC_SCRATCH_BYTES];

namespace {
constexpr int NOALLOC_MAX_DEVICES = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[NOALLOC_MAX_DEVICES] = {};
}  // namespace

extern "C" pkv_status paged_attention_decode_noalloc(
    void *out, pkv_dtype out_dtype, const void *q, const void *k_cache, const void *v_cache,
    pkv_dtype dtype, const int32_t *block_tables, int max_blocks, const int32_t *context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
    int num_blocks, float scale, int partition_tokens, pkv_stream_t stream) {
  // Size check first: a request that does not fit is refused before any
  // CUDA call.
  if (max_blocks <= 0 || block_size <= 0) return PKV_ERR_RANGE;
  const long long max_context = (long long)max_blocks * block_size;
  if (max_context > INT_MAX) return PKV_ERR_RANGE;
  const size_t need = paged_attention_workspace_bytes(num_seqs, num_q_heads, head_dim,
                                                      (int)max_context, partition_tokens);
  if (need == (size_t)-1) return PKV_ERR_RANGE;
  if (need > (size_t)PKV_NOALLOC_SCRATCH_BYTES) return PKV_ERR_WORKSPACE;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PKV_ERR_CUDA;
  if (dev < 0 || dev >= NOALLOC_MAX_DEVICES) return PKV_ERR_RANGE;
  void *scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
      void *addr = nullptr;
      if (cudaGetSymbolAddress(&addr, g_noalloc_scratch) != cudaSuccess || !addr)
        return PKV_ERR_CUDA;
      g_noalloc_addr[dev] = addr;
    }
    scratch = g_noalloc_addr[dev];
  }
  return paged_attention_decode(out, out_dtype, q, k_cache, v_cache, dtype, block_tables,
                                max_blocks, context_lens, num_seqs, num_q_heads, num_kv_heads,
                                head_dim, block_size, num_blocks, scale, partition_tokens,
                                scratch, (size_t)PKV_NOALLOC_SCRATCH_BYTES, stream);
}
