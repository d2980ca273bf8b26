// pkv_noalloc.cu -- paged_decode_attention for callers that cannot allocate device memory.
//
// paged_decode_attention needs a caller-provided workspace when the launcher splits
// long contexts into partitions.  Some callers have no way to provide one: code that
// runs where device allocation is forbidden or unsafe -- a host framework or plugin
// that owns all device memory and hands out none, a real-time loop that must not call
// cudaMalloc (it can synchronise the device and its latency is unbounded), or a
// caller without a CUDA allocator of its own.  This entry point serves them: it runs
// the same kernels with the partition workspace placed in a fixed array compiled into
// the library, so the call itself allocates nothing.
//
// The array below is a file-scope __device__ variable.  Every GPU that loads the
// library holds kNoAllocScratchBytes of it until the process exits.  In host code its
// name is only a host-side stand-in, so its device address is fetched once per device
// with cudaGetSymbolAddress and cached.
#include <cuda_runtime.h>

#include <mutex>

#include "pkv_internal.h"

namespace pkv {
namespace {

constexpr size_t kNoAllocScratchBytes = PKV_NOALLOC_SCRATCH_BYTES;  // 32 MiB
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void *g_noalloc_ptr[kMaxDevices];

// Device address of g_noalloc_scratch on the current device (looked up once per device).
int scratch_address(void **out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "paged_decode_attention_noalloc: cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices)
    return set_error(PKV_ERR_CUDA, "paged_decode_attention_noalloc: device index %d", dev);
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
    if (e != cudaSuccess || !p)
      return cuda_error(e, "paged_decode_attention_noalloc: cudaGetSymbolAddress(scratch)");
    g_noalloc_ptr[dev] = p;
  }
  *out = g_noalloc_ptr[dev];
  return PKV_OK;
}

}  // namespace
}  // namespace pkv

PKV_API int paged_decode_attention_noalloc(pkv_bf16 *out, const pkv_bf16 *q,
                                           const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                                           const int32_t *block_tables,
                                           int32_t max_blocks_per_seq,
                                           const int32_t *context_lens, int32_t max_context_len,
                                           int32_t num_seqs, int32_t num_q_heads,
                                           const pkv_cache_desc *cache, float scale,
                                           void *stream) {
  using namespace pkv;
  static const char *const kFn = "paged_decode_attention_noalloc";
  if (!cache) return set_error(PKV_ERR_NULL, "%s: cache descriptor is NULL", kFn);
  if (num_seqs < 0 || num_q_heads <= 0 || cache->num_kv_heads <= 0 || max_context_len < 0)
    return set_error(PKV_ERR_SHAPE, "%s: bad sizes", kFn);
  // The size the launcher's plan needs, checked before any device call.
  const size_t need = paged_decode_workspace_size(num_seqs, num_q_heads, cache->num_kv_heads,
                                                  cache->head_dim, max_context_len);
  if (need > kNoAllocScratchBytes)
    return set_error(PKV_ERR_WORKSPACE,
                     "%s: these sizes need %zu bytes of partition workspace, more than the "
                     "library's fixed %zu-byte scratch; call paged_decode_attention with a "
                     "workspace instead",
                     kFn, need, kNoAllocScratchBytes);
  // Every argument check of paged_decode_attention, before any device call: a call
  // that is refused leaves nothing queued on the stream and never touches the array.
  int rc = check_decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                  context_lens, max_context_len, num_seqs, num_q_heads, cache,
                                  kNoAllocScratchBytes, kFn);
  if (rc) return rc;
  if (num_seqs == 0) {
    clear_error();
    return PKV_OK;
  }
  // First call on this device: look up the array's device address (see the header).
  void *scratch = nullptr;
  rc = scratch_address(&scratch);
  if (rc) return rc;
  // The decode keeps one completion counter per (sequence, kv head), then two work
  // scheduling words, at the start of its workspace; they must be zero when the kernel
  // starts.  A completed call leaves them zero, but clear them anyway so a call never
  // depends on the previous one.  The plan was accepted above, so `need` covers them
  // and lies within the array.
  size_t clear = (size_t)num_seqs * cache->num_kv_heads * 4 + 8;
  if (clear > need) clear = need;
  const cudaError_t e = cudaMemsetAsync(scratch, 0, clear, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return cuda_error(e, "paged_decode_attention_noalloc: clear counters");
  return paged_decode_attention(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                context_lens, max_context_len, num_seqs, num_q_heads, cache,
                                scale, scratch, kNoAllocScratchBytes, stream);
}
