// pkv_write.cu -- the slot-mapping KV write.
//
// "vLLM-Style Llama Inference Engine with Tensor Parallelism", Features and scope:
// paged KV caching with block tables and slot mappings; each step writes the new
// tokens' K/V into the paged cache.  "mini-vLLM" README (throughput section) names
// a per-sequence Python write loop as its overhead; here the whole step's tokens
// are scattered by one launch.
//
// One thread moves one 16-byte vector (8 bf16) of K and the matching vector of V:
// consecutive threads cover consecutive vectors of a (token, kv head) row, so both
// the reads of k/v and the writes into the cache row are coalesced 16-byte accesses.
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {

__device__ unsigned int g_write_errors;

__global__ void __launch_bounds__(256) kv_write_kernel(const uint4 *__restrict__ k,
                                                       const uint4 *__restrict__ v,
                                                       const int64_t *__restrict__ slot_mapping,
                                                       int64_t num_vecs, uint4 *__restrict__ k_cache,
                                                       uint4 *__restrict__ v_cache,
                                                       int64_t num_blocks, int32_t num_kv_heads,
                                                       int32_t block_size, int32_t vecs_per_row) {
  // A decode kernel launched right after this one (programmatic dependent launch) may
  // start its prologue now; it waits for this grid's writes before reading the cache.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int64_t row_vecs = (int64_t)num_kv_heads * vecs_per_row;  // vectors per token
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < num_vecs;
       i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t tok = i / row_vecs;
    const int64_t rem = i - tok * row_vecs;
    const int64_t h = rem / vecs_per_row;
    const int64_t e = rem - h * vecs_per_row;
    const int64_t slot = __ldg(slot_mapping + tok);
    if (slot < 0) continue;  // padding
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    if (blk >= num_blocks) {
      atomicOr(&g_write_errors, (unsigned)PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * vecs_per_row + e;
    const uint4 kv = __ldg(k + i);
    const uint4 vv = __ldg(v + i);
    k_cache[dst] = kv;
    v_cache[dst] = vv;
  }
}

cudaError_t read_write_errors(uint32_t *flags, int clear) {
  unsigned int f = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&f, g_write_errors, sizeof f);
  if (e != cudaSuccess) return e;
  *flags |= f;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_write_errors, &zero, sizeof zero);
  }
  return e;
}

// Host checks of paged_kv_write's arguments (nothing is enqueued).
int check_write(const void *k, const void *v, const int64_t *slot_mapping, int64_t num_tokens,
                const void *k_cache, const void *v_cache, const pkv_cache_desc *cache) {
  if (!cache) return set_error(PKV_ERR_NULL, "paged_kv_write: cache descriptor is NULL");
  if (num_tokens < 0) return set_error(PKV_ERR_SHAPE, "paged_kv_write: num_tokens < 0");
  if (cache->num_blocks <= 0 || cache->block_size <= 0 || cache->num_kv_heads <= 0 ||
      cache->head_dim <= 0)
    return set_error(PKV_ERR_SHAPE, "paged_kv_write: cache sizes must be positive");
  if (cache->head_dim % 8 != 0)
    return set_error(PKV_ERR_UNSUPPORTED, "paged_kv_write: head_dim %d is not a multiple of 8",
                     cache->head_dim);
  if (num_tokens == 0) return PKV_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache)
    return set_error(PKV_ERR_NULL, "paged_kv_write: NULL tensor pointer");
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache))
    return set_error(PKV_ERR_ALIGN, "paged_kv_write: k, v and the caches must be 16-byte aligned");
  if ((reinterpret_cast<uintptr_t>(slot_mapping) & 7u) != 0)
    return set_error(PKV_ERR_ALIGN, "paged_kv_write: slot_mapping must be 8-byte aligned");
  return PKV_OK;
}

// Enqueues the write kernel (arguments already checked).
int launch_write(const pkv_bf16 *k, const pkv_bf16 *v, const int64_t *slot_mapping,
                 int64_t num_tokens, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                 const pkv_cache_desc &c, cudaStream_t stream) {
  if (num_tokens == 0) return PKV_OK;
  const int32_t vpr = c.head_dim / 8;
  const int64_t num_vecs = num_tokens * c.num_kv_heads * (int64_t)vpr;
  const int threads = 256;
  int64_t blocks = (num_vecs + threads - 1) / threads;
  if (blocks > 65535LL * 32) blocks = 65535LL * 32;  // grid-stride beyond this
  kv_write_kernel<<<(unsigned)blocks, threads, 0, stream>>>(
      reinterpret_cast<const uint4 *>(k), reinterpret_cast<const uint4 *>(v), slot_mapping,
      num_vecs, reinterpret_cast<uint4 *>(k_cache), reinterpret_cast<uint4 *>(v_cache),
      c.num_blocks, c.num_kv_heads, c.block_size, vpr);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "paged_kv_write launch");
  return PKV_OK;
}

}  // namespace pkv

PKV_API int paged_kv_write(const pkv_bf16 *k, const pkv_bf16 *v, const int64_t *slot_mapping,
                           int64_t num_tokens, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                           const pkv_cache_desc *cache, void *stream) {
  int rc = pkv::check_write(k, v, slot_mapping, num_tokens, k_cache, v_cache, cache);
  if (!rc) rc = pkv::launch_write(k, v, slot_mapping, num_tokens, k_cache, v_cache, *cache,
                                  static_cast<cudaStream_t>(stream));
  if (!rc) pkv::clear_error();
  return rc;
}
