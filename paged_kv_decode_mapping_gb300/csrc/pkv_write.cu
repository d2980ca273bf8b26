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
    // the row's vectors are loaded together with its slot (i < num_vecs: always in
    // bounds), so the write pays one memory latency, not two in a row
    const int64_t slot = __ldg(slot_mapping + tok);
    const uint4 kv = __ldg(k + i);
    const uint4 vv = __ldg(v + i);
    if (slot < 0) continue;  // padding
    const int64_t blk = slot / block_size;
    const int64_t off = slot - blk * block_size;
    if (blk >= num_blocks) {
      atomicOr(&g_write_errors, (unsigned)PKV_DEVERR_SLOT);
      continue;
    }
    const int64_t dst = ((blk * num_kv_heads + h) * block_size + off) * vecs_per_row + e;
    k_cache[dst] = kv;
    v_cache[dst] = vv;
  }
}

// ---------------------------------------------------------------------------
// Slot write with rotary position embedding ("llm-stack", Serving engine: RoPE at
// absolute positions before keys enter the cache; "Building ... with tiny-vLLM": RoPE
// rotates coordinate pairs by sine/cosine of position-dependent angles).
//
// Rows: k [T][Hkv] (rotated, then written to the slot), q [T][Hq] (rotated in place,
// optional), v [T][Hkv] (written to the slot).  A rotated row splits into units: with
// rotate-half pairing a unit is the 16-byte chunk pair (c, c + r/16) holding pairs
// (e, e + r/2); with interleaved pairing one chunk holds four (2i, 2i+1) pairs; chunks
// at or past rotary_dim are copied.  One thread owns a whole unit, so the in-place q
// rotation reads everything it writes.  Each pair is rotated in fp32 with every
// product and sum rounded once (no fused multiply-add), then rounded to bf16:
//   x1' = x1*c - x2*s,  x2' = x2*c + x1*s.
struct RopeArgs {
  const uint4 *k, *v;
  uint4 *q;
  const int64_t *slot_mapping, *positions;
  const float *cos_sin;  // [max_position][r]: cos of pair i at i, sin at r/2 + i
  uint4 *k_cache, *v_cache;
  int64_t num_tokens, max_position, num_blocks;
  int32_t num_q_heads, num_kv_heads, block_size, head_dim, rotary_dim, neox;
};

__device__ __forceinline__ float rope_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float rope_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }
__device__ __forceinline__ uint32_t rope_pack(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
__device__ __forceinline__ void rope_pair(float x1, float x2, float c, float s, float &y1,
                                          float &y2) {
  y1 = __fsub_rn(__fmul_rn(x1, c), __fmul_rn(x2, s));
  y2 = __fadd_rn(__fmul_rn(x2, c), __fmul_rn(x1, s));
}

// Rotates unit u of the row at src (16-byte chunks) into dst; dst may equal src.
__device__ __forceinline__ void rope_unit(uint4 *dst, const uint4 *src, const float *cs, int u,
                                          const RopeArgs &a) {
  const int r = a.rotary_dim, half = r / 2;
  const int ur = a.neox ? r / 16 : r / 8;  // rotated units
  if (u >= ur) {                            // past rotary_dim: copy
    const int c = r / 8 + (u - ur);
    dst[c] = src[c];
    return;
  }
  if (a.neox) {
    const uint4 x1 = src[u], x2 = src[u + r / 16];
    const float4 c0 = *reinterpret_cast<const float4 *>(cs + 8 * u);
    const float4 c1 = *reinterpret_cast<const float4 *>(cs + 8 * u + 4);
    const float4 s0 = *reinterpret_cast<const float4 *>(cs + half + 8 * u);
    const float4 s1 = *reinterpret_cast<const float4 *>(cs + half + 8 * u + 4);
    const uint32_t w1[4] = {x1.x, x1.y, x1.z, x1.w}, w2[4] = {x2.x, x2.y, x2.z, x2.w};
    const float cc[8] = {c0.x, c0.y, c0.z, c0.w, c1.x, c1.y, c1.z, c1.w};
    const float ss[8] = {s0.x, s0.y, s0.z, s0.w, s1.x, s1.y, s1.z, s1.w};
    uint32_t o1[4], o2[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      float a1, a2, b1, b2;
      rope_pair(rope_lo(w1[j]), rope_lo(w2[j]), cc[2 * j], ss[2 * j], a1, a2);
      rope_pair(rope_hi(w1[j]), rope_hi(w2[j]), cc[2 * j + 1], ss[2 * j + 1], b1, b2);
      o1[j] = rope_pack(a1, b1);
      o2[j] = rope_pack(a2, b2);
    }
    dst[u] = make_uint4(o1[0], o1[1], o1[2], o1[3]);
    dst[u + r / 16] = make_uint4(o2[0], o2[1], o2[2], o2[3]);
  } else {
    const uint4 x = src[u];
    const float4 c4 = *reinterpret_cast<const float4 *>(cs + 4 * u);
    const float4 s4 = *reinterpret_cast<const float4 *>(cs + half + 4 * u);
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    const float cc[4] = {c4.x, c4.y, c4.z, c4.w}, ss[4] = {s4.x, s4.y, s4.z, s4.w};
    uint32_t o[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) {  // word j holds the pair (2(4u+j), 2(4u+j)+1)
      float y1, y2;
      rope_pair(rope_lo(w[j]), rope_hi(w[j]), cc[j], ss[j], y1, y2);
      o[j] = rope_pack(y1, y2);
    }
    dst[u] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

__global__ void __launch_bounds__(256) kv_write_rope_kernel(const RopeArgs a) {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  const int vpr = a.head_dim / 8;  // 16-byte chunks per row
  const int units = (a.neox ? a.rotary_dim / 16 : a.rotary_dim / 8) + (a.head_dim - a.rotary_dim) / 8;
  const int64_t nk = a.num_tokens * a.num_kv_heads * units;
  const int64_t nq = a.q ? a.num_tokens * a.num_q_heads * units : 0;
  const int64_t nv = a.num_tokens * a.num_kv_heads * vpr;
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nk + nq + nv;
       i += (int64_t)gridDim.x * blockDim.x) {
    if (i < nk + nq) {  // a rotated row: k (to the cache) or q (in place)
      const bool is_q = i >= nk;
      const int64_t j = is_q ? i - nk : i;
      const int64_t row = j / units;
      const int u = (int)(j - row * units);
      const int heads = is_q ? a.num_q_heads : a.num_kv_heads;
      const int64_t tok = row / heads;
      const int64_t pos = __ldg(a.positions + tok);
      const int64_t slot = is_q ? 0 : __ldg(a.slot_mapping + tok);  // in flight with pos
      if (pos < 0 || pos >= a.max_position) {
        if (u == 0 && row % heads == 0) atomicOr(&g_write_errors, (unsigned)PKV_DEVERR_POSITION);
        continue;
      }
      const float *cs = a.cos_sin + pos * a.rotary_dim;
      if (is_q) {
        uint4 *qrow = a.q + row * vpr;
        rope_unit(qrow, qrow, cs, u, a);
      } else {
        if (slot < 0) continue;
        const int64_t blk = slot / a.block_size, off = slot - blk * a.block_size;
        if (blk >= a.num_blocks) {
          atomicOr(&g_write_errors, (unsigned)PKV_DEVERR_SLOT);
          continue;
        }
        const int64_t h = row - tok * a.num_kv_heads;
        uint4 *dst = a.k_cache + ((blk * a.num_kv_heads + h) * a.block_size + off) * vpr;
        rope_unit(dst, a.k + row * vpr, cs, u, a);
      }
    } else {  // v: plain copy to the slot
      const int64_t j = i - nk - nq;
      const int64_t row = j / vpr;
      const int64_t e = j - row * vpr;
      const int64_t tok = row / a.num_kv_heads;
      const int64_t slot = __ldg(a.slot_mapping + tok);
      const uint4 vv = __ldg(a.v + j);  // in flight with the slot
      if (slot < 0) continue;
      const int64_t blk = slot / a.block_size, off = slot - blk * a.block_size;
      if (blk >= a.num_blocks) continue;  // reported by the k rows
      const int64_t h = row - tok * a.num_kv_heads;
      a.v_cache[((blk * a.num_kv_heads + h) * a.block_size + off) * vpr + e] = vv;
    }
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

namespace pkv {

int check_write_rope(const void *k, const void *v, const void *q, int32_t num_q_heads,
                     const int64_t *slot_mapping, const int64_t *positions, int64_t num_tokens,
                     const float *cos_sin, int64_t max_position, int32_t rotary_dim,
                     const void *k_cache, const void *v_cache, const pkv_cache_desc *cache) {
  int rc = check_write(k, v, slot_mapping, num_tokens, k_cache, v_cache, cache);
  if (rc) return rc;
  if (rotary_dim <= 0 || rotary_dim % 16 != 0 || rotary_dim > cache->head_dim)
    return set_error(PKV_ERR_UNSUPPORTED,
                     "paged_kv_write_rope: rotary_dim %d must be a positive multiple of 16 <= head_dim",
                     rotary_dim);
  if (max_position <= 0) return set_error(PKV_ERR_SHAPE, "paged_kv_write_rope: max_position <= 0");
  if (q && num_q_heads <= 0) return set_error(PKV_ERR_SHAPE, "paged_kv_write_rope: num_q_heads <= 0");
  if (num_tokens == 0) return PKV_OK;
  if (!positions || !cos_sin) return set_error(PKV_ERR_NULL, "paged_kv_write_rope: NULL positions/cos_sin");
  if (!aligned16(cos_sin) || (q && !aligned16(q)) || (reinterpret_cast<uintptr_t>(positions) & 7u))
    return set_error(PKV_ERR_ALIGN, "paged_kv_write_rope: cos_sin and q 16-byte, positions 8-byte aligned");
  return PKV_OK;
}

int launch_write_rope(const pkv_bf16 *k, const pkv_bf16 *v, pkv_bf16 *q, int32_t num_q_heads,
                      const int64_t *slot_mapping, const int64_t *positions, int64_t num_tokens,
                      const float *cos_sin, int64_t max_position, int32_t rotary_dim,
                      int32_t neox_style, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                      const pkv_cache_desc &c, cudaStream_t stream) {
  if (num_tokens == 0) return PKV_OK;
  RopeArgs a;
  a.k = reinterpret_cast<const uint4 *>(k);
  a.v = reinterpret_cast<const uint4 *>(v);
  a.q = reinterpret_cast<uint4 *>(q);
  a.slot_mapping = slot_mapping;
  a.positions = positions;
  a.cos_sin = cos_sin;
  a.k_cache = reinterpret_cast<uint4 *>(k_cache);
  a.v_cache = reinterpret_cast<uint4 *>(v_cache);
  a.num_tokens = num_tokens;
  a.max_position = max_position;
  a.num_blocks = c.num_blocks;
  a.num_q_heads = q ? num_q_heads : 0;
  a.num_kv_heads = c.num_kv_heads;
  a.block_size = c.block_size;
  a.head_dim = c.head_dim;
  a.rotary_dim = rotary_dim;
  a.neox = neox_style ? 1 : 0;
  const int units = (a.neox ? rotary_dim / 16 : rotary_dim / 8) + (c.head_dim - rotary_dim) / 8;
  const int64_t work = num_tokens * ((int64_t)(c.num_kv_heads + a.num_q_heads) * units +
                                     (int64_t)c.num_kv_heads * (c.head_dim / 8));
  int64_t blocks = (work + 255) / 256;
  if (blocks > 65535LL * 32) blocks = 65535LL * 32;
  kv_write_rope_kernel<<<(unsigned)blocks, 256, 0, stream>>>(a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "paged_kv_write_rope launch");
  return PKV_OK;
}

}  // namespace pkv

PKV_API int paged_kv_write_rope(const pkv_bf16 *k, const pkv_bf16 *v, pkv_bf16 *q,
                                int32_t num_q_heads, const int64_t *slot_mapping,
                                const int64_t *positions, int64_t num_tokens,
                                const float *cos_sin, int64_t max_position, int32_t rotary_dim,
                                int32_t neox_style, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                                const pkv_cache_desc *cache, void *stream) {
  using namespace pkv;
  int rc = check_write_rope(k, v, q, num_q_heads, slot_mapping, positions, num_tokens, cos_sin,
                            max_position, rotary_dim, k_cache, v_cache, cache);
  if (!rc)
    rc = launch_write_rope(k, v, q, num_q_heads, slot_mapping, positions, num_tokens, cos_sin,
                           max_position, rotary_dim, neox_style, k_cache, v_cache, *cache,
                           static_cast<cudaStream_t>(stream));
  if (!rc) clear_error();
  return rc;
}
