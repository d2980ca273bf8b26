// attn_device.cuh -- device pieces of the attention kernels: the per-translation-unit
// error word (decode and prefill; every includer gets its own, read through
// read_tu_errors()), and for the decode kernels the consumer-warp barrier, the
// swizzled stage layout and the TMA box issue of one KV block.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include "pkv_internal.h"

namespace pkv {

// Error word of the including translation unit (PKV_DEVERR_* bits).
static __device__ unsigned int g_attn_errors;

__device__ __forceinline__ void raise_error(unsigned bit) { atomicOr(&g_attn_errors, bit); }

// ORs this translation unit's error word into *flags; clear != 0 resets it.
static inline cudaError_t read_tu_errors(uint32_t *flags, int clear) {
  unsigned int f = 0;
  cudaError_t e = cudaMemcpyFromSymbol(&f, g_attn_errors, sizeof f);
  if (e != cudaSuccess) return e;
  *flags |= f;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_attn_errors, &zero, sizeof zero);
  }
  return e;
}

__device__ __forceinline__ void consumer_bar() {
  asm volatile("bar.sync 1, %0;" ::"n"(kConsumers) : "memory");
}

// Byte offset of 16-byte chunk `dch` (0 .. D/8-1) of key row `key` in a stage tile.
// The tile is D/64 sub-tiles [64 keys][128 B], each filled by 128-byte-swizzled TMA
// boxes: within a 1024-byte atom the chunk position is XORed with key & 7, so the
// eight rows an ldmatrix reads sit in eight different bank groups.
__device__ __forceinline__ uint32_t tile_off(int key, int dch) {
  return (uint32_t)((dch >> 3) * (kChunk * 128) + key * 128 + (((dch & 7) ^ (key & 7)) << 4));
}

// One TMA box (rb rows of one KV block, all head dims) of K and of V.
template <int D>
__device__ __forceinline__ void issue_box(uint32_t dst_k, uint32_t dst_v, const CUtensorMap *tmk,
                                          const CUtensorMap *tmv, int32_t row, uint32_t bar,
                                          uint64_t policy) {
  if constexpr (D == 64) {
    dev::tma_load_2d(dst_k, tmk, 0, row, bar, policy);
    dev::tma_load_2d(dst_v, tmv, 0, row, bar, policy);
  } else {
#pragma unroll
    for (int hh = 0; hh < D / 64; ++hh) {
      const uint32_t o = hh * (kChunk * 128);
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst_k + o),
          "l"(reinterpret_cast<uint64_t>(tmk)), "r"(0), "r"(hh), "r"(row), "r"(bar), "l"(policy)
          : "memory");
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(dst_v + o),
          "l"(reinterpret_cast<uint64_t>(tmv)), "r"(0), "r"(hh), "r"(row), "r"(bar), "l"(policy)
          : "memory");
    }
  }
}


}  // namespace pkv
