// pkv_decode.cu -- paged decode attention: single-pass / flash-decoding partition
// kernel, log-sum-exp combine kernel, and the host launcher.
//
// What is computed ("mini-vLLM" README, paged KV-cache paragraph and M4 test row;
// "vLLM-Style Llama Inference Engine", Features and scope / How it works;
// "llm-stack", Serving engine: the decode query is not causally masked):
//   for sequence b, query head h, kv head g = h / G, positions t < L_b:
//     K_t = k_cache[block_tables[b][t / BS]][g][t % BS],  s_t = scale * <q, K_t>,
//     out = sum_t softmax(s)_t V_t.
// The flash-decoding split and its merge follow the online-softmax algebra of
// FlashAttention-2 (the reference the first page lists).
//
// Design (GB300, sm_103a).  The path is HBM-bound: each K/V byte is read once and
// feeds G fused multiply-adds per query head group.  One CTA owns one (sequence,
// kv head, partition) and reads every K/V row of that range exactly once for all
// G query heads of the group.
//  * Staging: a producer warp walks the block table and issues 2-D/3-D tiled TMA
//    loads (cp.async.bulk.tensor, 128-byte swizzle, L2 evict-first) of whole KV
//    blocks into a ring of STAGES shared-memory stages of 64 keys each; mbarriers
//    with transaction counts signal "full", consumer arrivals signal "empty".
//  * Compute: four consumer warps take 16 keys of each stage.  The tiny products
//    S^T = K_tile . Q^T (16 keys x 8 heads x D) and O^T += V^T . P^T run on the
//    tensor pipe (mma.sync m16n8k16, bf16 in, fp32 accumulate); the query group is
//    padded to 8 heads.  P is fed as a bf16 hi + lo pair, so the products keep
//    ~16 significant bits.  Online softmax in fp32 (base 2), warp-shuffle maxima.
//  * Each warp keeps its own running (m, l, O); the four are merged through shared
//    memory at the end.  Single pass: bf16 output.  Split: normalised fp32 o_part
//    and natural-log lse_part, merged by combine_kernel.
// Every wait is bounded (about 2 s); on a timeout the kernel raises
// PKV_DEVERR_TIMEOUT and unwinds instead of hanging.
#include <cuda.h>  // CUtensorMap and its enums (header only; the entry point is fetched at run time)
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {

constexpr int kChunk = 64;          // keys per pipeline stage
constexpr int kConsumerWarps = 4;   // 16 keys each
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kMaxGroup = 8;        // query heads per kv head (one mma N tile)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

__device__ unsigned int g_decode_errors;

struct DecodeArgs {
  const uint16_t *q;           // [B][Hq][D] bf16
  const int32_t *block_tables; // [B][max_blocks]
  const int32_t *context_lens; // [B]
  uint16_t *out;               // single pass: [B][Hq][D] bf16
  float *o_part;               // split: [B][Hq][n_parts][D]
  float *lse_part;             // split: [B][Hq][n_parts]
  int64_t num_blocks;
  int32_t max_blocks, max_context_len, num_q_heads, num_kv_heads, group;
  int32_t block_size, log2_bs, box_rows, partition_tokens, n_parts, split;
  float scale_log2;            // scale * log2(e)
};

// Byte offset of 16-byte chunk `dch` (0 .. D/8-1) of key row `key` in a stage tile.
// The tile is D/64 sub-tiles [64 keys][128 B], each filled by 128-byte-swizzled TMA
// boxes: within a 1024-byte atom the chunk position is XORed with key & 7, so the
// eight rows an ldmatrix reads sit in eight different bank groups.
__device__ __forceinline__ uint32_t tile_off(int key, int dch) {
  return (uint32_t)((dch >> 3) * (kChunk * 128) + key * 128 + (((dch & 7) ^ (key & 7)) << 4));
}

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

template <int D, int STAGES>
__global__ void __launch_bounds__(kThreads, 2)
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
  constexpr int kTileBytes = kChunk * D * 2;  // K (or V) bytes of one stage
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int KS = D / 16;                  // 16-wide k steps / m tiles over the head dim

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t bar_full = base + STAGES * kStageBytes;
  const uint32_t bar_empty = bar_full + STAGES * 8;
  int *const s_flag = reinterpret_cast<int *>(base_ptr + STAGES * kStageBytes + STAGES * 16);

  const int part = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  int L = __ldg(a.context_lens + b);
  const int cap = (int)min((int64_t)a.max_blocks * a.block_size, (int64_t)a.max_context_len);
  if (L < 0 || L > cap) {
    if (tid == 0 && part == 0) atomicOr(&g_decode_errors, (unsigned)PKV_DEVERR_CONTEXT_LEN);
    L = L < 0 ? 0 : cap;
  }
  const int t_begin = part * a.partition_tokens;
  if (t_begin >= L) {
    if (!a.split && part == 0) {  // empty context: zero output
      uint16_t *o = a.out + ((int64_t)b * a.num_q_heads + g * a.group) * D;
      for (int i = tid; i < a.group * D; i += kThreads) o[i] = 0;
    }
    return;
  }
  const int t_end = min(t_begin + a.partition_tokens, L);
  const int n_chunks = (t_end - t_begin + kChunk - 1) / kChunk;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      dev::mbar_init(bar_full + 8 * s, 1);
      dev::mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    *s_flag = 0;
    dev::fence_mbar_init();
  }
  __syncthreads();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------- producer warp
    const uint64_t policy = dev::policy_evict_first();
    const int32_t *trow = a.block_tables + (int64_t)b * a.max_blocks;
    const int rb = a.box_rows;                    // keys per TMA box = min(BS, 64)
    const uint32_t box_bytes = (uint32_t)rb * 128u;  // per 64-dim half
    const int lb_last = (t_end - 1) >> a.log2_bs;
    int win = t_begin >> a.log2_bs;               // lanes hold table entries [win, win + 32)
    int tb = (win + lane <= lb_last) ? __ldg(trow + win + lane) : 0;
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % STAGES;
      if (c >= STAGES &&
          !__all_sync(0xffffffffu, dev::mbar_wait(bar_empty + 8 * s, ((c / STAGES) - 1) & 1))) {
        if (lane == 0) {
          atomicOr(&g_decode_errors, (unsigned)PKV_DEVERR_TIMEOUT);
          *s_flag = 1;
        }
        break;
      }
      const int k0 = t_begin + c * kChunk;
      const int nk = min(kChunk, t_end - k0);
      const int nbox = (nk + rb - 1) / rb;
      const int lb_hi = (k0 + (nbox - 1) * rb) >> a.log2_bs;
      if (lb_hi >= win + 32) {  // slide the table window
        win = k0 >> a.log2_bs;
        tb = (win + lane <= lb_last) ? __ldg(trow + win + lane) : 0;
      }
      const int key = k0 + lane * rb;  // first key of this lane's box
      const int src = min(max((key >> a.log2_bs) - win, 0), 31);
      const int64_t phys_raw = __shfl_sync(0xffffffffu, tb, src);
      if (lane == 0) dev::mbar_arrive_expect_tx(bar_full + 8 * s, 2u * nbox * box_bytes * (D / 64));
      __syncwarp();
      if (lane < nbox) {
        int64_t phys = phys_raw;
        if (phys < 0 || phys >= a.num_blocks) {
          atomicOr(&g_decode_errors, (unsigned)PKV_DEVERR_BLOCK_ID);
          phys = 0;
        }
        const int off = key & (a.block_size - 1);
        const int32_t row = (int32_t)((phys * a.num_kv_heads + g) * a.block_size + off);
        const uint32_t dk = base + s * kStageBytes + lane * box_bytes;
        issue_box<D>(dk, dk + kTileBytes, &tmk, &tmv, row, bar_full + 8 * s, policy);
      }
      __syncwarp();
    }
  } else {
    // ----------------------------------------------------------- consumer warps
    const int gid = lane >> 2, tig = lane & 3;  // mma group id / thread in group
    uint32_t qb[KS][2];
    {
      const bool hv = gid < a.group;
      const uint32_t *qrow = reinterpret_cast<const uint32_t *>(
          a.q + ((int64_t)b * a.num_q_heads + g * a.group + (hv ? gid : 0)) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[ks][0] = hv ? __ldg(qrow + 8 * ks + tig) : 0u;
        qb[ks][1] = hv ? __ldg(qrow + 8 * ks + 4 + tig) : 0u;
      }
    }
    float o[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;  // heads 2*tig, 2*tig+1

    const int lj = lane >> 3, lr = lane & 7;  // ldmatrix: matrix index / row within it
    // QK operand A = K rows: matrices (keys 0-7 | 8-15) x (dims lo | hi) of a k step.
    const int qk_key = 16 * warp + lr + ((lj & 1) << 3), qk_dsel = lj >> 1;
    // PV operand A = V^T: matrices (keys 0-7, dims lo), (keys 0-7, dims hi), (keys 8-15, ...).
    const int pv_key = 16 * warp + lr + ((lj >> 1) << 3), pv_dsel = lj & 1;

    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % STAGES;
      if (!__all_sync(0xffffffffu, dev::mbar_wait(bar_full + 8 * s, (c / STAGES) & 1))) {
        if (lane == 0) {
          atomicOr(&g_decode_errors, (unsigned)PKV_DEVERR_TIMEOUT);
          *s_flag = 1;
        }
        break;
      }
      const int key0 = t_begin + c * kChunk + 16 * warp;
      const int nvalid = min(16, t_end - key0);
      if (nvalid > 0) {
        const uint32_t kb = base + s * kStageBytes;
        const uint32_t vb = kb + kTileBytes;
        // S^T (16 keys x 8 heads) = K_tile . Q^T
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t ak[4];
          dev::ldsm_x4(ak, kb + tile_off(qk_key, 2 * ks + qk_dsel));
          dev::mma_bf16_16816(sc, ak, qb[ks][0], qb[ks][1]);
        }
        // scale to base 2, mask keys past the range
        const bool v0 = gid < nvalid, v1 = gid + 8 < nvalid;
        const float s0 = v0 ? sc[0] * a.scale_log2 : -INFINITY;
        const float s1 = v0 ? sc[1] * a.scale_log2 : -INFINITY;
        const float s2 = v1 ? sc[2] * a.scale_log2 : -INFINITY;
        const float s3 = v1 ? sc[3] * a.scale_log2 : -INFINITY;
        float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
        for (int x = 4; x < 32; x <<= 1) {
          mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
          mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
        }
        const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
        const float al0 = dev::ex2(m0 - mn0), al1 = dev::ex2(m1 - mn1);
        const float p0 = dev::ex2(s0 - mn0), p1 = dev::ex2(s1 - mn1);
        const float p2 = dev::ex2(s2 - mn0), p3 = dev::ex2(s3 - mn1);
        l0 = l0 * al0 + (p0 + p2);
        l1 = l1 * al1 + (p1 + p3);
        m0 = mn0;
        m1 = mn1;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[mt][0] *= al0;
          o[mt][1] *= al1;
          o[mt][2] *= al0;
          o[mt][3] *= al1;
        }
        // P^T as the B operand: bf16 hi part and the bf16 residual, transposed
        const uint32_t h01 = dev::pack_bf16x2(p0, p1), h23 = dev::pack_bf16x2(p2, p3);
        const uint32_t r01 = dev::pack_bf16x2(p0 - dev::bf16lo_to_f32(h01), p1 - dev::bf16hi_to_f32(h01));
        const uint32_t r23 = dev::pack_bf16x2(p2 - dev::bf16lo_to_f32(h23), p3 - dev::bf16hi_to_f32(h23));
        const uint32_t bh0 = dev::movmatrix_trans(h01), bh1 = dev::movmatrix_trans(h23);
        const uint32_t bl0 = dev::movmatrix_trans(r01), bl1 = dev::movmatrix_trans(r23);
        // O^T (D x 8 heads) += V^T . P^T; rows of V past the range are zeroed in
        // registers (never multiply an unloaded row: 0 * NaN would poison O)
        uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
        if (nvalid < 16) {
          const int kk = 2 * tig;
          mlo = (kk < nvalid ? 0x0000ffffu : 0u) | (kk + 1 < nvalid ? 0xffff0000u : 0u);
          mhi = (kk + 8 < nvalid ? 0x0000ffffu : 0u) | (kk + 9 < nvalid ? 0xffff0000u : 0u);
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          uint32_t av[4];
          dev::ldsm_x4_trans(av, vb + tile_off(pv_key, 2 * mt + pv_dsel));
          av[0] &= mlo;
          av[1] &= mlo;
          av[2] &= mhi;
          av[3] &= mhi;
          dev::mma_bf16_16816(o[mt], av, bh0, bh1);
          dev::mma_bf16_16816(o[mt], av, bl0, bl1);
        }
      }
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(bar_empty + 8 * s);
    }

    // ---- merge the four warps' (m, l, O) through shared memory
#pragma unroll
    for (int x = 4; x < 32; x <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, x);
      l1 += __shfl_xor_sync(0xffffffffu, l1, x);
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");  // stages are free now
    float *const red_o = reinterpret_cast<float *>(base_ptr);  // [warps][8 heads][D]
    float *const red_m = red_o + kConsumerWarps * kMaxGroup * D;  // [warps][8]
    float *const red_l = red_m + kConsumerWarps * kMaxGroup;      // [warps][8]
    if (gid == 0) {
      red_m[warp * kMaxGroup + 2 * tig] = m0;
      red_m[warp * kMaxGroup + 2 * tig + 1] = m1;
      red_l[warp * kMaxGroup + 2 * tig] = l0;
      red_l[warp * kMaxGroup + 2 * tig + 1] = l1;
    }
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) {
      float *r0 = red_o + (warp * kMaxGroup + 2 * tig) * D + 16 * mt + gid;
      float *r1 = r0 + D;
      r0[0] = o[mt][0];
      r1[0] = o[mt][1];
      r0[8] = o[mt][2];
      r1[8] = o[mt][3];
    }
    asm volatile("bar.sync 1, %0;" ::"n"(kConsumerWarps * 32) : "memory");
    const int64_t head0 = (int64_t)b * a.num_q_heads + g * a.group;
    for (int i = tid; i < a.group * D; i += kConsumerWarps * 32) {
      const int h = i / D, d = i - h * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, red_m[w * kMaxGroup + h]);
      float num = 0.f, den = 0.f;
#pragma unroll
      for (int w = 0; w < kConsumerWarps; ++w) {
        const float wt = dev::ex2(red_m[w * kMaxGroup + h] - M);
        num += wt * red_o[(w * kMaxGroup + h) * D + d];
        den += wt * red_l[w * kMaxGroup + h];
      }
      const float val = num / den;
      if (a.split) {
        const int64_t row = (head0 + h) * a.n_parts + part;
        a.o_part[row * D + d] = val;
        if (d == 0) a.lse_part[row] = (M + log2f(den)) * kLn2;
      } else {
        a.out[(head0 + h) * D + d] = (uint16_t)(dev::pack_bf16x2(val, 0.f) & 0xffffu);
      }
    }
  }

  // ---- a timed-out wait leaves copies possibly in flight: wait for them (bounded)
  __syncthreads();
  if (tid == 0 && *s_flag) {
    for (int s = 0; s < STAGES; ++s) {
      const int c_last = s + ((n_chunks - 1 - s) / STAGES) * STAGES;  // last chunk on stage s
      if (c_last >= 0 && c_last < n_chunks) (void)dev::mbar_wait(bar_full + 8 * s, (c_last / STAGES) & 1);
    }
  }
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge: one CTA per (sequence, query head).  Thread groups of D/4
// threads each read one partition row with float4 loads; groups take partitions
// round robin and are summed through shared memory.
template <int D>
__global__ void __launch_bounds__(128)
    combine_kernel(uint16_t *__restrict__ out, const float *__restrict__ o_part,
                   const float *__restrict__ lse_part, const int32_t *__restrict__ context_lens,
                   int32_t max_context_len, int32_t num_q_heads, int32_t partition_tokens,
                   int32_t n_parts) {
  constexpr int TPR = D / 4;          // threads per partition row
  constexpr int NGRP = 128 / TPR;     // partition groups
  __shared__ float s_red[NGRP][D];
  __shared__ float s_den[NGRP];
  __shared__ float s_max[4];
  const int row = blockIdx.x;         // b * Hq + h
  const int b = row / num_q_heads;
  const int tid = threadIdx.x, grp = tid / TPR, col = tid % TPR;
  int L = __ldg(context_lens + b);
  if (L < 0 || L > max_context_len) {
    if (tid == 0) atomicOr(&g_decode_errors, (unsigned)PKV_DEVERR_CONTEXT_LEN);
    L = L < 0 ? 0 : max_context_len;
  }
  const int n = (L + partition_tokens - 1) / partition_tokens;
  const float *lse = lse_part + (int64_t)row * n_parts;
  const float4 *op = reinterpret_cast<const float4 *>(o_part + (int64_t)row * n_parts * D);
  uint2 *o2 = reinterpret_cast<uint2 *>(out + (int64_t)row * D);
  if (n == 0) {
    if (tid < TPR) o2[tid] = make_uint2(0u, 0u);
    return;
  }
  float M = -INFINITY;
  for (int p = tid; p < n; p += 128) M = fmaxf(M, __ldg(lse + p));
#pragma unroll
  for (int x = 16; x > 0; x >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, x));
  if ((tid & 31) == 0) s_max[tid >> 5] = M;
  __syncthreads();
  M = fmaxf(fmaxf(s_max[0], s_max[1]), fmaxf(s_max[2], s_max[3]));
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  float den = 0.f;
#pragma unroll 4
  for (int p = grp; p < n; p += NGRP) {
    const float w = dev::ex2((__ldg(lse + p) - M) * kLog2e);
    const float4 x = __ldg(op + (int64_t)p * TPR + col);
    acc.x += w * x.x;
    acc.y += w * x.y;
    acc.z += w * x.z;
    acc.w += w * x.w;
    den += w;
  }
  s_red[grp][4 * col + 0] = acc.x;
  s_red[grp][4 * col + 1] = acc.y;
  s_red[grp][4 * col + 2] = acc.z;
  s_red[grp][4 * col + 3] = acc.w;
  if (col == 0) s_den[grp] = den;
  __syncthreads();
  if (grp == 0) {
    float t[4] = {0.f, 0.f, 0.f, 0.f}, dsum = 0.f;
#pragma unroll
    for (int q = 0; q < NGRP; ++q) {
#pragma unroll
      for (int j = 0; j < 4; ++j) t[j] += s_red[q][4 * col + j];
      dsum += s_den[q];
    }
    const float inv = 1.f / dsum;
    o2[col] = make_uint2(dev::pack_bf16x2(t[0] * inv, t[1] * inv),
                         dev::pack_bf16x2(t[2] * inv, t[3] * inv));
  }
}

// ---------------------------------------------------------------------------
// Host side.

static thread_local char g_msg[512];

int set_error(int code, const char *fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_msg, sizeof g_msg, fmt, ap);
  va_end(ap);
  return code;
}

void clear_error() { g_msg[0] = '\0'; }

int cuda_error(cudaError_t e, const char *what) {
  return set_error(PKV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_mu;
int g_sms[kMaxDevices];            // SM count per device (0 = not queried)
bool g_attr_set[kMaxDevices][2];   // dynamic smem attribute set, per head_dim variant

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int get_encoder() {
  if (g_encode) return PKV_OK;
  void *fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                   cudaEnableDefault, &q);
  if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || !fn)
    return set_error(PKV_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  return PKV_OK;
}

int device_sms(int *sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (dev < 0 || dev >= kMaxDevices) return set_error(PKV_ERR_CUDA, "device index %d", dev);
  if (!g_sms[dev]) {
    int n = 0;
    e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute");
    g_sms[dev] = n;
  }
  *sms = g_sms[dev];
  return PKV_OK;
}

// A small cache of encoded tensor maps, keyed by (pointer, pool shape).
struct MapEntry {
  const void *ptr;
  int64_t nb;
  int32_t hkv, bs, d;
  CUtensorMap map;
};
MapEntry g_maps[16];
int g_maps_next = 0;

int tensor_map(const void *cache_ptr, const pkv_cache_desc &c, CUtensorMap *out) {
  for (const MapEntry &m : g_maps)
    if (m.ptr == cache_ptr && m.nb == c.num_blocks && m.hkv == c.num_kv_heads &&
        m.bs == c.block_size && m.d == c.head_dim) {
      *out = m.map;
      return PKV_OK;
    }
  int rc = get_encoder();
  if (rc) return rc;
  const uint64_t rows = (uint64_t)c.num_blocks * c.num_kv_heads * c.block_size;
  const uint32_t box_rows = (uint32_t)(c.block_size < kChunk ? c.block_size : kChunk);
  CUtensorMap map;
  CUresult r;
  if (c.head_dim == 64) {
    cuuint64_t dims[2] = {64, rows};
    cuuint64_t strides[1] = {128};
    cuuint32_t box[2] = {64, box_rows};
    cuuint32_t es[2] = {1, 1};
    r = g_encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(cache_ptr), dims,
                 strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {64, (cuuint64_t)(c.head_dim / 64), rows};
    cuuint64_t strides[2] = {128, (cuuint64_t)c.head_dim * 2};
    cuuint32_t box[3] = {64, 1, box_rows};
    cuuint32_t es[3] = {1, 1, 1};
    r = g_encode(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(cache_ptr), dims,
                 strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                 CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return set_error(PKV_ERR_CUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
  MapEntry &m = g_maps[g_maps_next];
  g_maps_next = (g_maps_next + 1) % 16;
  m = MapEntry{cache_ptr, c.num_blocks, c.num_kv_heads, c.block_size, c.head_dim, map};
  *out = map;
  return PKV_OK;
}

constexpr int stages_for(int d) { return d == 64 ? 4 : 3; }
constexpr size_t smem_for(int d) {
  return 1024 + (size_t)stages_for(d) * 2 * kChunk * d * 2 + stages_for(d) * 16 + 16;
}

bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int ilog2(int x) {
  int r = 0;
  while ((1 << r) < x) ++r;
  return r;
}

// Checks shared by the split, single-pass and combined entry points.
int check_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *bt,
                 int32_t max_blocks, const int32_t *lens, int32_t max_len, int32_t num_seqs,
                 int32_t hq, const pkv_cache_desc *c, const char *fn) {
  if (!c) return set_error(PKV_ERR_NULL, "%s: cache descriptor is NULL", fn);
  if (num_seqs < 0 || hq <= 0) return set_error(PKV_ERR_SHAPE, "%s: num_seqs/num_q_heads", fn);
  if (c->num_blocks <= 0 || c->num_kv_heads <= 0 || c->block_size <= 0 || c->head_dim <= 0)
    return set_error(PKV_ERR_SHAPE, "%s: cache sizes must be positive", fn);
  if (hq % c->num_kv_heads != 0)
    return set_error(PKV_ERR_SHAPE, "%s: num_q_heads %d is not a multiple of num_kv_heads %d", fn,
                     hq, c->num_kv_heads);
  if (hq / c->num_kv_heads > kMaxGroup)
    return set_error(PKV_ERR_UNSUPPORTED, "%s: query group %d > %d", fn, hq / c->num_kv_heads,
                     kMaxGroup);
  if (c->head_dim != 64 && c->head_dim != 128)
    return set_error(PKV_ERR_UNSUPPORTED, "%s: head_dim %d (built: 64, 128)", fn, c->head_dim);
  if (!is_pow2(c->block_size) || c->block_size < 8 || c->block_size > 256)
    return set_error(PKV_ERR_UNSUPPORTED, "%s: block_size %d (built: powers of two 8..256)", fn,
                     c->block_size);
  if (num_seqs > 65535) return set_error(PKV_ERR_UNSUPPORTED, "%s: num_seqs > 65535", fn);
  if ((uint64_t)c->num_blocks * c->num_kv_heads * c->block_size > 0x7fffffffull)
    return set_error(PKV_ERR_UNSUPPORTED, "%s: pool has more than 2^31-1 rows", fn);
  if (max_blocks <= 0 || max_len < 0 || (int64_t)max_len > (int64_t)max_blocks * c->block_size)
    return set_error(PKV_ERR_SHAPE, "%s: need 0 <= max_context_len <= max_blocks_per_seq * block_size", fn);
  if (num_seqs > 0 && (!q || !k_cache || !v_cache || !bt || !lens))
    return set_error(PKV_ERR_NULL, "%s: NULL tensor pointer", fn);
  if (num_seqs > 0 && (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache)))
    return set_error(PKV_ERR_ALIGN, "%s: q, k_cache and v_cache must be 16-byte aligned", fn);
  return PKV_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

template <int D>
int launch_decode(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                  const int32_t *bt, int32_t max_blocks, const int32_t *lens, int32_t max_len,
                  int32_t num_seqs, int32_t hq, const pkv_cache_desc &c, float scale,
                  int32_t P, int split, pkv_bf16 *out, float *o_part, float *lse_part,
                  cudaStream_t stream) {
  CUtensorMap tmk, tmv;
  int rc;
  {
    std::lock_guard<std::mutex> lk(g_mu);
    if ((rc = tensor_map(k_cache, c, &tmk))) return rc;
    if ((rc = tensor_map(v_cache, c, &tmv))) return rc;
    int dev = 0;
    cudaGetDevice(&dev);
    const int vi = D == 64 ? 0 : 1;
    if (dev >= 0 && dev < kMaxDevices && !g_attr_set[dev][vi]) {
      cudaError_t e = cudaFuncSetAttribute(decode_kernel<D, stages_for(D)>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)smem_for(D));
      if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
      g_attr_set[dev][vi] = true;
    }
  }
  DecodeArgs a;
  a.q = q;
  a.block_tables = bt;
  a.context_lens = lens;
  a.out = out;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.num_blocks = c.num_blocks;
  a.max_blocks = max_blocks;
  a.max_context_len = max_len;
  a.num_q_heads = hq;
  a.num_kv_heads = c.num_kv_heads;
  a.group = hq / c.num_kv_heads;
  a.block_size = c.block_size;
  a.log2_bs = ilog2(c.block_size);
  a.box_rows = c.block_size < kChunk ? c.block_size : kChunk;
  a.partition_tokens = P;
  a.n_parts = (max_len + P - 1) / P;
  a.split = split;
  a.scale_log2 = scale * kLog2e;
  dim3 grid((unsigned)a.n_parts, (unsigned)c.num_kv_heads, (unsigned)num_seqs);
  decode_kernel<D, stages_for(D)><<<grid, kThreads, smem_for(D), stream>>>(tmk, tmv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "decode_kernel launch");
  return PKV_OK;
}

int launch_combine(pkv_bf16 *out, const float *o_part, const float *lse_part, const int32_t *lens,
                   int32_t max_len, int32_t num_seqs, int32_t hq, int32_t d, int32_t P,
                   cudaStream_t stream) {
  const int n_parts = (max_len + P - 1) / P;
  const unsigned rows = (unsigned)num_seqs * (unsigned)hq;
  if (d == 64)
    combine_kernel<64><<<rows, 128, 0, stream>>>(out, o_part, lse_part, lens, max_len, hq, P, n_parts);
  else
    combine_kernel<128><<<rows, 128, 0, stream>>>(out, o_part, lse_part, lens, max_len, hq, P, n_parts);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "combine_kernel launch");
  return PKV_OK;
}

int32_t plan(int32_t num_seqs, int32_t hkv, int32_t max_len, int32_t sms) {
  if (num_seqs <= 0 || hkv <= 0 || max_len <= 256) return 0;
  const int64_t units = (int64_t)num_seqs * hkv;
  const int64_t target = 4LL * sms;  // CTAs wanted: a few per SM
  int32_t P = 512;
  while (P > 128 && units * ((max_len + P - 1) / P) < target) P /= 2;
  if ((max_len + P - 1) / P <= 1) return 0;
  return P;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

PKV_API int32_t paged_decode_plan(int32_t num_seqs, int32_t num_kv_heads, int32_t max_context_len,
                                  int32_t num_sms) {
  if (num_sms <= 0) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (device_sms(&num_sms) != PKV_OK || num_sms <= 0) num_sms = 148;
  }
  return plan(num_seqs, num_kv_heads, max_context_len, num_sms);
}

PKV_API size_t paged_decode_split_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                                 int32_t head_dim, int32_t max_context_len,
                                                 int32_t partition_tokens) {
  if (num_seqs <= 0 || num_q_heads <= 0 || head_dim <= 0 || max_context_len <= 0 ||
      partition_tokens <= 0)
    return 0;
  const size_t parts = (size_t)((max_context_len + partition_tokens - 1) / partition_tokens);
  const size_t rows = (size_t)num_seqs * num_q_heads * parts;
  return align256(rows * head_dim * sizeof(float)) + align256(rows * sizeof(float));
}

PKV_API size_t paged_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads,
                                           int32_t num_kv_heads, int32_t head_dim,
                                           int32_t max_context_len) {
  const int32_t P = paged_decode_plan(num_seqs, num_kv_heads, max_context_len, 0);
  if (P == 0) return 0;
  return paged_decode_split_workspace_size(num_seqs, num_q_heads, head_dim, max_context_len, P);
}

PKV_API int paged_decode_split(float *o_part, float *lse_part, const pkv_bf16 *q,
                               const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                               const int32_t *block_tables, int32_t max_blocks_per_seq,
                               const int32_t *context_lens, int32_t max_context_len,
                               int32_t num_seqs, int32_t num_q_heads, const pkv_cache_desc *cache,
                               float scale, int32_t partition_tokens, void *stream) {
  int rc = check_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        max_context_len, num_seqs, num_q_heads, cache, "paged_decode_split");
  if (rc) return rc;
  if (partition_tokens <= 0 || partition_tokens % kChunk != 0)
    return set_error(PKV_ERR_SHAPE, "paged_decode_split: partition_tokens %d is not a positive multiple of %d",
                     partition_tokens, kChunk);
  if (num_seqs == 0 || max_context_len == 0) {
    clear_error();
    return PKV_OK;
  }
  if (!o_part || !lse_part) return set_error(PKV_ERR_NULL, "paged_decode_split: NULL o_part/lse_part");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  rc = cache->head_dim == 64
           ? launch_decode<64>(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                               max_context_len, num_seqs, num_q_heads, *cache, scale,
                               partition_tokens, 1, nullptr, o_part, lse_part, s)
           : launch_decode<128>(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                                max_context_len, num_seqs, num_q_heads, *cache, scale,
                                partition_tokens, 1, nullptr, o_part, lse_part, s);
  if (!rc) clear_error();
  return rc;
}

PKV_API int paged_decode_combine(pkv_bf16 *out, const float *o_part, const float *lse_part,
                                 const int32_t *context_lens, int32_t max_context_len,
                                 int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                 int32_t partition_tokens, void *stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || max_context_len < 0)
    return set_error(PKV_ERR_SHAPE, "paged_decode_combine: bad sizes");
  if (head_dim != 64 && head_dim != 128)
    return set_error(PKV_ERR_UNSUPPORTED, "paged_decode_combine: head_dim %d", head_dim);
  if (partition_tokens <= 0)
    return set_error(PKV_ERR_SHAPE, "paged_decode_combine: partition_tokens must be positive");
  if ((int64_t)num_seqs * num_q_heads > 0x7fffffffLL)
    return set_error(PKV_ERR_UNSUPPORTED, "paged_decode_combine: too many rows");
  if (num_seqs == 0) {
    clear_error();
    return PKV_OK;
  }
  if (!out || !context_lens || (max_context_len > 0 && (!o_part || !lse_part)))
    return set_error(PKV_ERR_NULL, "paged_decode_combine: NULL pointer");
  if ((reinterpret_cast<uintptr_t>(out) & 7u) || (o_part && !aligned16(o_part)))
    return set_error(PKV_ERR_ALIGN, "paged_decode_combine: out must be 8-byte and o_part 16-byte aligned");
  int rc = launch_combine(out, o_part, lse_part, context_lens, max_context_len, num_seqs,
                          num_q_heads, head_dim, partition_tokens > 0 ? partition_tokens : 1,
                          static_cast<cudaStream_t>(stream));
  if (!rc) clear_error();
  return rc;
}

PKV_API int paged_decode_attention(pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                   const pkv_bf16 *v_cache, const int32_t *block_tables,
                                   int32_t max_blocks_per_seq, const int32_t *context_lens,
                                   int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                                   const pkv_cache_desc *cache, float scale, void *workspace,
                                   size_t workspace_bytes, void *stream) {
  int rc = check_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        max_context_len, num_seqs, num_q_heads, cache, "paged_decode_attention");
  if (rc) return rc;
  if (num_seqs == 0) {
    clear_error();
    return PKV_OK;
  }
  if (!out) return set_error(PKV_ERR_NULL, "paged_decode_attention: out is NULL");
  if (reinterpret_cast<uintptr_t>(out) & 7u)
    return set_error(PKV_ERR_ALIGN, "paged_decode_attention: out must be 8-byte aligned");
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int32_t P = paged_decode_plan(num_seqs, cache->num_kv_heads, max_context_len, 0);
  const int D = cache->head_dim;
  if (P == 0) {
    const int32_t Pone = max_context_len > 0 ? ((max_context_len + kChunk - 1) / kChunk) * kChunk : kChunk;
    const int32_t mlen = max_context_len > 0 ? max_context_len : 1;
    rc = D == 64 ? launch_decode<64>(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                     context_lens, mlen, num_seqs, num_q_heads, *cache, scale,
                                     Pone, 0, out, nullptr, nullptr, s)
                 : launch_decode<128>(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                      context_lens, mlen, num_seqs, num_q_heads, *cache, scale,
                                      Pone, 0, out, nullptr, nullptr, s);
    if (!rc) clear_error();
    return rc;
  }
  const size_t need = paged_decode_split_workspace_size(num_seqs, num_q_heads, D, max_context_len, P);
  if (!workspace || workspace_bytes < need)
    return set_error(PKV_ERR_WORKSPACE, "paged_decode_attention: workspace %zu bytes < %zu needed",
                     workspace_bytes, need);
  if (!aligned16(workspace))
    return set_error(PKV_ERR_ALIGN, "paged_decode_attention: workspace must be 16-byte aligned");
  const int n_parts = (max_context_len + P - 1) / P;
  const size_t rows = (size_t)num_seqs * num_q_heads * n_parts;
  float *o_part = static_cast<float *>(workspace);
  float *lse_part = reinterpret_cast<float *>(static_cast<char *>(workspace) +
                                              align256(rows * D * sizeof(float)));
  rc = D == 64 ? launch_decode<64>(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                   context_lens, max_context_len, num_seqs, num_q_heads, *cache,
                                   scale, P, 1, nullptr, o_part, lse_part, s)
               : launch_decode<128>(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    context_lens, max_context_len, num_seqs, num_q_heads, *cache,
                                    scale, P, 1, nullptr, o_part, lse_part, s);
  if (rc) return rc;
  rc = launch_combine(out, o_part, lse_part, context_lens, max_context_len, num_seqs, num_q_heads,
                      D, P, s);
  if (!rc) clear_error();
  return rc;
}

PKV_API int pkv_device_errors(uint32_t *flags, int clear) {
  if (!flags) return set_error(PKV_ERR_NULL, "pkv_device_errors: flags is NULL");
  *flags = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_error(e, "cudaDeviceSynchronize");
  unsigned int f = 0;
  e = cudaMemcpyFromSymbol(&f, g_decode_errors, sizeof f);
  if (e != cudaSuccess) return cuda_error(e, "read decode error word");
  *flags |= f;
  if (clear) {
    const unsigned int zero = 0;
    e = cudaMemcpyToSymbol(g_decode_errors, &zero, sizeof zero);
    if (e != cudaSuccess) return cuda_error(e, "clear decode error word");
  }
  e = read_write_errors(flags, clear);
  if (e != cudaSuccess) return cuda_error(e, "read write error word");
  clear_error();
  return PKV_OK;
}

PKV_API const char *pkv_last_error(void) { return g_msg; }
