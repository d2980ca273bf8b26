// pkv_decode.cu -- paged decode attention: the flash-decoding partition kernel (fused
// with its merge for paged_decode_attention; partials only for paged_decode_split),
// the log-sum-exp combine kernel of paged_decode_combine, and the host launcher.
//
// What is computed ("mini-vLLM" README, paged KV-cache paragraph and M4 test row;
// "vLLM-Style Llama Inference Engine", Features and scope / How it works;
// "llm-stack", Serving engine: the decode query is not causally masked):
//   for sequence b, query head h, kv head g = h / G, positions t < L_b:
//     K_t = k_cache[block_tables[b][t / BS]][g][t % BS],  s_t = scale * <q, K_t>,
//     out = sum_t softmax(s)_t V_t.
// Splitting the keys of one (b, g) into partitions and merging the partitions'
// (output, log-sum-exp) follows the online-softmax algebra of FlashAttention-2 (the
// reference the first page lists).
//
// Design (GB300, sm_103a).  The path is HBM-bound: each K/V byte is read once and
// feeds G fused multiply-adds per query head group.  A CTA streams K/V rows of one
// kv head for all G query heads of the group at once.
//  * Staging: a producer warp walks the block table and issues 2-D/3-D tiled TMA
//    loads (cp.async.bulk.tensor, 128-byte swizzle, L2 evict-first) of whole KV
//    blocks into a ring of shared-memory stages of 64 keys; mbarriers with
//    transaction counts signal "full", consumer-warp arrivals signal "empty".
//  * Compute: four consumer warps take 16 keys of each stage.  S^T = K_tile . Q^T
//    (16 keys x 8 heads x D) and O^T += V^T . P^T run on the tensor pipe
//    (mma.sync m16n8k16, bf16 in, fp32 accumulate); the group is padded to 8 heads;
//    P enters as a bf16 hi + lo pair (~16 significant bits).  Online softmax in fp32
//    (base 2) with warp-shuffle maxima; each warp keeps its own (m, l, O), merged
//    through shared memory at the end of a segment.
//  * decode_kernel: one CTA per (sequence, kv head, partition of P tokens); the
//    launcher sizes P so that few (sequence, kv head) units still fill about one wave
//    of long partitions, and many units take 1024-token partitions.  For
//    paged_decode_attention it runs fused: a sequence with one partition writes bf16
//    directly; otherwise each partition writes its (o, lse) and the last of them to
//    finish (atomic ticket per (sequence, kv head); nobody waits) merges them.  For
//    paged_decode_split it only writes the partials, merged by combine_kernel.
// Every wait is bounded (about 2 s); on a timeout the kernel raises
// PKV_DEVERR_TIMEOUT and unwinds instead of hanging.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <atomic>
#include <mutex>

#include "attn_device.cuh"

namespace pkv {

// ---------------------------------------------------------------------------
// Per-warp state and the per-stage work of a consumer warp.

template <int D>
struct WarpAcc {
  float o[D / 16][4];  // O^T fragment: dims (16*mt + gid, +8) x heads (2*tig, 2*tig+1)
  float m0, m1, l0, l1;  // running max (base 2) and partial sum for heads 2*tig, 2*tig+1
};

template <int D>
__device__ __forceinline__ void acc_reset(WarpAcc<D> &a) {
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) a.o[mt][0] = a.o[mt][1] = a.o[mt][2] = a.o[mt][3] = 0.f;
  a.m0 = a.m1 = -INFINITY;
  a.l0 = a.l1 = 0.f;
}

// QK, online softmax and PV for this warp's 16 keys (nvalid of them in range) of the
// stage whose K tile is at kb and V tile at vb.
template <int D>
__device__ __forceinline__ void warp_tile(WarpAcc<D> &acc, const uint32_t (&qb)[D / 16][2],
                                          uint32_t kb, uint32_t vb, int warp, int lane, int nvalid,
                                          float scale_log2) {
  constexpr int KS = D / 16;
  const int gid = lane >> 2, tig = lane & 3;
  const int lj = lane >> 3, lr = lane & 7;  // ldmatrix: matrix index / row within it
  // QK operand A = K rows: matrices (keys 0-7 | 8-15) x (dims lo | hi) of a k step.
  const int qk_key = 16 * warp + lr + ((lj & 1) << 3), qk_dsel = lj >> 1;
  // PV operand A = V^T: matrices (keys 0-7, dims lo), (keys 0-7, dims hi), (keys 8-15, ...).
  const int pv_key = 16 * warp + lr + ((lj >> 1) << 3), pv_dsel = lj & 1;

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
  const float s0 = v0 ? sc[0] * scale_log2 : -INFINITY;
  const float s1 = v0 ? sc[1] * scale_log2 : -INFINITY;
  const float s2 = v1 ? sc[2] * scale_log2 : -INFINITY;
  const float s3 = v1 ? sc[3] * scale_log2 : -INFINITY;
  float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, x));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, x));
  }
  const float mn0 = fmaxf(acc.m0, mx0), mn1 = fmaxf(acc.m1, mx1);
  const float al0 = dev::ex2(acc.m0 - mn0), al1 = dev::ex2(acc.m1 - mn1);
  const float p0 = dev::ex2(s0 - mn0), p1 = dev::ex2(s1 - mn1);
  const float p2 = dev::ex2(s2 - mn0), p3 = dev::ex2(s3 - mn1);
  acc.l0 = acc.l0 * al0 + (p0 + p2);
  acc.l1 = acc.l1 * al1 + (p1 + p3);
  acc.m0 = mn0;
  acc.m1 = mn1;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    acc.o[mt][0] *= al0;
    acc.o[mt][1] *= al1;
    acc.o[mt][2] *= al0;
    acc.o[mt][3] *= al1;
  }
  // P^T as the B operand: bf16 hi part and the bf16 residual, transposed
  const uint32_t h01 = dev::pack_bf16x2(p0, p1), h23 = dev::pack_bf16x2(p2, p3);
  const uint32_t r01 = dev::pack_bf16x2(p0 - dev::bf16lo_to_f32(h01), p1 - dev::bf16hi_to_f32(h01));
  const uint32_t r23 = dev::pack_bf16x2(p2 - dev::bf16lo_to_f32(h23), p3 - dev::bf16hi_to_f32(h23));
  const uint32_t bh0 = dev::movmatrix_trans(h01), bh1 = dev::movmatrix_trans(h23);
  const uint32_t bl0 = dev::movmatrix_trans(r01), bl1 = dev::movmatrix_trans(r23);
  // O^T (D x 8 heads) += V^T . P^T; rows of V past the range are zeroed in registers
  // (never multiply an unloaded row: 0 * NaN would poison O)
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
    dev::mma_bf16_16816(acc.o[mt], av, bh0, bh1);
    dev::mma_bf16_16816(acc.o[mt], av, bl0, bl1);
  }
}

// ---------------------------------------------------------------------------
// The same per-stage work on the CUDA cores (the comparison form of the consumer
// warps; pkv_set_decode_consumer selects it for decode_kernel).  bf16 products are
// exact in fp32, so both forms accumulate the same products in fp32.
//  * QK: lane l takes key 16*warp + (l & 15) and half (l >> 4) of the dims; for each
//    16-byte chunk of its K row it issues mixed-precision FMAs (bf16 x bf16 + fp32,
//    fma.rn.f32.bf16) against the group's query rows, read from shared memory
//    (all lanes of a half read the same address: a broadcast).  The two halves are
//    added with one shuffle per head.
//  * softmax: as the tensor form (base 2, warp-shuffle maxima over the 16 keys); each
//    lane keeps (m, l) for every head, l as its own key's partial sum.
//  * PV: lane l owns dims l*D/32 .. +D/32 of every head; for each valid key it loads
//    those V elements, widens them to fp32 and takes each head's weight from the lane
//    that holds it (shuffle).
template <int D>
struct WarpAccF {
  float o[kMaxGroup][D / 32];   // O: head h, dims lane*(D/32) + v
  float m[kMaxGroup], l[kMaxGroup];
};

template <int D>
__device__ __forceinline__ void accf_reset(WarpAccF<D> &a) {
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
#pragma unroll
    for (int v = 0; v < D / 32; ++v) a.o[h][v] = 0.f;
    a.m[h] = -INFINITY;
    a.l[h] = 0.f;
  }
}

// c + a.lo * b.lo + a.hi * b.hi for bf16 pairs a, b: two mixed-precision FMAs.
__device__ __forceinline__ float fma_bf16x2(uint32_t a, uint32_t b, float c) {
  float d;
  asm("{\n\t.reg .b16 al, ah, bl, bh;\n\t.reg .f32 t;\n\t"
      "mov.b32 {al, ah}, %1;\n\tmov.b32 {bl, bh}, %2;\n\t"
      "fma.rn.f32.bf16 t, al, bl, %3;\n\tfma.rn.f32.bf16 %0, ah, bh, t;\n\t}"
      : "=f"(d)
      : "r"(a), "r"(b), "f"(c));
  return d;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "r"(addr));
  return v;
}

// qs: shared address of the group's query rows [G][D] bf16.
template <int D>
__device__ __forceinline__ void warp_tile_fma(WarpAccF<D> &acc, uint32_t qs, int G, uint32_t kb,
                                              uint32_t vb, int warp, int lane, int nvalid,
                                              float scale_log2) {
  constexpr int VPL = D / 32;  // dims per lane in PV
  constexpr int CH = D / 16;   // 16-byte chunks in half a row
  const int kk = lane & 15, hf = lane >> 4;
  const int key = 16 * warp + kk;
  float s[kMaxGroup];
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) s[h] = 0.f;
#pragma unroll
  for (int c = 0; c < CH; ++c) {
    const int dch = hf * CH + c;
    const uint4 kv = lds128(kb + tile_off(key, dch));
#pragma unroll
    for (int h = 0; h < kMaxGroup; ++h) {
      if (h < G) {
        const uint4 qv = lds128(qs + (uint32_t)(h * D + dch * 8) * 2u);
        float t = fma_bf16x2(kv.x, qv.x, s[h]);
        t = fma_bf16x2(kv.y, qv.y, t);
        t = fma_bf16x2(kv.z, qv.z, t);
        s[h] = fma_bf16x2(kv.w, qv.w, t);
      }
    }
  }
  const bool valid = kk < nvalid;
  float p[kMaxGroup];
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    if (h < G) {
      float sh = s[h] + __shfl_xor_sync(0xffffffffu, s[h], 16);
      sh = valid ? sh * scale_log2 : -INFINITY;
      float mx = sh;
#pragma unroll
      for (int x = 1; x < 16; x <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, x));
      const float mn = fmaxf(acc.m[h], mx);
      const float al = dev::ex2(acc.m[h] - mn);
      p[h] = dev::ex2(sh - mn);
      acc.l[h] = acc.l[h] * al + (hf == 0 ? p[h] : 0.f);
      acc.m[h] = mn;
#pragma unroll
      for (int v = 0; v < VPL; ++v) acc.o[h][v] *= al;
    } else {
      p[h] = 0.f;
    }
  }
  // PV over the valid keys (rows past the range are never read: 0 * NaN would poison O)
  const int d0 = lane * VPL;
  const uint32_t voff = (uint32_t)((d0 & 7) * 2);
#pragma unroll
  for (int t = 0; t < 16; ++t) {
    if (t < nvalid) {
      const uint32_t va = vb + tile_off(16 * warp + t, d0 >> 3) + voff;
      float vf[VPL];
      if constexpr (VPL == 2) {
        uint32_t w;
        asm volatile("ld.shared.b32 %0, [%1];" : "=r"(w) : "r"(va));
        vf[0] = dev::bf16lo_to_f32(w);
        vf[1] = dev::bf16hi_to_f32(w);
      } else {
        uint32_t w0, w1;
        asm volatile("ld.shared.v2.b32 {%0, %1}, [%2];" : "=r"(w0), "=r"(w1) : "r"(va));
        vf[0] = dev::bf16lo_to_f32(w0);
        vf[1] = dev::bf16hi_to_f32(w0);
        vf[2] = dev::bf16lo_to_f32(w1);
        vf[3] = dev::bf16hi_to_f32(w1);
      }
#pragma unroll
      for (int h = 0; h < kMaxGroup; ++h) {
        if (h < G) {
          const float ph = __shfl_sync(0xffffffffu, p[h], t);
#pragma unroll
          for (int v = 0; v < VPL; ++v) acc.o[h][v] = fmaf(ph, vf[v], acc.o[h][v]);
        }
      }
    }
  }
}

// Receive slots the largest case needs: n * ceil(G / n) over cluster sizes n >= 2 and
// groups G <= kMaxGroup.
constexpr int recv_slots_needed() {
  int m = 0;
  for (int n = 2; n <= kMaxClusterParts; ++n)
    for (int g = 1; g <= kMaxGroup; ++g) m = n * ((g + n - 1) / n) > m ? n * ((g + n - 1) / n) : m;
  return m;
}
static_assert(recv_slots_needed() <= kRecvSlots, "cluster merge receive area");

// Merge area of the four warps: red_o [warps][G][D], red_m / red_l [warps][8].
struct MergeArea {
  float *o, *m, *l;
};

// Reduces l over the warp and writes the warp's (m, l, O) for heads < G.
template <int D>
__device__ __forceinline__ void warp_stash(WarpAcc<D> &acc, const MergeArea &r, int G, int warp,
                                           int lane) {
  const int gid = lane >> 2, tig = lane & 3;
  float l0 = acc.l0, l1 = acc.l1;
#pragma unroll
  for (int x = 4; x < 32; x <<= 1) {
    l0 += __shfl_xor_sync(0xffffffffu, l0, x);
    l1 += __shfl_xor_sync(0xffffffffu, l1, x);
  }
  const int h0 = 2 * tig, h1 = h0 + 1;
  if (gid == 0) {
    r.m[warp * kMaxGroup + h0] = acc.m0;
    r.m[warp * kMaxGroup + h1] = acc.m1;
    r.l[warp * kMaxGroup + h0] = l0;
    r.l[warp * kMaxGroup + h1] = l1;
  }
#pragma unroll
  for (int mt = 0; mt < D / 16; ++mt) {
    const int d = 16 * mt + gid;
    if (h0 < G) {
      r.o[(warp * G + h0) * D + d] = acc.o[mt][0];
      r.o[(warp * G + h0) * D + d + 8] = acc.o[mt][2];
    }
    if (h1 < G) {
      r.o[(warp * G + h1) * D + d] = acc.o[mt][1];
      r.o[(warp * G + h1) * D + d + 8] = acc.o[mt][3];
    }
  }
}

// warp_stash for the CUDA-core form: the 16 key lanes' partial sums reduced per head,
// and the warp's (m, l, O) for heads < G written in the same merge-area layout.
template <int D>
__device__ __forceinline__ void warp_stash_fma(WarpAccF<D> &acc, const MergeArea &r, int G,
                                               int warp, int lane) {
  constexpr int VPL = D / 32;
#pragma unroll
  for (int h = 0; h < kMaxGroup; ++h) {
    float l = acc.l[h];
#pragma unroll
    for (int x = 1; x < 32; x <<= 1) l += __shfl_xor_sync(0xffffffffu, l, x);
    if (lane == 0) {
      r.m[warp * kMaxGroup + h] = acc.m[h];
      r.l[warp * kMaxGroup + h] = l;
    }
    if (h < G) {
#pragma unroll
      for (int v = 0; v < VPL; ++v) r.o[(warp * G + h) * D + lane * VPL + v] = acc.o[h][v];
    }
  }
}

// The four warps' softmax states merged for head h, dim d: the normalised output;
// *M2 gets the base-2 max and *den the sum, so lse2 = *M2 + log2(*den).  A warp that
// saw no key has m = -inf and weighs nothing.
template <int D>
__device__ __forceinline__ float cta_merge(const MergeArea &r, int G, int h, int d, float *M2,
                                           float *den) {
  float M = -INFINITY;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, r.m[w * kMaxGroup + h]);
  float num = 0.f, dn = 0.f;
#pragma unroll
  for (int w = 0; w < kConsumerWarps; ++w) {
    const float wt = dev::ex2(r.m[w * kMaxGroup + h] - M);
    num += wt * r.o[(w * G + h) * D + d];
    dn += wt * r.l[w * kMaxGroup + h];
  }
  *M2 = M;
  *den = dn;
  return num / dn;
}

__device__ __forceinline__ uint16_t to_bf16(float x) {
  return (uint16_t)(dev::pack_bf16x2(x, 0.f) & 0xffffu);
}

// Merges the n partition results of one query head -- row p: normalised output
// o_rows[p*D .. p*D+D) and natural-log lse_rows[p] -- into bf16 dst[0 .. D).  One warp:
// each lane owns D/32 dims; partitions are read 8 at a time with all loads in flight
// and folded in with the online-softmax rule.  Loads bypass L1 (__ldcg): the rows were
// written by other CTAs.
template <int D>
__device__ __forceinline__ void merge_rows(uint16_t *dst, const float *o_rows,
                                           const float *lse_rows, int n, int lane) {
  constexpr int VPL = D / 32;
  float M = -INFINITY, den = 0.f, acc[VPL];
#pragma unroll
  for (int v = 0; v < VPL; ++v) acc[v] = 0.f;
  for (int k0 = 0; k0 < n; k0 += 8) {
    float lk[8], ov[8][VPL];
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int k = k0 + u;
      lk[u] = -INFINITY;
#pragma unroll
      for (int v = 0; v < VPL; ++v) ov[u][v] = 0.f;
      if (k < n) {
        lk[u] = __ldcg(lse_rows + k) * kLog2e;
        const float *src = o_rows + (int64_t)k * D + lane * VPL;
        if constexpr (VPL == 2) {
          const float2 t2 = __ldcg(reinterpret_cast<const float2 *>(src));
          ov[u][0] = t2.x;
          ov[u][1] = t2.y;
        } else {
          const float4 t4 = __ldcg(reinterpret_cast<const float4 *>(src));
          ov[u][0] = t4.x;
          ov[u][1] = t4.y;
          ov[u][2] = t4.z;
          ov[u][3] = t4.w;
        }
      }
    }
    float mb = lk[0];
#pragma unroll
    for (int u = 1; u < 8; ++u) mb = fmaxf(mb, lk[u]);
    const float Mn = fmaxf(M, mb);
    const float sc = dev::ex2(M - Mn);
    den *= sc;
#pragma unroll
    for (int v = 0; v < VPL; ++v) acc[v] *= sc;
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const float wt = dev::ex2(lk[u] - Mn);
      den += wt;
#pragma unroll
      for (int v = 0; v < VPL; ++v) acc[v] += wt * ov[u][v];
    }
    M = Mn;
  }
  const float inv = 1.f / den;
  uint16_t *d = dst + lane * VPL;
  if constexpr (VPL == 2) {
    *reinterpret_cast<uint32_t *>(d) = dev::pack_bf16x2(acc[0] * inv, acc[1] * inv);
  } else {
    *reinterpret_cast<uint2 *>(d) = make_uint2(dev::pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                              dev::pack_bf16x2(acc[2] * inv, acc[3] * inv));
  }
}

// Cluster merge of one query head on the CTA that owns it: receive-area rows
// u * hpo + j (u = 0 .. n-1; j = the head's index among the CTA's heads) hold partition
// u's normalised output [D] and its base-2 lse (-inf for a partition without keys).
// One warp; each lane owns D/32 dims.  All -inf (empty context): zeros.
template <int D>
__device__ __forceinline__ void recv_merge_head(uint16_t *dst, const float *recv_o,
                                                const float *recv_l, int j, int hpo, int n,
                                                int lane) {
  constexpr int VPL = D / 32;
  float lk[kMaxClusterParts], ov[kMaxClusterParts][VPL];
  float M = -INFINITY;
#pragma unroll
  for (int u = 0; u < kMaxClusterParts; ++u) {
    lk[u] = -INFINITY;
#pragma unroll
    for (int v = 0; v < VPL; ++v) ov[u][v] = 0.f;
    if (u < n) {
      const int slot = u * hpo + j;
      lk[u] = recv_l[slot];
      const float *src = recv_o + slot * D + lane * VPL;
      if constexpr (VPL == 2) {
        const float2 t2 = *reinterpret_cast<const float2 *>(src);
        ov[u][0] = t2.x;
        ov[u][1] = t2.y;
      } else {
        const float4 t4 = *reinterpret_cast<const float4 *>(src);
        ov[u][0] = t4.x;
        ov[u][1] = t4.y;
        ov[u][2] = t4.z;
        ov[u][3] = t4.w;
      }
    }
    M = fmaxf(M, lk[u]);
  }
  float den = 0.f, acc[VPL];
#pragma unroll
  for (int v = 0; v < VPL; ++v) acc[v] = 0.f;
  if (M != -INFINITY) {
#pragma unroll
    for (int u = 0; u < kMaxClusterParts; ++u) {
      const float wt = dev::ex2(lk[u] - M);  // 0 for an empty partition
      den += wt;
#pragma unroll
      for (int v = 0; v < VPL; ++v) acc[v] += wt * ov[u][v];
    }
  }
  const float inv = den > 0.f ? 1.f / den : 0.f;
  uint16_t *d = dst + lane * VPL;
  if constexpr (VPL == 2) {
    *reinterpret_cast<uint32_t *>(d) = dev::pack_bf16x2(acc[0] * inv, acc[1] * inv);
  } else {
    *reinterpret_cast<uint2 *>(d) = make_uint2(dev::pack_bf16x2(acc[0] * inv, acc[1] * inv),
                                              dev::pack_bf16x2(acc[2] * inv, acc[3] * inv));
  }
}

// ===========================================================================
// decode_kernel: one CTA per (sequence, kv head, partition of P tokens).
// fused = 1 (paged_decode_attention): finished bf16 output, merging partitions itself.
// fused = 0 (paged_decode_split): normalised fp32 partials + natural-log lse only.

struct DecodeArgs {
  const uint16_t *q;           // [B][Hq][D] bf16
  const int32_t *block_tables; // [B][max_blocks]
  const int32_t *context_lens; // [B]
  float *o_part;               // [B][Hq][n_parts][D]
  float *lse_part;             // [B][Hq][n_parts]
  uint16_t *out;               // fused: [B][Hq][D] bf16
  uint32_t *counters;          // fused == 1: [B][Hkv] partitions finished; zero between calls
  int64_t num_blocks;
  int32_t max_blocks, max_context_len, num_q_heads, num_kv_heads, group;
  int32_t block_size, log2_bs, box_rows, partition_tokens, n_parts;
  int32_t fused;               // 0: partials only; 1: ticket merge; 2: cluster merge
  float scale_log2;            // scale * log2(e)
  uint32_t *sched;             // persistent: [0] next dynamic item, [1] CTAs finished
  int32_t num_seqs;            // persistent: sequences in the batch
  int32_t q_wait;              // q is written by the preceding kernel: read it after that grid
};

// The end of one partition (any mode but the cluster merge), on the consumer warps
// after warp_stash: a sequence held whole writes its bf16 output; otherwise the
// partition writes its (normalised o, natural-log lse) row and, fused, takes a ticket
// on the (sequence, kv head) counter -- the last partition to arrive merges them all
// (nobody waits).  The barrier orders every thread's partial stores before thread 0's
// ticket, an acquire-release atomic at GPU scope: its release publishes them (it is
// cumulative over what the barrier ordered before it), and for the last partition its
// acquire, passed on by the next barrier, makes the other partitions' rows visible.
template <int D>
__device__ __forceinline__ void finish_partition(const DecodeArgs &a, const MergeArea &r, int b,
                                                 int g, int part, int nparts_b, int tid, int warp,
                                                 int lane, volatile int *s_flag,
                                                 volatile int *s_last) {
  const int64_t head0 = (int64_t)b * a.num_q_heads + g * a.group;
  if (a.fused && nparts_b == 1) {  // the whole sequence is here: finished output
    for (int i = tid; i < a.group * D; i += kConsumers) {
      const int h = i / D, d = i - h * D;
      float M2, den;
      a.out[head0 * D + i] = to_bf16(cta_merge<D>(r, a.group, h, d, &M2, &den));
    }
    return;
  }
  for (int i = tid; i < a.group * D; i += kConsumers) {
    const int h = i / D, d = i - h * D;
    float M2, den;
    const float val = cta_merge<D>(r, a.group, h, d, &M2, &den);
    const int64_t row = (head0 + h) * a.n_parts + part;
    a.o_part[row * D + d] = val;
    if (d == 0) a.lse_part[row] = (M2 + log2f(den)) * kLn2;
  }
  if (!a.fused) return;
  consumer_bar();
  if (tid == 0) {
    int last = 0;
    if (!*s_flag) {
      const unsigned old = dev::atomic_add_acq_rel(a.counters + (int64_t)b * a.num_kv_heads + g, 1u);
      last = (old + 1 == (unsigned)nparts_b);
    }
    *s_last = last;
  }
  consumer_bar();
  if (*s_last) {
    for (int h = warp; h < a.group; h += kConsumerWarps)
      merge_rows<D>(a.out + (head0 + h) * D, a.o_part + (head0 + h) * a.n_parts * D,
                    a.lse_part + (head0 + h) * a.n_parts, nparts_b, lane);
    if (tid == 0) a.counters[(int64_t)b * a.num_kv_heads + g] = 0u;  // ready for the next call
  }
}

template <int D, int STAGES, bool kFma>
__global__ void __launch_bounds__(kThreads, split_occupancy(D))
    decode_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                  const DecodeArgs a) {
  constexpr int kTileBytes = kChunk * D * 2;  // K (or V) bytes of one stage
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int KS = D / 16;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t bar_full = base + STAGES * kStageBytes;
  const uint32_t bar_empty = bar_full + STAGES * 8;
  volatile int *const s_flag =
      reinterpret_cast<volatile int *>(base_ptr + STAGES * kStageBytes + STAGES * 16);
  volatile int *const s_last = s_flag + 1;  // ticket merge: this partition merges
  volatile int *const s_merge_timeout = s_last;  // cluster merge: its wait gave up
  // Cluster merge: a barrier whose phase completes when every CTA of the cluster has
  // pushed its results here, and the area they land in (rows of D floats, then the lse).
  const uint32_t bar_merge = bar_full + STAGES * 16 + 8;
  const uint32_t recv = bar_merge + 8;
  const float *const recv_o =
      reinterpret_cast<const float *>(base_ptr + STAGES * kStageBytes + STAGES * 16 + 16);
  const float *const recv_l = recv_o + kRecvSlots * D;
  // the group's query rows (bf16 [G][D]) for the CUDA-core form of the consumers
  const uint32_t q_area = recv + (uint32_t)(kRecvSlots * (D + 1) * 4);

  // grid: x = partition (fastest), y = kv head, z = sequence
  const int part = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int32_t *trow = a.block_tables + (int64_t)b * a.max_blocks;
  // The first block-table window does not depend on the context length (entries past
  // it are valid memory, just unused), so the producer loads it together with the length.
  const int win0 = (part * a.partition_tokens) >> a.log2_bs;
  int tb0 = 0;
  if (warp == kConsumerWarps && win0 + lane < a.max_blocks) tb0 = __ldg(trow + win0 + lane);
  // consumer warps: the group's query rows, loaded up front into shared memory with one
  // 16-byte load per thread (published by the set-up barrier below; q may be in host
  // memory, where few wide reads beat many narrow ones); the tensor form takes its mma B
  // fragments from there
  uint32_t qb[KS][2];
  if (warp < kConsumerWarps) {
    // In a step whose first kernel rotates q in place, q is read only after that grid.
    if (a.q_wait) asm volatile("griddepcontrol.wait;" ::: "memory");
    const uint16_t *qg = a.q + ((int64_t)b * a.num_q_heads + g * a.group) * D;
    if (tid < a.group * D / 8)
      *reinterpret_cast<uint4 *>(base_ptr + (q_area - base) + tid * 16) =
          __ldcg(reinterpret_cast<const uint4 *>(qg) + tid);
  }

  int L = __ldg(a.context_lens + b);
  const int cap = (int)min((int64_t)a.max_blocks * a.block_size, (int64_t)a.max_context_len);
  if (L < 0 || L > cap) {
    if (tid == 0 && part == 0) raise_error(PKV_DEVERR_CONTEXT_LEN);
    L = L < 0 ? 0 : cap;
  }
  const int t_begin = part * a.partition_tokens;
  const bool cluster = a.fused == 2;  // uniform over the grid
  if (t_begin >= L && !cluster) {  // empty range: nothing written (the merge skips it)
    if (a.fused && part == 0) {  // empty context: zero output
      uint16_t *o = a.out + ((int64_t)b * a.num_q_heads + g * a.group) * D;
      for (int i = tid; i < a.group * D; i += kThreads) o[i] = 0;
    }
    return;
  }
  // In a cluster every CTA takes part in the merge, so an empty range streams nothing
  // and publishes lse = -inf.
  const int t_end = min(t_begin + a.partition_tokens, L);
  const int n_chunks = t_end > t_begin ? (t_end - t_begin + kChunk - 1) / kChunk : 0;

  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      dev::mbar_init(bar_full + 8 * s, 1);
      dev::mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    if (cluster) {  // armed for the bytes the cluster pushes here: see the merge below
      const int n = (int)dev::cluster_nctarank(), rank = (int)dev::cluster_ctarank();
      const int owned = rank < a.group ? (a.group - rank + n - 1) / n : 0;
      dev::mbar_init(bar_merge, 1);
      dev::mbar_arrive_expect_tx(bar_merge, (uint32_t)(n * owned * (D + 1) * 4));
    }
    *s_flag = 0;
    *s_last = 0;
    dev::fence_mbar_init();
  }
  __syncthreads();
  // Every thread arrives on the cluster barrier now and waits on it before its first
  // access to another CTA's shared memory: by then every merge barrier is initialised.
  // (Its next phase is the closing handshake at the end of the kernel.)
  if (cluster) dev::cluster_arrive_relaxed();

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------- producer warp
    const uint64_t policy = dev::policy_evict_first();
    const int rb = a.box_rows;                       // keys per TMA box = min(BS, 64)
    const uint32_t box_bytes = (uint32_t)rb * 128u;  // per 64-dim half
    const int lb_last = (t_end - 1) >> a.log2_bs;
    int win = win0;                                  // lanes hold table entries [win, win + 32)
    int tb = tb0;
    // Launched as a programmatic dependent of the slot-write kernel, everything above
    // overlapped it; the cache is read only after that grid's writes are visible.
    // (Without a programmatic launch this returns at once.)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % STAGES;
      if (c >= STAGES &&
          !__all_sync(0xffffffffu, dev::mbar_wait(bar_empty + 8 * s, ((c / STAGES) - 1) & 1))) {
        if (lane == 0) {
          raise_error(PKV_DEVERR_TIMEOUT);
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
          raise_error(PKV_DEVERR_BLOCK_ID);
          phys = 0;
        }
        const int off = key & (a.block_size - 1);
        const int32_t row = (int32_t)((phys * a.num_kv_heads + g) * a.block_size + off);
        const uint32_t dk = base + s * kStageBytes + lane * box_bytes;
        issue_box<D>(dk, dk + kTileBytes, &tmk, &tmv, row, bar_full + 8 * s, policy);
      }
      __syncwarp();
    }
    if (cluster) dev::cluster_wait();
  } else {
    // ----------------------------------------------------------- consumer warps
    WarpAcc<D> acc;    // tensor form
    WarpAccF<D> accf;  // CUDA-core form
    if constexpr (kFma) {
      accf_reset(accf);
    } else {
      acc_reset(acc);
      const uint32_t *qs = reinterpret_cast<const uint32_t *>(base_ptr + (q_area - base));
      const int gid = lane >> 2, tig = lane & 3;
      const bool hv = gid < a.group;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[ks][0] = hv ? qs[gid * (D / 2) + 8 * ks + tig] : 0u;
        qb[ks][1] = hv ? qs[gid * (D / 2) + 8 * ks + 4 + tig] : 0u;
      }
    }
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % STAGES;
      if (!__all_sync(0xffffffffu, dev::mbar_wait(bar_full + 8 * s, (c / STAGES) & 1))) {
        if (lane == 0) {
          raise_error(PKV_DEVERR_TIMEOUT);
          *s_flag = 1;
        }
        break;
      }
      const int key0 = t_begin + c * kChunk + 16 * warp;
      const int nvalid = min(16, t_end - key0);
      if (nvalid > 0) {
        const uint32_t kb = base + s * kStageBytes;
        if constexpr (kFma)
          warp_tile_fma<D>(accf, q_area, a.group, kb, kb + kTileBytes, warp, lane, nvalid,
                           a.scale_log2);
        else
          warp_tile<D>(acc, qb, kb, kb + kTileBytes, warp, lane, nvalid, a.scale_log2);
      }
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(bar_empty + 8 * s);
    }
    // ---- merge the four warps through shared memory (the stages are free now)
    consumer_bar();
    MergeArea r;
    r.o = reinterpret_cast<float *>(base_ptr);
    r.m = r.o + kConsumerWarps * a.group * D;
    r.l = r.m + kConsumerWarps * kMaxGroup;
    if constexpr (kFma)
      warp_stash_fma<D>(accf, r, a.group, warp, lane);
    else
      warp_stash<D>(acc, r, a.group, warp, lane);
    consumer_bar();
    const int nparts_b = (L + a.partition_tokens - 1) / a.partition_tokens;  // non-empty ones
    if (cluster) {
      // Cluster merge.  CTA rank h % n merges head h.  Every CTA pushes its (normalised
      // o, base-2 lse) of each head into the owner's receive area with asynchronous
      // stores that count their bytes off the owner's merge barrier, which its one
      // arrival at set-up armed for all n * (heads owned) * (D + 1) * 4 bytes.  The
      // phase completes when the last byte has landed: the owner then merges from its
      // own shared memory, which nobody touches again, so no CTA waits for its peers
      // to finish reading.  Every wait on the way to the pushes is bounded, so they all
      // come; if the merge barrier still times out, the CTA records the error, skips the
      // merge and, before it exits, waits until no peer can still be storing into it
      // (the closing handshake at the end of the kernel).
      dev::cluster_wait();
      const int n = (int)dev::cluster_nctarank();
      const int rank = (int)dev::cluster_ctarank();
      if (n == a.n_parts && n <= kMaxClusterParts) {
        const int hpo = (a.group + n - 1) / n;  // heads each CTA merges, at most
        for (int i = tid; i < a.group * D / 2; i += kConsumers) {  // two dims per store
          const int h = i / (D / 2), d = 2 * (i - h * (D / 2));
          float M2, den, M2b, denb;
          const float v0 = cta_merge<D>(r, a.group, h, d, &M2, &den);
          const float v1 = cta_merge<D>(r, a.group, h, d + 1, &M2b, &denb);
          const bool live = den > 0.f;  // false (or NaN) when this range had no keys
          const int slot = rank * hpo + h / n;
          const uint32_t dst = dev::mapa(recv, (uint32_t)(h % n));
          const uint32_t dbar = dev::mapa(bar_merge, (uint32_t)(h % n));
          dev::st_async_v2(dst + (uint32_t)(slot * D + d) * 4u, live ? v0 : 0.f, live ? v1 : 0.f,
                           dbar);
          if (d == 0)
            dev::st_async(dst + (uint32_t)(kRecvSlots * D + slot) * 4u,
                          live ? M2 + log2f(den) : -INFINITY, dbar);
        }
        if (__all_sync(0xffffffffu, dev::mbar_wait_cluster(bar_merge, 0))) {
          const int64_t head0 = (int64_t)b * a.num_q_heads + g * a.group;
          for (int j = warp; j < hpo; j += kConsumerWarps) {
            const int h = rank + n * j;
            if (h < a.group)
              recv_merge_head<D>(a.out + (head0 + h) * D, recv_o, recv_l, j, hpo, n, lane);
          }
        } else if (lane == 0) {
          raise_error(PKV_DEVERR_TIMEOUT);
          *s_merge_timeout = 1;
        }
      } else if (tid == 0 && rank == 0) {
        raise_error(PKV_DEVERR_TIMEOUT);  // launched with the wrong cluster shape
      }
    } else {
      finish_partition<D>(a, r, b, g, part, nparts_b, tid, warp, lane, s_flag, s_last);
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
  // ---- closing handshake of the cluster merge.  Every thread of every CTA arrives
  // here, after all of its pushes were issued, and normally leaves at once: a CTA
  // whose merge barrier completed has received every byte aimed at it, so no store
  // can still be on its way in.  A CTA whose merge wait gave up instead waits for the
  // whole cluster to arrive -- every peer thread gets here through bounded waits only,
  // so this wait ends -- and then once more (bounded) on its merge barrier, whose
  // phase completes when the last of those already-issued stores has landed.  Only
  // then does it exit, so no peer's store can target a CTA that has left.
  if (cluster) {
    dev::cluster_arrive_relaxed();
    if (*s_merge_timeout) {
      dev::cluster_wait();
      if (tid == 0) (void)dev::mbar_wait_cluster(bar_merge, 0);
    }
  }
}


// ===========================================================================
// decode_persistent_kernel: the fused decode for many (sequence, kv head) units.
//
// A grid of about one wave of CTAs (warp roles, TMA ring, per-stage work and epilogue
// as in decode_kernel) takes work items -- one non-empty partition of P tokens of one
// (sequence, kv head) -- and streams them back to back through its ring.  The producer
// runs ahead across item boundaries: the next item's table window, query rows and
// first boxes are in flight while the consumers finish the current item, so a CTA pays
// its launch, set-up and first-copy latency once, not once per partition.
//
// Order: longest first.  All full partitions come first (by partition index,
// descending), then every sequence's last partition by its size, descending; within a
// category, by sequence, then kv head.  A single-partition sequence's size is its number
// q of 64-key chunks.  A multi-partition sequence is merged by whichever of its
// partitions finishes last: a store, a ticket and loads of the partials, about as much
// latency as streaming two chunks, and pure delay near the end, where no other CTA's
// streaming overlaps it.  So when the single-partition items alone fill one wave of CTAs
// (T > 0, T the smallest chunk count at which they do), every multi-partition last
// partition gets the largest size, Q + kMergeChunks: they follow the full partitions,
// all merges happen while most of the work is still ahead, and the order ends with
// single-partition items alone.  When they do not (T = 0; few, long sequences), moving
// the merges up would put long single-partition items last instead, so a multi-partition
// last partition only counts its merge: size q + kMergeChunks.  (Measured on batches of
// 64 to 512 sequences: each rule is the faster one where it is used.)  Each CTA derives the same
// order from the context lengths (histograms in shared memory, on its consumer warps).
// So that no CTA's first copy waits for that, CTA c < Ex * Hkv (Ex = gridDim.x / Hkv)
// first streams a provisional item, partition 0 of unit c, which the order leaves out;
// after it, and for the other CTAs from the start, items come from a global counter,
// each claimed when the current item is two chunks from its last issue -- so the
// largest items left go to the CTAs about to run dry (list scheduling).  No CTA waits
// for another; the last CTA to stop claiming resets the counter for the next call.

constexpr int kMaxPersistSeqs = 1024;  // sequences per batch (a warp scans 32 x 32 of them)
constexpr int kMaxCategories = 64;     // full-partition levels + last-partition sizes
constexpr int kMergeChunks = 2;        // what a merge adds to a last partition's size

// What the producer tells the consumers about the chunk in a stage.
struct ItemDesc {
  int32_t b, g;               // sequence, kv head
  int32_t t_begin, t_end;     // the item's token range
  int32_t key0;               // first key of this chunk
  int32_t flags;              // kFirst | kLast | kStop
  int32_t np;                 // partitions of the sequence
  int32_t pad;
};
constexpr int32_t kFirst = 1, kLast = 2, kStop = 4;

// Shared-memory layout after the 1024-byte aligned base.
template <int D, int STAGES>
struct PersistSmem {
  static constexpr uint32_t kStageBytes = 2 * kChunk * D * 2;
  static constexpr uint32_t kQSlot = kMaxGroup * D * 2;
  static constexpr uint32_t q = STAGES * kStageBytes;
  static constexpr uint32_t desc = q + STAGES * kQSlot;
  static constexpr uint32_t bars = desc + STAGES * sizeof(ItemDesc);  // full[STAGES], empty[STAGES]
  static constexpr uint32_t flags = bars + STAGES * 16;               // flag, last, issued, T
  static constexpr uint32_t ord = flags + 16;                         // order-ready barrier, ex0
  static constexpr uint32_t hist_nf = ord + 16;                       // full partitions by nf
  static constexpr uint32_t hist_lc = hist_nf + kMaxCategories * 4;   // single partitions by q
  static constexpr uint32_t hist_ml = hist_lc + kMaxCategories * 4;   // multi-partition last, by q
  static constexpr uint32_t off = hist_ml + kMaxCategories * 4;       // [kMaxCategories + 1]
  static constexpr uint32_t lt = off + (kMaxCategories + 4) * 4;      // u16 [kMaxPersistSeqs]
  static constexpr uint32_t nf = lt + kMaxPersistSeqs * 2;            // u8 [kMaxPersistSeqs]
  static constexpr uint32_t total = nf + kMaxPersistSeqs;
};
static_assert(PersistSmem<64, 4>::lt % 16 == 0 && PersistSmem<128, 3>::lt % 16 == 0 &&
                  PersistSmem<64, 4>::nf % 16 == 0 && PersistSmem<128, 3>::nf % 16 == 0,
              "per-sequence arrays are read as 16-byte vectors");

struct Item {
  int b, g, t_begin, t_end, np;
};

// Item k of the order above (false when k >= the number of items).  All 32 lanes of the
// producer warp take part; the result is the same on every lane.
//   s_off: exclusive prefix of the categories' item counts, s_off[ncat] = total;
//   category c < R-1: full partition r = R-2-c of sequences with nf > r;
//   category c >= R-1: last partition of sequences whose size (q = ceil(lt / 64) if
//                      nf = 0, else Q + kMergeChunks if T > 0, else q + kMergeChunks)
//                      is Q + kMergeChunks - (c - (R-1)).
__device__ __forceinline__ bool find_item(int k, const int *s_off, int ncat, int R, int P, int Hkv,
                                          int T, int num_seqs, int Ex, const uint16_t *s_lt,
                                          const uint8_t *s_nf, int lane, Item &it) {
  if (k >= s_off[ncat]) return false;
  // category: the last c with s_off[c] <= k (s_off is nondecreasing; that one is non-empty)
  const unsigned m0 = __ballot_sync(0xffffffffu, lane < ncat && s_off[lane] <= k);
  const unsigned m1 = __ballot_sync(0xffffffffu, lane + 32 < ncat && s_off[lane + 32] <= k);
  const int cat = __popc(m0) + __popc(m1) - 1;
  const int j = k - s_off[cat];
  const int m = j / Hkv;
  it.g = j - m * Hkv;
  const bool full = cat < R - 1;
  const int r = R - 2 - cat;                                   // full: partition index
  const int q = (P / kChunk) + kMergeChunks - (cat - (R - 1));  // last partition: its size
  // select the m-th sequence (ascending) of the category; lane w holds sequences [32w, 32w+32).
  // Partition 0 of sequences b < Ex is not in the order (those are the provisional first
  // items): excluded from the full level r = 0 and, for single-partition sequences, from
  // the last-partition categories.
  const int rem = Ex - 32 * lane;
  const unsigned exmask = rem >= 32 ? 0xffffffffu : (rem > 0 ? (1u << rem) - 1u : 0u);
  unsigned bits = 0;
  if (32 * lane >= num_seqs) {
    // no sequences in this lane's word (the arrays are written up to num_seqs rounded to 32)
  } else {
    const uint4 *vn = reinterpret_cast<const uint4 *>(s_nf + 32 * lane);
    const uint4 n0 = vn[0], n1 = vn[1];
    const uint32_t wn[8] = {n0.x, n0.y, n0.z, n0.w, n1.x, n1.y, n1.z, n1.w};
    if (full) {
#pragma unroll
      for (int t = 0; t < 32; ++t) bits |= (int)((wn[t >> 2] >> (8 * (t & 3))) & 0xffu) > r ? 1u << t : 0u;
      if (r == 0) bits &= ~exmask;
    } else {
      const uint4 *v = reinterpret_cast<const uint4 *>(s_lt + 32 * lane);
      uint32_t wd[16];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const uint4 x = v[u];
        wd[4 * u] = x.x;
        wd[4 * u + 1] = x.y;
        wd[4 * u + 2] = x.z;
        wd[4 * u + 3] = x.w;
      }
#pragma unroll
      for (int t = 0; t < 32; ++t) {
        const int lt = (int)((wd[t >> 1] >> (16 * (t & 1))) & 0xffffu);
        const int nf = (int)((wn[t >> 2] >> (8 * (t & 3))) & 0xffu);
        const int qt = (lt + kChunk - 1) / kChunk;
        const int size = nf == 0 ? qt : (T > 0 ? P / kChunk : qt) + kMergeChunks;
        const bool excluded = nf == 0 && ((exmask >> t) & 1u);
        bits |= (lt > 0 && size == q && !excluded) ? 1u << t : 0u;
      }
    }
  }
  const int pc = __popc(bits);
  int incl = pc;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  const unsigned sel = __ballot_sync(0xffffffffu, incl > m);
  if (sel == 0u) {  // cannot happen (the counts come from the same arrays): stop cleanly
    if (lane == 0) raise_error(PKV_DEVERR_CONTEXT_LEN);
    return false;
  }
  const int w = __ffs(sel) - 1;
  const int before = __shfl_sync(0xffffffffu, incl - pc, w);
  unsigned wb = __shfl_sync(0xffffffffu, bits, w);
  for (int i = 0; i < m - before; ++i) wb &= wb - 1;
  it.b = 32 * w + __ffs(wb) - 1;
  const int nf = s_nf[it.b], lt = s_lt[it.b];
  it.np = nf + (lt > 0 ? 1 : 0);
  if (full) {
    it.t_begin = r * P;
    it.t_end = it.t_begin + P;
  } else {
    it.t_begin = nf * P;
    it.t_end = it.t_begin + lt;
  }
  return true;
}

template <int D, int STAGES>
__global__ void __launch_bounds__(kThreads, split_occupancy(D))
    decode_persistent_kernel(const __grid_constant__ CUtensorMap tmk,
                             const __grid_constant__ CUtensorMap tmv, const DecodeArgs a) {
  using SL = PersistSmem<D, STAGES>;
  constexpr int kTileBytes = kChunk * D * 2;
  constexpr int KS = D / 16;

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t bar_full = base + SL::bars;
  const uint32_t bar_empty = bar_full + STAGES * 8;
  volatile int *const s_flag = reinterpret_cast<volatile int *>(base_ptr + SL::flags);
  volatile int *const s_last = s_flag + 1;
  volatile int *const s_issued = s_flag + 2;
  volatile int *const s_T = s_flag + 3;
  ItemDesc *const s_desc = reinterpret_cast<ItemDesc *>(base_ptr + SL::desc);
  int *const s_hist_nf = reinterpret_cast<int *>(base_ptr + SL::hist_nf);
  int *const s_hist_lc = reinterpret_cast<int *>(base_ptr + SL::hist_lc);
  int *const s_hist_ml = reinterpret_cast<int *>(base_ptr + SL::hist_ml);
  int *const s_off = reinterpret_cast<int *>(base_ptr + SL::off);
  uint16_t *const s_lt = reinterpret_cast<uint16_t *>(base_ptr + SL::lt);
  uint8_t *const s_nf = base_ptr + SL::nf;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int P = a.partition_tokens, R = a.n_parts, Q = P / kChunk;
  const int ncat = R - 1 + Q + kMergeChunks;
  const int Hkv = a.num_kv_heads;
  const int cap = (int)min((int64_t)a.max_blocks * a.block_size, (int64_t)a.max_context_len);
  const int bpad = (a.num_seqs + 31) & ~31;
  // Provisional first items: CTA c < Ex * Hkv starts at once on partition 0 of unit c
  // (sequence c / Hkv, kv head c % Hkv) instead of waiting for the order, whose set-up
  // (every context length, histograms, the category scan) then runs on the consumer
  // warps while the first stages are in flight.  The order holds every other item.
  const int Ex = (int)gridDim.x / Hkv;  // sequences whose partition 0 is taken this way
  const uint32_t bar_order = base + SL::ord;  // phase 0: the order's tables are written
  volatile int *const s_ex0 = reinterpret_cast<volatile int *>(base_ptr + SL::ord + 8);

  // ---- set-up: barriers; the consumer warps load every context length at once
  constexpr int kLensPerThread = (kMaxPersistSeqs + kConsumers - 1) / kConsumers;
  int lens[kLensPerThread];
  if (warp < kConsumerWarps) {
#pragma unroll
    for (int k = 0; k < kLensPerThread; ++k) {
      const int bb = tid + k * kConsumers;
      lens[k] = bb < a.num_seqs ? __ldg(a.context_lens + bb) : 0;
    }
  }
  if (tid == 0) {
#pragma unroll
    for (int s = 0; s < STAGES; ++s) {
      dev::mbar_init(bar_full + 8 * s, 1);
      dev::mbar_init(bar_empty + 8 * s, kConsumerWarps);
    }
    dev::mbar_init(bar_order, 32);  // every lane of warp 0, after the scan
    *s_flag = 0;
    *s_issued = 0;
    *s_ex0 = 0;
    dev::fence_mbar_init();
  }
  for (int i = tid; i < 3 * kMaxCategories; i += kThreads) s_hist_nf[i] = 0;  // all three
  __syncthreads();

  if (warp < kConsumerWarps) {
    // ---- the order's histograms (consumer warps), then its category scan (warp 0)
#pragma unroll
    for (int k = 0; k < kLensPerThread; ++k) {
      const int bb = tid + k * kConsumers;
      if (bb >= bpad) break;
      int nf = 0, lt = 0;
      if (bb < a.num_seqs) {
        int L = lens[k];
        if (L < 0 || L > cap) {
          if (blockIdx.x == 0) raise_error(PKV_DEVERR_CONTEXT_LEN);
          L = L < 0 ? 0 : cap;
        }
        if (L > 0) {
          nf = (L - 1) / P;
          lt = L - nf * P;
          const int q = (lt + kChunk - 1) / kChunk;
          if (nf > 0) {
            atomicAdd(s_hist_nf + nf, 1);
            atomicAdd(s_hist_ml + q, 1);
            if (bb < Ex) atomicAdd(const_cast<int *>(s_ex0), 1);  // its partition 0 is provisional
          } else if (bb >= Ex) {
            atomicAdd(s_hist_lc + q, 1);
          }
        } else if (bb % (int)gridDim.x == (int)blockIdx.x) {  // empty context: zero output
          uint2 *o = reinterpret_cast<uint2 *>(a.out + (int64_t)bb * a.num_q_heads * D);
          for (int i = 0; i < a.num_q_heads * D / 4; ++i) o[i] = make_uint2(0u, 0u);
        }
      }
      s_nf[bb] = (uint8_t)nf;
      s_lt[bb] = (uint16_t)lt;
    }
    consumer_bar();
  }
  if (warp == 0) {  // T, the item counts of the categories, then their exclusive prefix
    int T = 0;
    {  // single-partition items of at most q chunks, q = lane + 1 and lane + 33
      int i0 = lane + 1 <= Q ? s_hist_lc[lane + 1] * Hkv : 0;
      int i1 = lane + 33 <= Q ? s_hist_lc[lane + 33] * Hkv : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y0 = __shfl_up_sync(0xffffffffu, i0, o), y1 = __shfl_up_sync(0xffffffffu, i1, o);
        if (lane >= o) {
          i0 += y0;
          i1 += y1;
        }
      }
      i1 += __shfl_sync(0xffffffffu, i0, 31);
      const unsigned b0 = __ballot_sync(0xffffffffu, lane + 1 <= Q && i0 >= (int)gridDim.x);
      const unsigned b1 = __ballot_sync(0xffffffffu, lane + 33 <= Q && i1 >= (int)gridDim.x);
      T = b0 ? __ffs(b0) : (b1 ? 32 + __ffs(b1) : 0);
    }
    int cnt[2];
#pragma unroll
    for (int hh = 0; hh < 2; ++hh) {
      const int c = lane + 32 * hh;
      int n = 0;
      if (c < R - 1) {  // full partition r = R-2-c: sequences with nf > r
        for (int x = R - 1 - c; x <= R - 1; ++x) n += s_hist_nf[x];
        if (c == R - 2) n -= *s_ex0;  // r = 0 of sequences b < Ex: provisional
      } else if (c < ncat) {  // last partitions of size sz
        const int sz = Q + kMergeChunks - (c - (R - 1));
        if (sz <= Q) n = s_hist_lc[sz];
        if (T > 0) {  // every multi-partition last partition in the largest size
          if (sz == Q + kMergeChunks)
            for (int qm = 1; qm <= Q; ++qm) n += s_hist_ml[qm];
        } else if (sz - kMergeChunks >= 1) {
          n += s_hist_ml[sz - kMergeChunks];
        }
      }
      cnt[hh] = n * Hkv;
    }
    int i0 = cnt[0], i1 = cnt[1];
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y0 = __shfl_up_sync(0xffffffffu, i0, o), y1 = __shfl_up_sync(0xffffffffu, i1, o);
      if (lane >= o) {
        i0 += y0;
        i1 += y1;
      }
    }
    const int t0 = __shfl_sync(0xffffffffu, i0, 31);
    const int total = t0 + __shfl_sync(0xffffffffu, i1, 31);
    if (lane < ncat) s_off[lane] = i0 - cnt[0];
    if (lane + 32 < ncat) s_off[lane + 32] = t0 + i1 - cnt[1];
    if (lane == 0) {
      s_off[ncat] = total;
      *s_T = T;
    }
    dev::mbar_arrive(bar_order);  // releases this lane's writes; phase 0 after all 32
  }

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------- producer warp
    const uint64_t policy = dev::policy_evict_first();
    const int rb = a.box_rows;
    const uint32_t box_bytes = (uint32_t)rb * 128u;
    const uint32_t q_bytes = (uint32_t)a.group * D * 2u;
    // The provisional first item (partition 0 of unit blockIdx.x, for CTAs below Ex * Hkv
    // whose sequence is not empty), and the first 32 entries of its table row; neither
    // needs the order.
    Item it;
    bool have = false, pre = false;
    int tb_pre = 0;
    if ((int)blockIdx.x < Ex * Hkv) {
      const int b0 = (int)blockIdx.x / Hkv;
      int L0 = __ldg(a.context_lens + b0);
      tb_pre = lane < a.max_blocks ? __ldg(a.block_tables + (int64_t)b0 * a.max_blocks + lane) : 0;
      if (L0 > cap) L0 = cap;  // out-of-range lengths are flagged by the histogram pass
      if (L0 > 0) {
        const int nf0 = (L0 - 1) / P;
        it.b = b0;
        it.g = (int)blockIdx.x - b0 * Hkv;
        it.t_begin = 0;
        it.t_end = nf0 > 0 ? P : L0;
        it.np = nf0 + 1;
        have = pre = true;
      }
    }
    asm volatile("griddepcontrol.wait;" ::: "memory");  // see decode_kernel
    int c = 0;  // chunks issued, over all items
    bool ok = true;
    int T = 0;
    bool order = false;  // the order's tables are visible to this warp
    auto wait_order = [&]() -> bool {
      if (order) return true;
      if (!__all_sync(0xffffffffu, dev::mbar_wait(bar_order, 0))) {
        if (lane == 0) {
          raise_error(PKV_DEVERR_TIMEOUT);
          *s_flag = 1;
        }
        return false;
      }
      T = *s_T;
      order = true;
      return true;
    };
    if (!have) {  // no provisional item: the first claim
      if (wait_order()) {
        int k0 = 0;
        if (lane == 0) k0 = (int)atomicAdd(a.sched, 1u);
        k0 = __shfl_sync(0xffffffffu, k0, 0);
        have = find_item(k0, s_off, ncat, R, P, Hkv, T, a.num_seqs, Ex, s_lt, s_nf, lane, it);
      } else {
        ok = false;
      }
    }
    while (have && ok) {
      int k_next = 0;  // lane 0: the item after this one
      const int32_t *trow = a.block_tables + (int64_t)it.b * a.max_blocks;
      const int lb_last = (it.t_end - 1) >> a.log2_bs;
      int win = it.t_begin >> a.log2_bs;
      int tb = pre ? tb_pre : ((win + lane <= lb_last) ? __ldg(trow + win + lane) : 0);
      pre = false;
      const int n_chunks = (it.t_end - it.t_begin + kChunk - 1) / kChunk;
      for (int i = 0; i < n_chunks; ++i, ++c) {
        const int s = c % STAGES;
        if (c >= STAGES &&
            !__all_sync(0xffffffffu, dev::mbar_wait(bar_empty + 8 * s, ((c / STAGES) - 1) & 1))) {
          if (lane == 0) {
            raise_error(PKV_DEVERR_TIMEOUT);
            *s_flag = 1;
          }
          ok = false;
          break;
        }
        // The next item is claimed two chunks before this one's last issue, when this
        // CTA is about to run out of work: CTAs that finish early take the larger items
        // still left (the order is longest first), and the claim's latency hides behind
        // the stages already queued.
        if (lane == 0 && i == max(n_chunks - 2, 0)) k_next = (int)atomicAdd(a.sched, 1u);
        const int k0 = it.t_begin + i * kChunk;
        const int nk = min(kChunk, it.t_end - k0);
        const int nbox = (nk + rb - 1) / rb;
        const int lb_hi = (k0 + (nbox - 1) * rb) >> a.log2_bs;
        if (lb_hi >= win + 32) {  // slide the table window
          win = k0 >> a.log2_bs;
          tb = (win + lane <= lb_last) ? __ldg(trow + win + lane) : 0;
        }
        const int key = k0 + lane * rb;
        const int src = min(max((key >> a.log2_bs) - win, 0), 31);
        const int64_t phys_raw = __shfl_sync(0xffffffffu, tb, src);
        if (lane == 0) {
          ItemDesc dsc;
          dsc.b = it.b;
          dsc.g = it.g;
          dsc.t_begin = it.t_begin;
          dsc.t_end = it.t_end;
          dsc.key0 = k0;
          dsc.flags = (i == 0 ? kFirst : 0) | (i == n_chunks - 1 ? kLast : 0);
          dsc.np = it.np;
          dsc.pad = 0;
          s_desc[s] = dsc;
          dev::mbar_arrive_expect_tx(bar_full + 8 * s,
                                     2u * nbox * box_bytes * (D / 64) + (i == 0 ? q_bytes : 0u));
          if (i == 0)  // the group's query rows, contiguous in q
            dev::bulk_load(base + SL::q + s * SL::kQSlot,
                           a.q + ((int64_t)it.b * a.num_q_heads + it.g * a.group) * D, q_bytes,
                           bar_full + 8 * s);
        }
        __syncwarp();
        if (lane < nbox) {
          int64_t phys = phys_raw;
          if (phys < 0 || phys >= a.num_blocks) {
            raise_error(PKV_DEVERR_BLOCK_ID);
            phys = 0;
          }
          const int off = key & (a.block_size - 1);
          const int32_t row = (int32_t)((phys * a.num_kv_heads + it.g) * a.block_size + off);
          const uint32_t dk = base + s * SL::kStageBytes + lane * box_bytes;
          issue_box<D>(dk, dk + kTileBytes, &tmk, &tmv, row, bar_full + 8 * s, policy);
        }
        __syncwarp();
      }
      if (!ok) break;
      const int k = __shfl_sync(0xffffffffu, k_next, 0);
      if (!wait_order()) {
        ok = false;
        break;
      }
      have = find_item(k, s_off, ncat, R, P, Hkv, T, a.num_seqs, Ex, s_lt, s_nf, lane, it);
    }
    // This CTA has made its last claim (or given up): count it done.  The CTA that
    // completes the count has seen every CTA of this call stop claiming, so it resets
    // both words for the next call; the atomic's round trip overlaps the last stages.
    unsigned done_before = 0u;
    if (lane == 0) done_before = atomicAdd(a.sched + 1, 1u);
    if (ok) {  // no item follows: a stop marker in the next stage
      const int s = c % STAGES;
      if (c >= STAGES &&
          !__all_sync(0xffffffffu, dev::mbar_wait(bar_empty + 8 * s, ((c / STAGES) - 1) & 1))) {
        if (lane == 0) {
          raise_error(PKV_DEVERR_TIMEOUT);
          *s_flag = 1;
        }
      } else if (lane == 0) {
        s_desc[s].flags = kStop;
        dev::mbar_arrive(bar_full + 8 * s);
      }
    }
    if (lane == 0) *s_issued = c;
    if (lane == 0 && done_before == gridDim.x - 1) {
      a.sched[0] = 0u;
      a.sched[1] = 0u;
    }
  } else {
    // ----------------------------------------------------------- consumer warps
    WarpAcc<D> acc;
    acc_reset(acc);
    uint32_t qb[KS][2];
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) qb[ks][0] = qb[ks][1] = 0u;
    const int gid = lane >> 2, tig = lane & 3;
    for (int c = 0;; ++c) {
      const int s = c % STAGES;
      if (!__all_sync(0xffffffffu, dev::mbar_wait(bar_full + 8 * s, (c / STAGES) & 1))) {
        if (lane == 0) {
          raise_error(PKV_DEVERR_TIMEOUT);
          *s_flag = 1;
        }
        break;
      }
      const ItemDesc d = s_desc[s];
      if (d.flags & kStop) break;
      if (d.flags & kFirst) {  // a new item: its query rows and a fresh softmax state
        const uint32_t *qs = reinterpret_cast<const uint32_t *>(base_ptr + SL::q + s * SL::kQSlot);
        const bool hv = gid < a.group;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qb[ks][0] = hv ? qs[gid * (D / 2) + 8 * ks + tig] : 0u;
          qb[ks][1] = hv ? qs[gid * (D / 2) + 8 * ks + 4 + tig] : 0u;
        }
        acc_reset(acc);
      }
      const int key0 = d.key0 + 16 * warp;
      const int nvalid = min(16, d.t_end - key0);
      const uint32_t kb = base + s * SL::kStageBytes;
      if (nvalid > 0) warp_tile<D>(acc, qb, kb, kb + kTileBytes, warp, lane, nvalid, a.scale_log2);
      if (d.flags & kLast) {
        consumer_bar();  // every warp is done with this stage's tiles: reuse it to merge
        MergeArea r;
        r.o = reinterpret_cast<float *>(base_ptr + s * SL::kStageBytes);
        r.m = r.o + kConsumerWarps * a.group * D;
        r.l = r.m + kConsumerWarps * kMaxGroup;
        warp_stash<D>(acc, r, a.group, warp, lane);
        consumer_bar();
        finish_partition<D>(a, r, d.b, d.g, d.t_begin / P, d.np, tid, warp, lane, s_flag, s_last);
      }
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(bar_empty + 8 * s);
    }
  }

  // ---- a timed-out wait leaves copies possibly in flight: wait for them (bounded)
  __syncthreads();
  if (tid == 0 && *s_flag) {
    const int issued = *s_issued;
    for (int s = 0; s < STAGES; ++s) {
      const int c_last = s + ((issued - 1 - s) / STAGES) * STAGES;  // last chunk on stage s
      if (c_last >= 0 && c_last < issued) (void)dev::mbar_wait(bar_full + 8 * s, (c_last / STAGES) & 1);
    }
  }
}

// ---------------------------------------------------------------------------
// Log-sum-exp merge of fixed partitions: one CTA per (sequence, query head).  Thread
// groups of D/4 threads each read one partition row with float4 loads; groups take
// partitions round robin and are summed through shared memory.
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
    if (tid == 0) raise_error(PKV_DEVERR_CONTEXT_LEN);
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

cudaError_t read_decode_errors(uint32_t *flags, int clear) { return read_tu_errors(flags, clear); }

namespace {

bool g_split_attr[kMaxDevices][2][2];  // dynamic smem attribute of decode_kernel set [D][form]
bool g_persist_attr[kMaxDevices][2];  // ... of decode_persistent_kernel
// Arithmetic of decode_kernel's consumer warps (PKV_CONSUMER_*), process-wide.
std::atomic<int> g_consumer{PKV_CONSUMER_TENSOR};

// Partition size for paged_decode_attention.  Few (sequence, kv head) units: cut each
// into as many partitions as make about one wave of CTAs, so every CTA streams a long
// range.  Many units: 1536-token work items of the persistent kernel (batches of at
// most kMaxPersistSeqs sequences), 1024-token CTAs of decode_kernel beyond that.
// Never below min(context, 512) tokens, so short contexts are not cut into tiny pieces.
int32_t plan_partition(int32_t num_seqs, int32_t hkv, int32_t d, int32_t max_len, int sms) {
  const int64_t units = (int64_t)num_seqs * hkv;
  const int64_t slots = (int64_t)sms * split_occupancy(d);
  const int64_t lr = ((int64_t)max_len + kChunk - 1) / kChunk * kChunk;
  int64_t P;
  if (units >= slots) {
    const int64_t pm = num_seqs <= kMaxPersistSeqs ? 1536 : 1024;
    P = lr < pm ? lr : pm;
  } else {
    const int64_t parts = slots / units;
    P = ((max_len + parts - 1) / parts + kChunk - 1) / kChunk * kChunk;
  }
  const int64_t floor_p = lr < 512 ? lr : 512;
  if (P < floor_p) P = floor_p;
  if (P < kChunk) P = kChunk;
  return (int32_t)P;
}
// Cluster size of the fused decode: when every partition of the grid is resident at
// once (few (sequence, kv head) units) and a unit has 2..8 partitions, the partitions
// of a unit form one cluster and merge through distributed shared memory; otherwise 0
// (the last partition to finish merges through global memory).
int cluster_parts(int32_t num_seqs, int32_t hkv, int32_t d, int32_t max_len, int32_t P, int sms) {
  const int64_t units = (int64_t)num_seqs * hkv;
  const int64_t n_parts = ((int64_t)max_len + P - 1) / P;
  const int64_t slots = (int64_t)sms * split_occupancy(d);
  if (n_parts < 2 || n_parts > kMaxClusterParts || units * n_parts > slots) return 0;
  return (int)n_parts;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

// Workspace of paged_decode_attention: merge counters [B*Hkv] u32 and the persistent
// kernel's two scheduling words, then paged_decode_split's partials for the planned
// partition size.
struct FusedLayout {
  size_t counters, sched, o_part, lse_part, total;
};

FusedLayout fused_layout(int32_t num_seqs, int32_t hq, int32_t hkv, int32_t d, int32_t mlen,
                         int32_t P) {
  FusedLayout f;
  const size_t rows = (size_t)num_seqs * hq * (size_t)((mlen + P - 1) / P);
  f.counters = 0;
  f.sched = (size_t)num_seqs * hkv * 4;
  f.o_part = align256(f.sched + 8);
  f.lse_part = f.o_part + align256(rows * d * sizeof(float));
  f.total = f.lse_part + align256(rows * sizeof(float));
  return f;
}
template <int D>
int launch_split(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                 const int32_t *bt, int32_t max_blocks, const int32_t *lens, int32_t max_len,
                 int32_t num_seqs, int32_t hq, const pkv_cache_desc &c, float scale, int32_t P,
                 float *o_part, float *lse_part, pkv_bf16 *out, uint32_t *counters,
                 cudaStream_t stream, bool programmatic = false, int cluster = 0,
                 bool q_wait = false) {
  CUtensorMap tmk, tmv;
  const bool fma = g_consumer.load(std::memory_order_relaxed) == PKV_CONSUMER_FMA;
  void (*const kern)(const CUtensorMap, const CUtensorMap, const DecodeArgs) =
      fma ? decode_kernel<D, split_stages(D), true> : decode_kernel<D, split_stages(D), false>;
  {
    std::lock_guard<std::mutex> lk(attn_mutex());
    int rc = maps_for(k_cache, v_cache, c, &tmk, &tmv);
    if (rc) return rc;
    int dev = 0;
    if ((rc = current_device(&dev))) return rc;
    const int vi = D == 64 ? 0 : 1;
    if (!g_split_attr[dev][vi][fma ? 1 : 0]) {
      cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)split_smem(D));
      if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
      e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(carveout)");
      g_split_attr[dev][vi][fma ? 1 : 0] = true;
    }
  }
  DecodeArgs a;
  a.q = q;
  a.block_tables = bt;
  a.context_lens = lens;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.out = out;
  a.counters = counters;
  a.fused = out == nullptr ? 0 : (cluster > 1 ? 2 : 1);
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
  a.scale_log2 = scale * kLog2e;
  a.sched = nullptr;
  a.num_seqs = num_seqs;
  a.q_wait = q_wait ? 1 : 0;
  dim3 grid((unsigned)a.n_parts, (unsigned)c.num_kv_heads, (unsigned)num_seqs);
  cudaError_t e;
  if (!programmatic && cluster <= 1) {
    kern<<<grid, kThreads, split_smem(D), stream>>>(tmk, tmv, a);
    e = cudaGetLastError();
  } else {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = split_smem(D);
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    unsigned n = 0;
    if (programmatic) {  // may start while the previous kernel (the slot write) still runs
      attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
      attr[n].val.programmaticStreamSerializationAllowed = 1;
      ++n;
    }
    if (cluster > 1) {  // the partitions of one (sequence, kv head) form a cluster
      attr[n].id = cudaLaunchAttributeClusterDimension;
      attr[n].val.clusterDim.x = (unsigned)cluster;
      attr[n].val.clusterDim.y = 1;
      attr[n].val.clusterDim.z = 1;
      ++n;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    e = cudaLaunchKernelEx(&cfg, kern, tmk, tmv, a);
  }
  if (e != cudaSuccess) return cuda_error(e, "decode_kernel launch");
  return PKV_OK;
}

constexpr int persist_stages(int d) { return d == 64 ? 4 : 3; }
constexpr size_t persist_smem(int d) {
  return 1024 + (d == 64 ? PersistSmem<64, persist_stages(64)>::total
                         : PersistSmem<128, persist_stages(128)>::total);
}
static_assert(persist_smem(64) * 3 + 3 * 1024 <= 228 * 1024 &&
                  persist_smem(128) * 2 + 2 * 1024 <= 228 * 1024,
              "the persistent kernel keeps decode_kernel's CTAs per SM");

// Whether the persistent kernel takes the fused decode: many (sequence, kv head) units
// (at least a wave of CTAs), a batch its per-CTA order tables hold, and a category
// count (full-partition levels + last-partition chunk counts) within kMaxCategories.
bool use_persistent(int32_t num_seqs, int32_t hkv, int32_t d, int32_t max_len, int32_t P,
                    int sms) {
  const int64_t units = (int64_t)num_seqs * hkv;
  const int64_t R = ((int64_t)max_len + P - 1) / P;
  const int64_t Q = P / kChunk;
  return units >= (int64_t)sms * split_occupancy(d) && num_seqs <= kMaxPersistSeqs &&
         P % kChunk == 0 && Q + kMergeChunks < kMaxCategories &&
         R - 1 + Q + kMergeChunks <= kMaxCategories;
}

template <int D>
int launch_persistent(const pkv_bf16 *q, const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                      const int32_t *bt, int32_t max_blocks, const int32_t *lens, int32_t max_len,
                      int32_t num_seqs, int32_t hq, const pkv_cache_desc &c, float scale,
                      int32_t P, float *o_part, float *lse_part, pkv_bf16 *out,
                      uint32_t *counters, uint32_t *sched, cudaStream_t stream,
                      bool programmatic) {
  constexpr int S = persist_stages(D);
  CUtensorMap tmk, tmv;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lk(attn_mutex());
    int rc = maps_for(k_cache, v_cache, c, &tmk, &tmv);
    if (rc) return rc;
    int dev = 0;
    if ((rc = current_device(&dev))) return rc;
    if ((rc = device_sms(&sms))) return rc;
    const int vi = D == 64 ? 0 : 1;
    if (!g_persist_attr[dev][vi]) {
      cudaError_t e = cudaFuncSetAttribute(decode_persistent_kernel<D, S>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)persist_smem(D));
      if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
      e = cudaFuncSetAttribute(decode_persistent_kernel<D, S>,
                               cudaFuncAttributePreferredSharedMemoryCarveout, 100);
      if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(carveout)");
      g_persist_attr[dev][vi] = true;
    }
  }
  DecodeArgs a;
  a.q = q;
  a.block_tables = bt;
  a.context_lens = lens;
  a.o_part = o_part;
  a.lse_part = lse_part;
  a.out = out;
  a.counters = counters;
  a.fused = 1;
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
  a.scale_log2 = scale * kLog2e;
  a.sched = sched;
  a.num_seqs = num_seqs;
  a.q_wait = 0;  // q arrives by the producer's bulk copy, issued after its griddepcontrol.wait
  // one wave: every CTA starts at once, none waits for another
  const int64_t items_max = (int64_t)num_seqs * c.num_kv_heads * a.n_parts;
  const int64_t slots = (int64_t)sms * split_occupancy(D);
  const unsigned grid = (unsigned)(items_max < slots ? items_max : slots);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = persist_smem(D);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = programmatic ? 1 : 0;
  const cudaError_t e = cudaLaunchKernelEx(&cfg, decode_persistent_kernel<D, S>, tmk, tmv, a);
  if (e != cudaSuccess) return cuda_error(e, "decode_persistent_kernel launch");
  return PKV_OK;
}

// The fused decode's kernel arrangement for these sizes on `sms` SMs (PKV_PATH_*).
int decode_path(int32_t num_seqs, int32_t hkv, int32_t d, int32_t max_len, int32_t P, int sms) {
  if (use_persistent(num_seqs, hkv, d, max_len, P, sms)) return PKV_PATH_PERSISTENT;
  if (cluster_parts(num_seqs, hkv, d, max_len, P, sms) > 1) return PKV_PATH_CLUSTER;
  return PKV_PATH_PARTITIONS;
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

int sms_or_default(int32_t num_sms) {
  if (num_sms > 0) return num_sms;
  std::lock_guard<std::mutex> lk(attn_mutex());
  int n = 0;
  if (device_sms(&n) != PKV_OK || n <= 0) n = 148;
  return n;
}

}  // namespace
}  // namespace pkv

using namespace pkv;

PKV_API int32_t paged_decode_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_context_len, int32_t num_sms) {
  if (num_seqs <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_q_heads % num_kv_heads ||
      num_q_heads / num_kv_heads > kMaxGroup || (head_dim != 64 && head_dim != 128) ||
      max_context_len <= 0)
    return 0;
  return plan_partition(num_seqs, num_kv_heads, head_dim, max_context_len, sms_or_default(num_sms));
}

PKV_API int32_t pkv_set_decode_consumer(int32_t consumer) {
  if (consumer != PKV_CONSUMER_TENSOR && consumer != PKV_CONSUMER_FMA)
    return set_error(PKV_ERR_UNSUPPORTED, "pkv_set_decode_consumer: unknown form %d", consumer);
  clear_error();
  return g_consumer.exchange(consumer);
}

namespace {
template <int D>
int32_t ctas_per_sm(int32_t path) {
  std::lock_guard<std::mutex> lk(attn_mutex());
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  const int vi = D == 64 ? 0 : 1;
  void (*kern)(const CUtensorMap, const CUtensorMap, const DecodeArgs);
  size_t smem;
  bool *attr;
  if (path == PKV_PATH_PERSISTENT) {
    kern = decode_persistent_kernel<D, persist_stages(D)>;
    smem = persist_smem(D);
    attr = &g_persist_attr[dev][vi];
  } else {
    const bool fma = g_consumer.load(std::memory_order_relaxed) == PKV_CONSUMER_FMA;
    kern = fma ? decode_kernel<D, split_stages(D), true> : decode_kernel<D, split_stages(D), false>;
    smem = split_smem(D);
    attr = &g_split_attr[dev][vi][fma ? 1 : 0];
  }
  if (!*attr) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute(carveout)");
    *attr = true;
  }
  int n = 0;
  const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kern, kThreads, smem);
  if (e != cudaSuccess) return cuda_error(e, "cudaOccupancyMaxActiveBlocksPerMultiprocessor");
  clear_error();
  return n;
}
}  // namespace

PKV_API int32_t pkv_decode_ctas_per_sm(int32_t head_dim, int32_t path) {
  if (path != PKV_PATH_PARTITIONS && path != PKV_PATH_CLUSTER && path != PKV_PATH_PERSISTENT)
    return set_error(PKV_ERR_UNSUPPORTED, "pkv_decode_ctas_per_sm: unknown path %d", path);
  if (head_dim == 64) return ctas_per_sm<64>(path);
  if (head_dim == 128) return ctas_per_sm<128>(path);
  return set_error(PKV_ERR_UNSUPPORTED, "pkv_decode_ctas_per_sm: head_dim %d", head_dim);
}

PKV_API int32_t paged_decode_path(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int32_t max_context_len, int32_t num_sms) {
  const int32_t mlen = max_context_len > 0 ? max_context_len : 1;
  const int sms = sms_or_default(num_sms);
  const int32_t P = paged_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, mlen, sms);
  if (P <= 0) return 0;
  return decode_path(num_seqs, num_kv_heads, head_dim, mlen, P, sms);
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
  const int32_t mlen = max_context_len > 0 ? max_context_len : 1;
  const int32_t P = paged_decode_plan(num_seqs, num_q_heads, num_kv_heads, head_dim, mlen, 0);
  if (P <= 0) return 0;
  return fused_layout(num_seqs, num_q_heads, num_kv_heads, head_dim, mlen, P).total;
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
           ? launch_split<64>(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                              max_context_len, num_seqs, num_q_heads, *cache, scale,
                              partition_tokens, o_part, lse_part, nullptr, nullptr, s)
           : launch_split<128>(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                               max_context_len, num_seqs, num_q_heads, *cache, scale,
                               partition_tokens, o_part, lse_part, nullptr, nullptr, s);
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
                          num_q_heads, head_dim, partition_tokens, static_cast<cudaStream_t>(stream));
  if (!rc) clear_error();
  return rc;
}

namespace pkv {
namespace {

// Checks and launches the fused decode; `programmatic` only when the previous kernel on
// the stream is this library's slot write (which writes nothing but cache rows).
int decode_fused(pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                 const pkv_bf16 *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                 const int32_t *context_lens, int32_t max_context_len, int32_t num_seqs,
                 int32_t num_q_heads, const pkv_cache_desc *cache, float scale, void *workspace,
                 size_t workspace_bytes, cudaStream_t s, bool programmatic, bool launch,
                 const char *fn, bool q_wait = false) {
  int rc = check_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        max_context_len, num_seqs, num_q_heads, cache, fn);
  if (rc) return rc;
  if (num_seqs == 0) return PKV_OK;
  if (!out) return set_error(PKV_ERR_NULL, "%s: out is NULL", fn);
  if (reinterpret_cast<uintptr_t>(out) & 7u)
    return set_error(PKV_ERR_ALIGN, "%s: out must be 8-byte aligned", fn);
  const int D = cache->head_dim;
  const int32_t mlen = max_context_len > 0 ? max_context_len : 1;  // all-empty: zero outputs
  const int32_t P = paged_decode_plan(num_seqs, num_q_heads, cache->num_kv_heads, D, mlen, 0);
  const FusedLayout f = fused_layout(num_seqs, num_q_heads, cache->num_kv_heads, D, mlen, P);
  if (!workspace || workspace_bytes < f.total)
    return set_error(PKV_ERR_WORKSPACE, "%s: workspace %zu bytes < %zu needed", fn,
                     workspace_bytes, f.total);
  if (!aligned16(workspace))
    return set_error(PKV_ERR_ALIGN, "%s: workspace must be 16-byte aligned", fn);
  if (!launch) return PKV_OK;
  char *ws = static_cast<char *>(workspace);
  uint32_t *counters = reinterpret_cast<uint32_t *>(ws + f.counters);
  float *o_part = reinterpret_cast<float *>(ws + f.o_part);
  float *lse_part = reinterpret_cast<float *>(ws + f.lse_part);
  const int path = decode_path(num_seqs, cache->num_kv_heads, D, mlen, P, sms_or_default(0));
  if (path == PKV_PATH_PERSISTENT) {
    uint32_t *sched = reinterpret_cast<uint32_t *>(ws + f.sched);
    return D == 64 ? launch_persistent<64>(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                           context_lens, mlen, num_seqs, num_q_heads, *cache,
                                           scale, P, o_part, lse_part, out, counters, sched, s,
                                           programmatic)
                   : launch_persistent<128>(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                            context_lens, mlen, num_seqs, num_q_heads, *cache,
                                            scale, P, o_part, lse_part, out, counters, sched, s,
                                            programmatic);
  }
  const int cluster = path == PKV_PATH_CLUSTER ? (mlen + P - 1) / P : 0;
  return D == 64 ? launch_split<64>(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                    context_lens, mlen, num_seqs, num_q_heads, *cache, scale, P,
                                    o_part, lse_part, out, counters, s, programmatic, cluster,
                                    q_wait)
                 : launch_split<128>(q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                                     context_lens, mlen, num_seqs, num_q_heads, *cache, scale, P,
                                     o_part, lse_part, out, counters, s, programmatic, cluster,
                                     q_wait);
}

}  // namespace

int check_decode_attention(const pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                           const pkv_bf16 *v_cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                           const pkv_cache_desc *cache, size_t workspace_bytes, const char *fn) {
  // Without a launch, decode_fused looks at the workspace pointer only to reject a NULL
  // or misaligned one; this stands for the caller's aligned buffer and is never used.
  void *const aligned_stand_in = reinterpret_cast<void *>(uintptr_t(256));
  return decode_fused(const_cast<pkv_bf16 *>(out), q, k_cache, v_cache, block_tables,
                      max_blocks_per_seq, context_lens, max_context_len, num_seqs, num_q_heads,
                      cache, 1.f, aligned_stand_in, workspace_bytes, nullptr, false, false, fn);
}

}  // namespace pkv

PKV_API int paged_decode_attention(pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                   const pkv_bf16 *v_cache, const int32_t *block_tables,
                                   int32_t max_blocks_per_seq, const int32_t *context_lens,
                                   int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                                   const pkv_cache_desc *cache, float scale, void *workspace,
                                   size_t workspace_bytes, void *stream) {
  const int rc = decode_fused(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                              context_lens, max_context_len, num_seqs, num_q_heads, cache, scale,
                              workspace, workspace_bytes, static_cast<cudaStream_t>(stream), false,
                              true, "paged_decode_attention");
  if (!rc) clear_error();
  return rc;
}

PKV_API int paged_decode_step(pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k,
                              const pkv_bf16 *v, const int64_t *slot_mapping, int64_t num_tokens,
                              pkv_bf16 *k_cache, pkv_bf16 *v_cache, const int32_t *block_tables,
                              int32_t max_blocks_per_seq, const int32_t *context_lens,
                              int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                              const pkv_cache_desc *cache, float scale, void *workspace,
                              size_t workspace_bytes, void *stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // check both halves before enqueuing either
  int rc = check_write(k, v, slot_mapping, num_tokens, k_cache, v_cache, cache);
  if (!rc)
    rc = decode_fused(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                      max_context_len, num_seqs, num_q_heads, cache, scale, workspace,
                      workspace_bytes, s, false, false, "paged_decode_step");
  if (rc) return rc;
  rc = launch_write(k, v, slot_mapping, num_tokens, k_cache, v_cache, *cache, s);
  if (!rc)
    rc = decode_fused(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                      max_context_len, num_seqs, num_q_heads, cache, scale, workspace,
                      workspace_bytes, s, num_tokens > 0, true, "paged_decode_step");
  if (!rc) clear_error();
  return rc;
}

PKV_API int paged_decode_step_rope(pkv_bf16 *out, pkv_bf16 *q, const pkv_bf16 *k,
                                   const pkv_bf16 *v, const int64_t *slot_mapping,
                                   const int64_t *positions, const float *cos_sin,
                                   int64_t max_position, int32_t rotary_dim, int32_t neox_style,
                                   pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                                   const int32_t *block_tables, int32_t max_blocks_per_seq,
                                   const int32_t *context_lens, int32_t max_context_len,
                                   int32_t num_seqs, int32_t num_q_heads,
                                   const pkv_cache_desc *cache, float scale, void *workspace,
                                   size_t workspace_bytes, void *stream) {
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // check both halves before enqueuing either; token b is sequence b's new token
  int rc = check_write_rope(k, v, q, num_q_heads, slot_mapping, positions, num_seqs, cos_sin,
                            max_position, rotary_dim, k_cache, v_cache, cache);
  if (!rc)
    rc = decode_fused(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                      max_context_len, num_seqs, num_q_heads, cache, scale, workspace,
                      workspace_bytes, s, false, false, "paged_decode_step_rope");
  if (rc) return rc;
  rc = launch_write_rope(k, v, q, num_q_heads, slot_mapping, positions, num_seqs, cos_sin,
                         max_position, rotary_dim, neox_style, k_cache, v_cache, *cache, s);
  if (!rc)
    rc = decode_fused(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                      max_context_len, num_seqs, num_q_heads, cache, scale, workspace,
                      workspace_bytes, s, num_seqs > 0, true, "paged_decode_step_rope", true);
  if (!rc) clear_error();
  return rc;
}
