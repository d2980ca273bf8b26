// pkv_prefill.cu -- paged prefill attention: causal multi-query attention of each
// sequence's newest tokens over the paged KV cache.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "attn_device.cuh"
#include "pkv_exp2.cuh"

// Of the 16 column pairs of each 32-column chunk of a score row, how many take their
// exponentials on the FMA pipe (exp2_fma) rather than the special-function unit, in
// row_block_exp and in the one-pass weights.  0: every fraction tried measured slower
// (2 pairs: -4 to -6%, 4 pairs: -8 to -15% on the four prefill workloads): the softmax
// waits on latency and issue, not on the special-function unit.
#ifndef PKV_PREFILL_POLY_PAIRS
#define PKV_PREFILL_POLY_PAIRS 0
#endif
// Row maxima with three-input max instructions (1) or two-input ones (0).
#ifndef PKV_PREFILL_MAX3
#define PKV_PREFILL_MAX3 1
#endif
// Scaled, max-subtracted scores two at a time with packed fp32 FMAs (1) or one at a time (0).
#ifndef PKV_PREFILL_FMA2
#define PKV_PREFILL_FMA2 1
#endif
// Row sums of the two-tile kernel at head_dim 64 formed by the tensor core (a column of
// ones appended to V) instead of by the softmax threads.
#ifndef PKV_PREFILL_SUM_MMA64
#define PKV_PREFILL_SUM_MMA64 1
#endif

// Row sums of the bf16 weights with mixed-precision adds (1) or widen-then-add (0).
#ifndef PKV_PREFILL_SUM_MIXED
#define PKV_PREFILL_SUM_MIXED 1
#endif

namespace pkv {

// ===========================================================================
// Paged prefill: causal attention of each sequence's newest tokens over the paged cache
// ("vLLM-Style Llama Inference Engine", How it works: prefill and recomputation use
// causal attention).  Sequence b holds L_b tokens; its last n_b = query_start[b+1] -
// query_start[b] are the queries; query i sits at position L_b - n_b + i and sees keys
// t <= that position.  A query row is a (query token, head of the kv head's group) pair.
struct PrefillArgs {
  const uint16_t *q;            // [Nq][Hq][D]
  const int32_t *block_tables;  // [B][max_blocks]
  const int32_t *context_lens;  // [B]
  const int32_t *query_start;   // [B + 1]
  uint16_t *out;                // [Nq][Hq][D]
  int64_t num_blocks;
  int32_t max_blocks, cap, num_q_heads, num_kv_heads, group, block_size, log2_bs, box_rows;
  float scale_log2;
};

// ===========================================================================
// prefill_tc_kernel: the same causal attention on the 5th-generation tensor cores.
//
// One CTA owns one (sequence, kv head, tile of 128 query rows) and walks the keys up to
// the tile's last position in blocks of 128.  Warps 0-3 run the softmax with one thread
// per row, warps 4 and 6 are the TMA producers (K and V), and one thread of warp 5
// issues the tensor-core instructions (with the build option of two softmax threads per
// row: warps 0-7, 8 and 10, and 9):
//   S_j = Q . K_j^T   tcgen05.mma M=128 N=128 K=D, Q and K_j K-major in shared memory
//                     (128-byte swizzle), S in TMEM, two buffers: S_{j+1} is computed
//                     while the softmax works on S_j;
//   softmax            per row in fp32, base 2, read straight out of TMEM; P_j =
//                     exp2(S - m) rounded to bf16, two buffers: at head_dim 128 in
//                     TMEM after O, at 64 in shared memory (K-major);
//   O += P_j . V_j    tcgen05.mma M=128 N=D K=128, P_j from TMEM (head_dim 128) or
//                     shared memory, V_j MN-major, O in TMEM.
// A row's reference max m moves only when a block raises it by more than 8 (a factor
// 256): then O and the row sum are rescaled in TMEM.  Otherwise P is taken against the
// older m, which the final division by the row sum cancels.  The row sum adds the
// bf16-rounded P values that the tensor cores multiply.  K and V stream through
// separate rings so that K runs a block ahead of V.
constexpr int kTcRows = 128;     // query rows per CTA
constexpr int kTcKeys = 128;     // keys per block
// One-tile kernel: softmax warps 0 .. 4H-1 (H threads per query row), producer warp 4H
// (the K ring, and the V ring unless warp 4H+2 fills it), MMA warp 4H+1.  One warp takes
// ~110 cycles per TMA box, so at block_size 32 a block's sixteen boxes took longer than
// its tensor-core work; with a second producer workload 5 went from 818 to 967 TFLOP/s.
#ifndef PKV_PREFILL_TC_TWO_PRODUCERS
#define PKV_PREFILL_TC_TWO_PRODUCERS 1
#endif
// One-tile kernel at head_dim 128: P in TMEM, two buffers at columns 256 + D and
// 320 + D (after O), read by P.V as its A operand (1), or in shared memory (0); and then
// the stages of the K and V rings: 2 (with the one-pass softmax, rings of 3 measured 8%
// slower on 4 sequences of 32K at block_size 32 and 64, 1% at 16).
#ifndef PKV_PREFILL_TC_P_TMEM
#define PKV_PREFILL_TC_P_TMEM 1
#endif
#ifndef PKV_PREFILL_TC_KS128
#define PKV_PREFILL_TC_KS128 2
#endif
// One-tile kernel at head_dim 128 (P in TMEM): softmax threads per query row (two
// measured 2% below one, with rings of 2), and with two the stages of the V ring.
#ifndef PKV_PREFILL_TC_HALVES128
#define PKV_PREFILL_TC_HALVES128 1
#endif
#ifndef PKV_PREFILL_TC_KSV128_H2
#define PKV_PREFILL_TC_KSV128_H2 2
#endif
constexpr int kTcProducers = PKV_PREFILL_TC_TWO_PRODUCERS ? 2 : 1;
template <int H>
__host__ __device__ constexpr int tc_threads() { return 32 * (4 * H + 1 + kTcProducers); }
constexpr float kTcRescale = 8.f;

// Whether the softmax reads a row's block from TMEM once into registers (1) or in each
// of the two passes (0), by head_dim: once at 128 (measured 7% faster).  At 64 twice was
// faster while P went through shared memory (the extra live registers cost more than
// the second read); with P in TMEM and the weights and max in one pass, once is.
#ifndef PKV_PREFILL_ROW_ONCE128
#define PKV_PREFILL_ROW_ONCE128 1
#endif
#ifndef PKV_PREFILL_ROW_ONCE64
#define PKV_PREFILL_ROW_ONCE64 1
#endif
template <int D>
__host__ __device__ constexpr bool row_once() { return D == 128 ? PKV_PREFILL_ROW_ONCE128 != 0 : PKV_PREFILL_ROW_ONCE64 != 0; }

template <int D, int H = 1>
struct TcSmem {
  // head_dim 128: P in TMEM (two 64-column buffers after O), no P buffers here
  static constexpr bool kPT = D == 128 && row_once<D>() && PKV_PREFILL_TC_P_TMEM != 0;
  static_assert(H == 1 || kPT, "two threads per row only with P in TMEM");
  static constexpr int KSK = D == 64 ? 3 : (kPT ? PKV_PREFILL_TC_KS128 : 2);  // K ring stages
  static constexpr int KSV = H == 2 ? PKV_PREFILL_TC_KSV128_H2 : KSK;         // V ring stages
  static constexpr uint32_t kSub = kTcKeys * 128;      // one 64-dim sub-tile of 128 rows
  static constexpr uint32_t kTile = kSub * (D / 64);   // one K or V block / the Q tile
  static constexpr uint32_t k = 0;
  static constexpr uint32_t v = k + KSK * kTile;
  static constexpr uint32_t q = v + KSV * kTile;       // [D/64][128 rows][128 B]
  static constexpr uint32_t p = q + kTile;             // two buffers of [2][128 rows][128 B]
  static constexpr uint32_t kP = 2 * kSub;
  // H = 2: the halves' row values, [2 buffers][2 halves][128 rows] fp32
  static constexpr uint32_t xchg = p + (kPT ? 0 : 2 * kP);
  static constexpr uint32_t bars = xchg + (H == 2 ? 2 * 2 * kTcRows * 4 : 0);
  // the rings, s_full/s_free/p_full/pv_done per buffer, q_ready, mma_done, and with
  // H = 2 one barrier per lane quadrant where the two halves of its rows meet
  static constexpr int kBars = 2 * KSK + 2 * KSV + 10 + (H == 2 ? 4 : 0);
  static constexpr uint32_t tslot = bars + kBars * 8;
  static constexpr uint32_t flag = tslot + 8;
  static constexpr uint32_t total = flag + 8;
};

// Loads keys [k0, k0 + nk) of one kv head into a block tile [D/64][128][128 B] (one TMA
// box of min(BS, 64) rows per lane), completing on `bar`.  win/tb: this ring's window of
// 32 block-table entries.
template <int D>
__device__ __forceinline__ void tc_load_block(const CUtensorMap *tm, uint32_t dst, uint32_t bar,
                                              int k0, int nk, int &win, int &tb,
                                              const int32_t *trow, int lb_last,
                                              const PrefillArgs &a, int g, int lane,
                                              uint64_t policy) {
  const int rb = a.box_rows;
  const int nbox = (nk + rb - 1) / rb;
  const int lb_hi = (k0 + (nbox - 1) * rb) >> a.log2_bs;
  if (lb_hi >= win + 32 || (k0 >> a.log2_bs) < win) {
    win = k0 >> a.log2_bs;
    tb = (win + lane <= lb_last) ? __ldg(trow + win + lane) : 0;
  }
  // one box per lane: box i = lane / (D / 64), 64-dim half lane % (D / 64), so that every
  // box of the block leaves from one instruction (block_size >= 8: nbox * D / 64 <= 32)
  constexpr int kH = D / 64;
  const int bi = lane / kH, hh = lane % kH;
  const int key = k0 + bi * rb;
  const int src = min(max((key >> a.log2_bs) - win, 0), 31);
  const int64_t phys_raw = __shfl_sync(0xffffffffu, tb, src);
  if (lane == 0) dev::mbar_arrive_expect_tx(bar, (uint32_t)nbox * rb * 128u * kH);
  __syncwarp();
  if (bi < nbox) {
    int64_t phys = phys_raw;
    if (phys < 0 || phys >= a.num_blocks) {
      raise_error(PKV_DEVERR_BLOCK_ID);
      phys = 0;
    }
    const int off = key & (a.block_size - 1);
    const int32_t row = (int32_t)((phys * a.num_kv_heads + g) * a.block_size + off);
    const uint32_t d = dst + (uint32_t)(bi * rb) * 128u;
    if constexpr (D == 64) {
      dev::tma_load_2d(d, tm, 0, row, bar, policy);
    } else {
      asm volatile(
          "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
          ".L2::cache_hint [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(d + hh * TcSmem<D>::kSub),
          "l"(reinterpret_cast<uint64_t>(tm)), "r"(0), "r"(hh), "r"(row), "r"(bar), "l"(policy)
          : "memory");
    }
  }
  __syncwarp();
}

// ---------------------------------------------------------------------------
// The softmax warps' work on one 128-column block of a score row in TMEM (one thread =
// one row = one TMEM lane).  TMEM is read in 32-column chunks with the next chunk's load
// in flight while the current one is processed.

// Waits for this thread's TMEM loads; the 32 registers the last one fills are tied to
// the wait, so that nothing reads them before it.
__device__ __forceinline__ void tmem_wait_ld_regs(uint32_t (&x)[32]) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(x[0]), "+r"(x[1]), "+r"(x[2]), "+r"(x[3]), "+r"(x[4]), "+r"(x[5]),
                 "+r"(x[6]), "+r"(x[7]), "+r"(x[8]), "+r"(x[9]), "+r"(x[10]), "+r"(x[11]),
                 "+r"(x[12]), "+r"(x[13]), "+r"(x[14]), "+r"(x[15]), "+r"(x[16]), "+r"(x[17]),
                 "+r"(x[18]), "+r"(x[19]), "+r"(x[20]), "+r"(x[21]), "+r"(x[22]), "+r"(x[23]),
                 "+r"(x[24]), "+r"(x[25]), "+r"(x[26]), "+r"(x[27]), "+r"(x[28]), "+r"(x[29]),
                 "+r"(x[30]), "+r"(x[31])
               :
               : "memory");
}

// c + lo(x) + hi(x) for a bf16 pair x: two mixed-precision adds (bf16 + fp32).
__device__ __forceinline__ float add_bf16x2(uint32_t x, float c) {
  float d;
  asm("{\n\t.reg .b16 lo, hi;\n\t.reg .f32 t;\n\t"
      "mov.b32 {lo, hi}, %1;\n\t"
      "add.rn.f32.bf16 t, lo, %2;\n\tadd.rn.f32.bf16 %0, hi, t;\n\t}"
      : "=f"(d)
      : "r"(x), "f"(c));
  return d;
}

// (x0, x1) * s + c, both lanes rounded once (fused), in one packed instruction.
__device__ __forceinline__ void fma_f32x2(float x0, float x1, float s, float c, float &d0,
                                          float &d1) {
  asm("{\n\t.reg .b64 x, sc, cc, d;\n\t"
      "mov.b64 x, {%2, %3};\n\tmov.b64 sc, {%4, %4};\n\tmov.b64 cc, {%5, %5};\n\t"
      "fma.rn.f32x2 d, x, sc, cc;\n\tmov.b64 {%0, %1}, d;\n\t}"
      : "=f"(d0), "=f"(d1)
      : "f"(x0), "f"(x1), "f"(s), "f"(c));
}

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// One 32-bit TMEM column of this thread's lane (load: complete with a wait).
__device__ __forceinline__ uint32_t tmem_ld1(uint32_t taddr) {
  uint32_t x;
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x1.b32 {%0}, [%1];" : "=r"(x) : "r"(taddr));
  return x;
}
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t x) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(x) : "memory");
}

// Pass 1: the row's maximum scaled score over the columns c <= lim (all of them when
// `whole`) of NCH 32-column chunks starting at chunk ch0.  With a positive scale, the
// max of the raw scores scaled once equals the max of the scaled scores (rounding is
// monotonic).
template <int NCH>
__device__ __forceinline__ float row_block_max(uint32_t sb, int ch0, int lim, bool whole,
                                               bool pos_scale, float scale_log2) {
  float mx[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
  const float sc = pos_scale ? 1.f : scale_log2;
  uint32_t xa[32], xb[32];
  dev::tmem_ld32(sb + ch0 * 32, xa);
  tmem_wait_ld_regs(xa);
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    uint32_t(&cur)[32] = (ch & 1) ? xb : xa;
    uint32_t(&nxt)[32] = (ch & 1) ? xa : xb;
    if (ch + 1 < NCH) dev::tmem_ld32(sb + (ch0 + ch + 1) * 32, nxt);
    const int lc = lim - (ch0 + ch) * 32;
    if (whole && pos_scale) {
#if PKV_PREFILL_MAX3
#pragma unroll
      for (int i = 0; i < 32; i += 2)
        mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], __uint_as_float(cur[i]), __uint_as_float(cur[i + 1]));
#else
#pragma unroll
      for (int i = 0; i < 32; ++i) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(cur[i]));
#endif
    } else if (whole) {
#pragma unroll
      for (int i = 0; i < 32; ++i) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(cur[i]) * sc);
    } else {
#pragma unroll
      for (int i = 0; i < 32; ++i)
        mx[i & 7] = fmaxf(mx[i & 7], i <= lc ? __uint_as_float(cur[i]) * sc : -INFINITY);
    }
    if (ch + 1 < NCH) tmem_wait_ld_regs(nxt);
  }
  float bmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                     fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
  return pos_scale ? bmax * scale_log2 : bmax;
}

// Pass 2: P = exp2(S * scale - m_ref) for the columns c <= lim (0 past it) of NCH
// 32-column chunks starting at chunk ch0, rounded to bf16 and stored into row r of the
// P buffer at shared offset `prow` (K-major, 128-byte swizzle: two 64-column sub-tiles
// `sub` bytes apart); returns the sum of the rounded values, which is what the tensor
// cores multiply.  The first PKV_PREFILL_POLY_PAIRS column pairs of each chunk take
// exp2_fma.
template <int NCH, bool kSum = true>
__device__ __forceinline__ float row_block_exp(uint32_t sb, int ch0, uint8_t *bp, uint32_t prow,
                                               uint32_t sub, int r, int lim, bool whole,
                                               float scale_log2, float m_ref) {
  float ls[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) ls[u] = 0.f;
  uint32_t xa[32], xb[32];
  dev::tmem_ld32(sb + ch0 * 32, xa);
  tmem_wait_ld_regs(xa);
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    uint32_t(&cur)[32] = (ch & 1) ? xb : xa;
    uint32_t(&nxt)[32] = (ch & 1) ? xa : xb;
    if (ch + 1 < NCH) dev::tmem_ld32(sb + (ch0 + ch + 1) * 32, nxt);
    const int cha = ch0 + ch;  // absolute chunk
    const int lc = whole ? 32 : lim - cha * 32;
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
#if PKV_PREFILL_FMA2
      float a0, a1;
      fma_f32x2(__uint_as_float(cur[2 * e]), __uint_as_float(cur[2 * e + 1]), scale_log2, -m_ref,
                a0, a1);
#else
      const float a0 = fmaf(__uint_as_float(cur[2 * e]), scale_log2, -m_ref);
      const float a1 = fmaf(__uint_as_float(cur[2 * e + 1]), scale_log2, -m_ref);
#endif
      float p0, p1;
      if (e < PKV_PREFILL_POLY_PAIRS) {
        p0 = dev::exp2_fma(a0);
        p1 = dev::exp2_fma(a1);
      } else {
        p0 = dev::ex2(a0);
        p1 = dev::ex2(a1);
      }
      if (!whole) {
        p0 = 2 * e <= lc ? p0 : 0.f;
        p1 = 2 * e + 1 <= lc ? p1 : 0.f;
      }
      pk[e] = dev::pack_bf16x2(p0, p1);
      // sum what the tensor cores multiply: with a stale reference max the largest P is
      // not a power of two, and only this keeps the weights a convex combination
      if constexpr (kSum) {
#if PKV_PREFILL_SUM_MIXED
        ls[e & 7] = add_bf16x2(pk[e], ls[e & 7]);
#else
        ls[(2 * e) & 7] += dev::bf16lo_to_f32(pk[e]);
        ls[(2 * e + 1) & 7] += dev::bf16hi_to_f32(pk[e]);
#endif
      }
    }
    const uint32_t dst = prow + (cha >> 1) * sub;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c16 = (cha & 1) * 4 + u;
      *reinterpret_cast<uint4 *>(bp + dst + ((c16 ^ (r & 7)) << 4)) =
          make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
    }
    if (ch + 1 < NCH) tmem_wait_ld_regs(nxt);
  }
  return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
}

// The same two passes from one read of the row's chunks into registers (TMEM is read
// once per block instead of twice).
template <int NCH>
__device__ __forceinline__ void row_block_load(uint32_t sb, int ch0, uint32_t (&x)[NCH * 32]) {
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    uint32_t(&c)[32] = *reinterpret_cast<uint32_t(*)[32]>(&x[ch * 32]);
    dev::tmem_ld32(sb + (ch0 + ch) * 32, c);
  }
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    uint32_t(&c)[32] = *reinterpret_cast<uint32_t(*)[32]>(&x[ch * 32]);
    if (ch == 0)
      tmem_wait_ld_regs(c);  // one wait covers every load above
    else
      asm volatile("" : "+r"(c[0]), "+r"(c[1]), "+r"(c[2]), "+r"(c[3]), "+r"(c[4]), "+r"(c[5]),
                   "+r"(c[6]), "+r"(c[7]), "+r"(c[8]), "+r"(c[9]), "+r"(c[10]), "+r"(c[11]),
                   "+r"(c[12]), "+r"(c[13]), "+r"(c[14]), "+r"(c[15]), "+r"(c[16]), "+r"(c[17]),
                   "+r"(c[18]), "+r"(c[19]), "+r"(c[20]), "+r"(c[21]), "+r"(c[22]), "+r"(c[23]),
                   "+r"(c[24]), "+r"(c[25]), "+r"(c[26]), "+r"(c[27]), "+r"(c[28]), "+r"(c[29]),
                   "+r"(c[30]), "+r"(c[31]));
  }
}

template <int NCH>
__device__ __forceinline__ float row_regs_max(const uint32_t (&x)[NCH * 32], int ch0, int lim,
                                              bool whole, bool pos_scale, float scale_log2) {
  float mx[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
  const float sc = pos_scale ? 1.f : scale_log2;
  if (whole && pos_scale) {
#pragma unroll
    for (int i = 0; i < NCH * 32; i += 2)
      mx[(i >> 1) & 7] = fmax3(mx[(i >> 1) & 7], __uint_as_float(x[i]), __uint_as_float(x[i + 1]));
  } else if (whole) {
#pragma unroll
    for (int i = 0; i < NCH * 32; ++i) mx[i & 7] = fmaxf(mx[i & 7], __uint_as_float(x[i]) * sc);
  } else {
    const int lc = lim - ch0 * 32;
#pragma unroll
    for (int i = 0; i < NCH * 32; ++i)
      mx[i & 7] = fmaxf(mx[i & 7], i <= lc ? __uint_as_float(x[i]) * sc : -INFINITY);
  }
  const float bmax = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                           fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
  return pos_scale ? bmax * scale_log2 : bmax;
}

template <int NCH>
__device__ __forceinline__ float row_regs_exp(const uint32_t (&x)[NCH * 32], int ch0, uint8_t *bp,
                                              uint32_t prow, uint32_t sub, int r, int lim,
                                              bool whole, float scale_log2, float m_ref) {
  float ls[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) ls[u] = 0.f;
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const int cha = ch0 + ch;
    const int lc = whole ? 32 : lim - cha * 32;
    uint32_t pk[16];
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float a0, a1;
      fma_f32x2(__uint_as_float(x[ch * 32 + 2 * e]), __uint_as_float(x[ch * 32 + 2 * e + 1]),
                scale_log2, -m_ref, a0, a1);
      float p0 = dev::ex2(a0), p1 = dev::ex2(a1);
      if (!whole) {
        p0 = 2 * e <= lc ? p0 : 0.f;
        p1 = 2 * e + 1 <= lc ? p1 : 0.f;
      }
      pk[e] = dev::pack_bf16x2(p0, p1);
      ls[e & 7] = add_bf16x2(pk[e], ls[e & 7]);
    }
    const uint32_t dst = prow + (cha >> 1) * sub;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c16 = (cha & 1) * 4 + u;
      *reinterpret_cast<uint4 *>(bp + dst + ((c16 ^ (r & 7)) << 4)) =
          make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
    }
  }
  return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
}

// Pass 2 from registers, without the stores: the rounded weights stay packed in `pk`
// (column pair e of chunk ch at pk[16 ch + e]) until the P buffer is free; returns their
// sum, as row_regs_exp.
template <int NCH, bool kSum = true>
__device__ __forceinline__ float row_regs_exp_pk(const uint32_t (&x)[NCH * 32], int ch0, int lim,
                                                 bool whole, float scale_log2, float m_ref,
                                                 uint32_t (&pk)[NCH * 16]) {
  float ls[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) ls[u] = 0.f;
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const int lc = whole ? 32 : lim - (ch0 + ch) * 32;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      float a0, a1;
      fma_f32x2(__uint_as_float(x[ch * 32 + 2 * e]), __uint_as_float(x[ch * 32 + 2 * e + 1]),
                scale_log2, -m_ref, a0, a1);
      float p0 = dev::ex2(a0), p1 = dev::ex2(a1);
      if (!whole) {
        p0 = 2 * e <= lc ? p0 : 0.f;
        p1 = 2 * e + 1 <= lc ? p1 : 0.f;
      }
      pk[ch * 16 + e] = dev::pack_bf16x2(p0, p1);
      if constexpr (kSum) ls[e & 7] = add_bf16x2(pk[ch * 16 + e], ls[e & 7]);
    }
  }
  return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
}

// The body of row_regs_exp_pk_max for one masking mode, the running maxima in mx.
template <int NCH, bool kSum, int kMode>  // kMode 0: whole, positive scale; 1: whole; 2: masked
__device__ __forceinline__ float row_regs_exp_pk_max_impl(const uint32_t (&x)[NCH * 32], int ch0,
                                                          int lim, float sc, float scale_log2,
                                                          float m_ref, uint32_t (&pk)[NCH * 16],
                                                          float (&mx)[8]) {
  float ls[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) ls[u] = 0.f;
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const int lc = kMode == 2 ? lim - (ch0 + ch) * 32 : 32;
#pragma unroll
    for (int e = 0; e < 16; ++e) {
      const float x0 = __uint_as_float(x[ch * 32 + 2 * e]), x1 = __uint_as_float(x[ch * 32 + 2 * e + 1]);
      if constexpr (kMode == 0)
        mx[e & 7] = fmax3(mx[e & 7], x0, x1);
      else if constexpr (kMode == 1)
        mx[e & 7] = fmax3(mx[e & 7], x0 * sc, x1 * sc);
      else
        mx[e & 7] = fmax3(mx[e & 7], 2 * e <= lc ? x0 * sc : -INFINITY,
                          2 * e + 1 <= lc ? x1 * sc : -INFINITY);
      float a0, a1;
      fma_f32x2(x0, x1, scale_log2, -m_ref, a0, a1);
      float p0, p1;
      if (e < PKV_PREFILL_POLY_PAIRS) {
        p0 = dev::exp2_fma(a0);
        p1 = dev::exp2_fma(a1);
      } else {
        p0 = dev::ex2(a0);
        p1 = dev::ex2(a1);
      }
      if constexpr (kMode == 2) {
        p0 = 2 * e <= lc ? p0 : 0.f;
        p1 = 2 * e + 1 <= lc ? p1 : 0.f;
      }
      pk[ch * 16 + e] = dev::pack_bf16x2(p0, p1);
      if constexpr (kSum) ls[e & 7] = add_bf16x2(pk[ch * 16 + e], ls[e & 7]);
    }
  }
  return ((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7]));
}

// row_regs_exp_pk and row_regs_max in one pass: the weights against a reference m_ref
// taken before the block's max is known, and that max (as row_regs_max returns it) in
// *bmax.  Weights of columns far above m_ref may overflow; the caller recomputes them
// once the max says the reference must move.
template <int NCH, bool kSum = true>
__device__ __forceinline__ float row_regs_exp_pk_max(const uint32_t (&x)[NCH * 32], int ch0, int lim,
                                                     bool whole, bool pos_scale, float scale_log2,
                                                     float m_ref, uint32_t (&pk)[NCH * 16],
                                                     float *bmax) {
  float mx[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) mx[u] = -INFINITY;
  const float sc = pos_scale ? 1.f : scale_log2;
  float ls;
  if (whole && pos_scale)
    ls = row_regs_exp_pk_max_impl<NCH, kSum, 0>(x, ch0, lim, sc, scale_log2, m_ref, pk, mx);
  else if (whole)
    ls = row_regs_exp_pk_max_impl<NCH, kSum, 1>(x, ch0, lim, sc, scale_log2, m_ref, pk, mx);
  else
    ls = row_regs_exp_pk_max_impl<NCH, kSum, 2>(x, ch0, lim, sc, scale_log2, m_ref, pk, mx);
  const float m = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                        fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
  *bmax = pos_scale ? m * scale_log2 : m;
  return ls;
}

// Stores the packed weights of row_regs_exp_pk into row r of the P buffer (K-major,
// 128-byte swizzle, two 64-column sub-tiles `sub` bytes apart).
template <int NCH>
__device__ __forceinline__ void row_store_p(const uint32_t (&pk)[NCH * 16], int ch0, uint8_t *bp,
                                            uint32_t prow, uint32_t sub, int r) {
#pragma unroll
  for (int ch = 0; ch < NCH; ++ch) {
    const int cha = ch0 + ch;
    const uint32_t dst = prow + (cha >> 1) * sub;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int c16 = (cha & 1) * 4 + u;
      *reinterpret_cast<uint4 *>(bp + dst + ((c16 ^ (r & 7)) << 4)) =
          make_uint4(pk[ch * 16 + 4 * u], pk[ch * 16 + 4 * u + 1], pk[ch * 16 + 4 * u + 2],
                     pk[ch * 16 + 4 * u + 3]);
    }
  }
}


// Two-tile kernel, rows read once: the softmax releases S_t(j) (s_free) as soon as it
// holds the block in registers, so S_t(j+1) runs on the tensor core during the block's
// exponentials instead of after them, and it waits for PV_t(j-1) only once its weights
// are computed, right before it overwrites the P buffer (1); or S_t(j+1) is issued once
// P_t(j) is complete and the wait comes before the exponentials (0).
#ifndef PKV_PREFILL_EARLY_S
#define PKV_PREFILL_EARLY_S 1
#endif
// Two-tile kernel at head_dim 128: the softmax writes P into TMEM over its S buffer
// (the columns it has read) and P.V reads it from there (A operand in TMEM), so P never passes
// through shared memory, whose bandwidth the operand reads of both MMAs, the TMA writes
// and the P stores otherwise share; the freed buffers give V a second stage.  The
// tensor core then takes PV_t(j) before S_t(j+1) overwrites the buffer (the MMAs of
// one thread run in issue order).  Takes precedence over PKV_PREFILL_EARLY_S.
#ifndef PKV_PREFILL_P_TMEM
#define PKV_PREFILL_P_TMEM 1
#endif
// With P in TMEM, blocks after the first take their weights against the reference max
// they start with and their max in the same pass, recomputing the weights only when the
// block moves the reference (1); or the max first, then the weights (0).
#ifndef PKV_PREFILL_ONE_PASS
#define PKV_PREFILL_ONE_PASS 1
#endif
// The same at head_dim 64 (there with rows read once, PKV_PREFILL_ROW_ONCE64): alone
// within 1% of P in shared memory, 10% / 7% faster on the two D = 64 workloads once the
// one-pass weights came with it.
#ifndef PKV_PREFILL_P_TMEM64
#define PKV_PREFILL_P_TMEM64 1
#endif
// K and V ring stages of the two-tile kernel at head_dim 128 with P in TMEM.
#ifndef PKV_PREFILL_KSK128
#define PKV_PREFILL_KSK128 2
#endif
#ifndef PKV_PREFILL_KSV128
#define PKV_PREFILL_KSV128 2
#endif

// ---------------------------------------------------------------------------
// Tensor-core issue.  A tcgen05.mma returns to the issuing thread only once the tensor
// core has taken it, about as long as it then runs (~65 cycles for M=128, N<=128, K=16),
// so any work the thread does between two of them leaves the tensor core idle.  The MMA
// thread therefore builds every descriptor before a sequence and issues four at a time
// from one straight-line block: the first accumulates per `acc_first`, the others always.

// Adds a byte offset (a multiple of 16) to a shared-memory descriptor's start address.
__device__ __forceinline__ uint64_t desc_add(uint64_t desc, uint32_t bytes) {
  return desc + (uint64_t)(bytes >> 4);
}

__device__ __forceinline__ void umma4(uint32_t d_tmem, uint64_t a0, uint64_t a1, uint64_t a2,
                                      uint64_t a3, uint64_t b0, uint64_t b1, uint64_t b2,
                                      uint64_t b3, uint32_t idesc, uint32_t acc_first) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %10, 0;\n\tsetp.eq.u32 q, 1, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %5, %9, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %2, %6, %9, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %3, %7, %9, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %4, %8, %9, q;\n\t}" ::"r"(d_tmem),
      "l"(a0), "l"(a1), "l"(a2), "l"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(idesc),
      "r"(acc_first)
      : "memory");
}

// S = Q . K^T over D: D/16 MMAs of K = 16.  q, k: descriptors of the K-major, 128-byte
// swizzled tiles (64-dim sub-tiles `sub` bytes apart).
template <int D>
__device__ __forceinline__ void issue_qk(uint32_t d_tmem, uint64_t q, uint64_t k, uint32_t sub,
                                         uint32_t idesc) {
#pragma unroll
  for (int g4 = 0; g4 < D / 64; ++g4) {
    const uint32_t o = g4 * sub;
    umma4(d_tmem, desc_add(q, o), desc_add(q, o + 32), desc_add(q, o + 64), desc_add(q, o + 96),
          desc_add(k, o), desc_add(k, o + 32), desc_add(k, o + 64), desc_add(k, o + 96), idesc,
          g4 > 0 ? 1u : 0u);
  }
}

// O (+)= P . V over a block of kTcKeys keys: kTcKeys/16 MMAs of K = 16.  p: descriptor of
// the K-major P buffer (64-key sub-tiles `sub` bytes apart); v: descriptor of the
// MN-major V tile (16 keys = 2048 bytes apart).
__device__ __forceinline__ void issue_pv(uint32_t d_tmem, uint64_t p, uint64_t v, uint32_t sub,
                                         uint32_t idesc, uint32_t acc_first) {
#pragma unroll
  for (int g4 = 0; g4 < kTcKeys / 64; ++g4) {
    const uint32_t o = g4 * sub, vo = g4 * 4 * 2048u;
    umma4(d_tmem, desc_add(p, o), desc_add(p, o + 32), desc_add(p, o + 64), desc_add(p, o + 96),
          desc_add(v, vo), desc_add(v, vo + 2048), desc_add(v, vo + 4096), desc_add(v, vo + 6144),
          idesc, g4 > 0 ? 1u : acc_first);
  }
}

// The same with P read from TMEM (the A operand in TMEM: row i in lane i, column c
// holding keys 2c and 2c+1): p_tmem is P's first column; K slice kk is 8 columns on.
__device__ __forceinline__ void umma4_ts(uint32_t d_tmem, uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint64_t b0, uint64_t b1, uint64_t b2,
                                         uint64_t b3, uint32_t idesc, uint32_t acc_first) {
  asm volatile(
      "{\n\t.reg .pred p, q;\n\tsetp.ne.b32 p, %10, 0;\n\tsetp.eq.u32 q, 1, 1;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %5, %9, p;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %9, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %9, q;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%4], %8, %9, q;\n\t}" ::"r"(d_tmem),
      "r"(a0), "r"(a1), "r"(a2), "r"(a3), "l"(b0), "l"(b1), "l"(b2), "l"(b3), "r"(idesc),
      "r"(acc_first)
      : "memory");
}
__device__ __forceinline__ void issue_pv_ts(uint32_t d_tmem, uint32_t p_tmem, uint64_t v,
                                            uint32_t idesc, uint32_t acc_first,
                                            uint32_t group_cols = 32u) {
#pragma unroll
  for (int g4 = 0; g4 < kTcKeys / 64; ++g4) {
    const uint32_t a = p_tmem + group_cols * g4, vo = g4 * 4 * 2048u;
    umma4_ts(d_tmem, a, a + 8, a + 16, a + 24, desc_add(v, vo), desc_add(v, vo + 2048),
             desc_add(v, vo + 4096), desc_add(v, vo + 6144), idesc, g4 > 0 ? 1u : acc_first);
  }
}

template <int D, int H>
__global__ void __launch_bounds__(tc_threads<H>(), 1)
    prefill_tc_kernel(const __grid_constant__ CUtensorMap tmk,
                      const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
  using SL = TcSmem<D, H>;
  constexpr int KSK = SL::KSK, KSV = SL::KSV;
  constexpr int kSoftWarps = 4 * H;
  constexpr int kProducer = kSoftWarps, kMma = kSoftWarps + 1, kProducerV = kSoftWarps + 2;
  constexpr int NCH = kTcKeys / 32 / H;  // 32-column chunks of a block per thread
  constexpr bool kOnePass = SL::kPT && PKV_PREFILL_ONE_PASS != 0;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const bp = smem_raw + (base - raw);
  const uint32_t bars = base + SL::bars;
  constexpr int R4 = 2 * KSK + 2 * KSV;  // barriers of the two rings
  auto k_full = [&](int s) { return bars + 8u * s; };
  auto k_empty = [&](int s) { return bars + 8u * (KSK + s); };
  auto v_full = [&](int s) { return bars + 8u * (2 * KSK + s); };
  auto v_empty = [&](int s) { return bars + 8u * (2 * KSK + KSV + s); };
  // two of each of these, one per S (and P) buffer, so that no barrier can run two
  // phases ahead of its waiter
  auto s_full = [&](int i) { return bars + 8u * (R4 + i); };
  auto s_free = [&](int i) { return bars + 8u * (R4 + 2 + i); };
  auto p_full = [&](int i) { return bars + 8u * (R4 + 4 + i); };
  auto pv_done = [&](int i) { return bars + 8u * (R4 + 6 + i); };
  const uint32_t q_ready = bars + 8u * (R4 + 8);
  const uint32_t mma_done = bars + 8u * (R4 + 9);
  auto pair_bar = [&](int wq) { return bars + 8u * (R4 + 10 + wq); };
  volatile uint32_t *const s_tmem = reinterpret_cast<volatile uint32_t *>(bp + SL::tslot);
  volatile int *const s_flag = reinterpret_cast<volatile int *>(bp + SL::flag);

  const int tile = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.group;

  int L = __ldg(a.context_lens + b);
  const int q0 = __ldg(a.query_start + b);
  int n = __ldg(a.query_start + b + 1) - q0;
  if (L < 0 || L > a.cap || n < 0 || n > L) {
    if (tid == 0 && tile == 0) raise_error(PKV_DEVERR_CONTEXT_LEN);
    L = L < 0 ? 0 : (L > a.cap ? a.cap : L);
    n = n < 0 ? 0 : (n > L ? L : n);
  }
  const int rows = n * G;  // query rows of this (b, g)
  const int row0 = tile * kTcRows;
  // rows past the grid (n_b > max_query_len) would go unwritten: flag it
  if (tile == 0 && tid == 0 && (int64_t)rows > (int64_t)gridDim.x * kTcRows)
    raise_error(PKV_DEVERR_CONTEXT_LEN);
  if (row0 >= rows) return;
  const int last_row = min(row0 + kTcRows, rows) - 1;
  const int t_end = L - n + last_row / G + 1;  // keys the tile needs: [0, t_end)
  const int nblk = (t_end + kTcKeys - 1) / kTcKeys;

  // the producers' first window of block-table entries, under the set-up below
  const bool is_producer = warp == kProducer || (kTcProducers == 2 && warp == kProducerV);
  const int32_t *const trow = a.block_tables + (int64_t)b * a.max_blocks;
  const int lb_last = (t_end - 1) >> a.log2_bs;
  const int tb_first = (is_producer && lane <= lb_last) ? __ldg(trow + lane) : 0;

  if (tid == 0) {
    // one arrival each (the producer, or a tensor-core commit), except s_free, p_full and
    // q_ready: one arrival per softmax warp; and the pair barriers: every thread of the
    // two warps that share a lane quadrant
    for (int i = 0; i < SL::kBars; ++i) {
      const uint32_t bar = bars + 8u * i;
      const bool per_warp = bar == s_free(0) || bar == s_free(1) || bar == p_full(0) ||
                            bar == p_full(1) || bar == q_ready;
      dev::mbar_init(bar, i >= R4 + 10 ? 64u : per_warp ? (uint32_t)kSoftWarps : 1u);
    }
    *s_flag = 0;
    dev::fence_mbar_init();
  }
  if (warp == 0) dev::tmem_alloc(base + SL::tslot, 512);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *s_tmem;  // S buffers at columns 0 and 128, O at 256

  auto fail = [&](bool ok) {
    if (!ok) {
      raise_error(PKV_DEVERR_TIMEOUT);
      *s_flag = 1;
    }
    return ok;
  };
  int k_issued = 0, v_issued = 0;  // producer: blocks loaded into each ring

  if (warp == kProducer || (kTcProducers == 2 && warp == kProducerV)) {
    // ---------------------------------------------------------- producer warp(s)
    const bool do_k = warp == kProducer, do_v = kTcProducers == 1 || warp == kProducerV;
    // every query tile of this (sequence, kv head) reads the same blocks: keep them in L2
    const uint64_t policy = dev::policy_evict_last();
    int kwin = 0, vwin = 0;
    int ktb = tb_first;
    int vtb = ktb;
    for (int j = 0; j <= nblk; ++j) {  // K runs one block ahead of V
      if (do_k && j < nblk) {
        const int s = j % KSK;
        if (j >= KSK && !__all_sync(0xffffffffu, dev::mbar_wait(k_empty(s), ((j / KSK) - 1) & 1))) {
          if (lane == 0) fail(false);
          break;
        }
        tc_load_block<D>(&tmk, base + SL::k + s * SL::kTile, k_full(s), j * kTcKeys,
                         min(kTcKeys, t_end - j * kTcKeys), kwin, ktb, trow, lb_last, a, g, lane,
                         policy);
        k_issued = j + 1;
      }
      if (do_v && j >= 1) {
        const int jv = j - 1, s = jv % KSV;
        if (jv >= KSV && !__all_sync(0xffffffffu, dev::mbar_wait(v_empty(s), ((jv / KSV) - 1) & 1))) {
          if (lane == 0) fail(false);
          break;
        }
        tc_load_block<D>(&tmv, base + SL::v + s * SL::kTile, v_full(s), jv * kTcKeys,
                         min(kTcKeys, t_end - jv * kTcKeys), vwin, vtb, trow, lb_last, a, g, lane,
                         policy);
        v_issued = jv + 1;
      }
    }
  } else if (warp == kMma) {
    // ------------------------------------------------- tensor-core issue (one thread)
    if (lane == 0) {
      constexpr uint32_t id_s = dev::idesc_bf16_f32(kTcRows, kTcKeys, 0);
      constexpr uint32_t id_o = dev::idesc_bf16_f32(kTcRows, D, 1);
      // descriptors of the Q tile, K stage 0, V stage 0 and P buffer 0 (the others are
      // whole tiles / buffers further on)
      const uint64_t dq = dev::smem_desc(base + SL::q, 16, 1024);
      const uint64_t dk0 = dev::smem_desc(base + SL::k, 16, 1024);
      const uint64_t dv0 = dev::smem_desc(base + SL::v, SL::kSub, 1024);
      const uint64_t dp0 = dev::smem_desc(base + SL::p, 16, 1024);
      bool ok = fail(dev::mbar_wait(q_ready, 0));
      auto issue_s = [&](int j) {
        const int s = j % KSK;
        if (!fail(dev::mbar_wait(k_full(s), (j / KSK) & 1))) return false;
        if (j >= 2 && !fail(dev::mbar_wait(s_free(j & 1), ((j >> 1) - 1) & 1))) return false;
        dev::tc_fence_after();
        issue_qk<D>(tmem + 128u * (j & 1), dq, desc_add(dk0, s * SL::kTile), SL::kSub, id_s);
        dev::umma_commit(s_full(j & 1));
        dev::umma_commit(k_empty(s));
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nblk; ++j) {
        if (j + 1 < nblk && !(ok = issue_s(j + 1))) break;
        const int s = j % KSV;
        if (!(ok = fail(dev::mbar_wait(p_full(j & 1), (j >> 1) & 1)))) break;
        if (!(ok = fail(dev::mbar_wait(v_full(s), (j / KSV) & 1)))) break;
        dev::tc_fence_after();
        if constexpr (SL::kPT)
          issue_pv_ts(tmem + 256u, tmem + 256u + D + 64u * (j & 1), desc_add(dv0, s * SL::kTile),
                      id_o, j > 0 ? 1u : 0u);
        else
          issue_pv(tmem + 256u, desc_add(dp0, (j & 1) * SL::kP), desc_add(dv0, s * SL::kTile),
                   SL::kSub, id_o, j > 0 ? 1u : 0u);
        dev::umma_commit(pv_done(j & 1));
        dev::umma_commit(v_empty(s));
      }
      dev::umma_commit(mma_done);  // arrives once everything issued above has completed
    }
  } else {
    // ---------------------------------------- softmax warps: row r, half hc of each block
    const int wq = warp & 3;    // TMEM lane quadrant of this warp
    const int hc = warp >> 2;   // which H-th of the columns
    const int r = 32 * wq + lane;
    const int gr = row0 + r;
    const bool valid = gr < rows;
    const int qi = valid ? gr / G : last_row / G;
    const int h = valid ? gr - (gr / G) * G : 0;
    const int pos = L - n + qi;                    // keys t <= pos are seen
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    // The two halves of a row exchange a value through shared memory: exchange k writes
    // buffer k & 1 and arrives on the quadrant's pair barrier (every thread of both
    // warps), whose phase k then publishes both values.  A half is at most one phase ahead
    // of the other, so it never overwrites a buffer its partner has yet to read.  The wait
    // is bounded; if it gives up, the row keeps its own value and the error is raised.
    float *const xchg = reinterpret_cast<float *>(bp + SL::xchg);  // [buf][half][row]
    int xuse = 0;
    auto other_half = [&](float v, bool &good) -> float {
      if constexpr (H == 2) {
        const int use = xuse++;
        xchg[((use & 1) * 2 + hc) * kTcRows + r] = v;
        dev::mbar_arrive(pair_bar(wq));
        if (!__all_sync(0xffffffffu, dev::mbar_wait(pair_bar(wq), use & 1))) {
          good = false;
          return v;
        }
        return xchg[((use & 1) * 2 + (hc ^ 1)) * kTcRows + r];
      } else {
        return v;
      }
    };
    // the tile's query rows into shared memory (K-major, 128-byte swizzle); zeros past the
    // end; this half's chunks [hc D/8/H, (hc+1) D/8/H)
    {
      const uint4 *src = reinterpret_cast<const uint4 *>(
          a.q + ((int64_t)(q0 + qi) * a.num_q_heads + g * G + h) * D);
#pragma unroll
      for (int cc = 0; cc < D / 8 / H; ++cc) {
        const int c = hc * (D / 8 / H) + cc;
        const uint4 v = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(bp + SL::q + (c >> 3) * SL::kSub + r * 128 +
                                   (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      dev::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(q_ready);
    }
    float m_ref = -INFINITY, lsum = 0.f;
    const bool pos_scale = a.scale_log2 > 0.f;
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      const int k0 = j * kTcKeys;
      const int nk = min(kTcKeys, t_end - k0);
      const int lim = min(pos, t_end - 1) - k0;  // columns c <= lim are seen by this row
      if (!(ok = __all_sync(0xffffffffu, dev::mbar_wait(s_full(j & 1), (j >> 1) & 1)))) break;
      dev::tc_fence_after();
      // this thread's part of the S row: NCH chunks of 32 columns
      const uint32_t sbase = tmem + lane_base + 128u * (j & 1);
      // the same for both halves of a row: its rows and the block are the same
      const bool whole = __all_sync(0xffffffffu, lim >= kTcKeys - 1);  // no column masked
      uint32_t xrow[row_once<D>() ? NCH * 32 : 1];
      const bool one_pass = kOnePass && j > 0;  // the max comes with the weights below
      float hmax = -INFINITY;
      if constexpr (row_once<D>()) {
        row_block_load<NCH>(sbase, hc * NCH, xrow);
        if (!one_pass) hmax = row_regs_max<NCH>(xrow, hc * NCH, lim, whole, pos_scale, a.scale_log2);
      } else {
        hmax = row_block_max<NCH>(sbase, hc * NCH, lim, whole, pos_scale, a.scale_log2);
      }
      // O_t moves by f (and the row sum with it) once the previous P.V is in
      auto rescale_o = [&](float f) {
        if (!__all_sync(0xffffffffu, dev::mbar_wait(pv_done((j - 1) & 1), ((j - 1) >> 1) & 1)))
          return false;
        dev::tc_fence_after();
#pragma unroll 1
        for (int ch = hc * (D / 32 / H); ch < (hc + 1) * (D / 32 / H); ++ch) {
          uint32_t o[32];
          dev::tmem_ld32(tmem + lane_base + 256u + ch * 32, o);
          dev::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          dev::tmem_st32(tmem + lane_base + 256u + ch * 32, o);
        }
        dev::tmem_wait_st();
        lsum *= f;
        return true;
      };
      if (!one_pass) {
        const float bmax = fmaxf(hmax, other_half(hmax, ok));
        if (!ok) break;
        if (j > 0) {
          const bool need = bmax > m_ref + kTcRescale;
          if (__any_sync(0xffffffffu, need)) {
            const float m_new = fmaxf(m_ref, bmax);
            if (!(ok = rescale_o(need ? dev::ex2(m_ref - m_new) : 1.f))) break;
            if (need) m_ref = m_new;
          }
        } else {
          m_ref = bmax;  // block 0 holds key 0, which every row sees
        }
      }
      // P = exp2(S - m_ref) as bf16 into TMEM (or shared memory), and its row sum
      if constexpr (SL::kPT) {
        uint32_t pk[NCH * 16];
        float ls;
        if (one_pass) {
          float bm;
          ls = row_regs_exp_pk_max<NCH>(xrow, hc * NCH, lim, whole, pos_scale, a.scale_log2,
                                        m_ref, pk, &bm);
          bm = fmaxf(bm, other_half(bm, ok));
          if (!ok) break;
          const bool need = bm > m_ref + kTcRescale;
          if (__any_sync(0xffffffffu, need)) {  // the reference moves: the weights again,
                                                // from S_j read once more
            const float m_new = fmaxf(m_ref, bm);
            if (!(ok = rescale_o(need ? dev::ex2(m_ref - m_new) : 1.f))) break;
            if (need) m_ref = m_new;
            row_block_load<NCH>(sbase, hc * NCH, xrow);
            ls = row_regs_exp_pk<NCH>(xrow, hc * NCH, lim, whole, a.scale_log2, m_ref, pk);
          }
        } else {
          ls = row_regs_exp_pk<NCH>(xrow, hc * NCH, lim, whole, a.scale_log2, m_ref, pk);
        }
        lsum += ls;
        // this P buffer is free once the P.V of two blocks back has completed
        if (j >= 2 && !(ok = __all_sync(0xffffffffu,
                                        dev::mbar_wait(pv_done(j & 1), ((j - 2) >> 1) & 1))))
          break;
        const uint32_t pb = tmem + lane_base + 256u + D + 64u * (j & 1) + 32u * (hc * NCH / 2);
#pragma unroll
        for (int i = 0; i < NCH / 2; ++i)
          dev::tmem_st32(pb + 32u * i, *reinterpret_cast<uint32_t(*)[32]>(&pk[32 * i]));
        dev::tmem_wait_st();
      } else {
        // this P buffer is free once the P.V of two blocks back has completed
        if (j >= 2 && !(ok = __all_sync(0xffffffffu,
                                        dev::mbar_wait(pv_done(j & 1), ((j - 2) >> 1) & 1))))
          break;
        if constexpr (row_once<D>())
          lsum += row_regs_exp<kTcKeys / 32>(xrow, 0, bp, SL::p + (j & 1) * SL::kP + r * 128,
                                             SL::kSub, r, lim, whole, a.scale_log2, m_ref);
        else
          lsum += row_block_exp<kTcKeys / 32>(sbase, 0, bp, SL::p + (j & 1) * SL::kP + r * 128,
                                              SL::kSub, r, lim, whole, a.scale_log2, m_ref);
      }
      // S read: the MMA warp may refill this buffer
      dev::tc_fence_before();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(s_free(j & 1));
      if (nk < kTcKeys) {  // last block: V rows past the keys hold stale or unowned data
        const int s = j % KSV;
        if (!(ok = __all_sync(0xffffffffu, dev::mbar_wait(v_full(s), (j / KSV) & 1)))) break;
        const uint32_t vt = SL::v + s * SL::kTile;
        for (int idx = hc * kTcRows + r; idx < (kTcKeys - nk) * (D / 8); idx += H * kTcRows) {
          const int row = nk + idx / (D / 8), c = idx % (D / 8);
          *reinterpret_cast<uint4 *>(bp + vt + (c >> 3) * SL::kSub + row * 128 +
                                     (((c & 7) ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      dev::tc_fence_before();
      dev::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(p_full(j & 1));
    }
    if (!ok && lane == 0) fail(false);
    // the row sum: both halves' parts
    float ltot = lsum;
    if (H == 2 && ok) ltot = lsum + other_half(lsum, ok);
    // epilogue: O / l as bf16, this half's D/H columns
    if (ok && __all_sync(0xffffffffu, dev::mbar_wait(pv_done((nblk - 1) & 1), ((nblk - 1) >> 1) & 1))) {
      dev::tc_fence_after();
      const float inv = 1.f / ltot;
      uint4 *dst = reinterpret_cast<uint4 *>(
          a.out + ((int64_t)(q0 + qi) * a.num_q_heads + g * G + h) * D);
#pragma unroll 1
      for (int ch = hc * (D / 32 / H); ch < (hc + 1) * (D / 32 / H); ++ch) {
        uint32_t o[32];
        dev::tmem_ld32(tmem + lane_base + 256u + ch * 32, o);
        dev::tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w4[e] = dev::pack_bf16x2(__uint_as_float(o[8 * u + 2 * e]) * inv,
                                       __uint_as_float(o[8 * u + 2 * e + 1]) * inv);
            dst[ch * 4 + u] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
    } else if (ok && lane == 0) {
      fail(false);
    }
  }

  // ---- teardown: no tensor-core op or copy may still be in flight when TMEM is freed
  if (tid == 0) (void)dev::mbar_wait(mma_done, 0);
  if ((warp == kProducer || (kTcProducers == 2 && warp == kProducerV)) && lane == 0 && *s_flag) {
    for (int s = 0; s < KSK; ++s) {
      const int kl = s + ((k_issued - 1 - s) / KSK) * KSK;
      if (kl >= 0 && kl < k_issued) (void)dev::mbar_wait(k_full(s), (kl / KSK) & 1);
    }
    for (int s = 0; s < KSV; ++s) {
      const int vl = s + ((v_issued - 1 - s) / KSV) * KSV;
      if (vl >= 0 && vl < v_issued) (void)dev::mbar_wait(v_full(s), (vl / KSV) & 1);
    }
  }
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  if (warp == 0) dev::tmem_dealloc(tmem, 512);
}

// ===========================================================================
// prefill_tc2_kernel: two query tiles per CTA in ping-pong.
//
// A CTA owns 256 query rows as two 128-row tiles of the same (sequence, kv head):
// softmax warps of tile t own its rows, and while one tile's warps work on its scores
// the tensor core works on the other tile; every K/V block staged feeds 256 rows.  Each
// tile has one S buffer in TMEM.
//  * P in TMEM (the default at both head dims): P_t(j) is written into TMEM over
//    columns of S_t(j) that the softmax has read, and the tensor-core thread issues
//    PV_0(j), S_0(j+1), PV_1(j), S_1(j+1): the MMAs of one thread run in issue order, so
//    S_t(j+1) overwrites the buffer only after PV_t(j) has read it, and s_full(t) (which
//    tracks every MMA issued before it) tells the softmax that O_t is stable.  K and V
//    rings of 2 at head_dim 128, each filled by its own producer warp; of 3 at 64, one
//    producer for both.
//  * P in shared memory (build options): one P buffer per tile.  The tensor-core thread
//    issues S_0(j+1), PV_0(j), S_1(j+1), PV_1(j): S_t(j+1) goes out once P_t(j) is
//    complete (p_full), ahead of PV_t(j), and the softmax waits for PV_t(j) (pv_done)
//    before it rescales O_t or overwrites P_t.
// Row arithmetic (positions, masking, lazy rescale, bf16 row sums) is the one-tile
// kernel's.  H softmax threads per query row (2 at head_dim 128, 1 at 64): with H = 2,
// two warps share each 32-row lane quadrant, one taking the first 64 columns of every
// key block, the other the last 64; their row maxima and row sums are combined through
// shared memory.  Warps 0 .. 8H-1 are the two tiles' softmax warps (tile t: warps
// 4H t .. 4H t + 4H - 1), then the producer, the MMA warp and (head_dim 128) the V
// producer.
// Producer warps of the two-tile kernel: at head_dim 128 one for the K ring and one for
// the V ring (a block's sixteen 2 KB boxes take a warp ~1800 cycles to issue at
// block_size 16, as long as the block's tensor-core work: measured +1.3%); at head_dim
// 64 one for both (two, and rings of 4, measured within 1%: the softmax sets the pace).
#ifndef PKV_PREFILL_TWO_PRODUCERS128
#define PKV_PREFILL_TWO_PRODUCERS128 1
#endif
#ifndef PKV_PREFILL_TWO_PRODUCERS64
#define PKV_PREFILL_TWO_PRODUCERS64 0
#endif
// K and V ring stages of the two-tile kernel at head_dim 64.
#ifndef PKV_PREFILL_KS64
#define PKV_PREFILL_KS64 3
#endif
template <int D>
__host__ __device__ constexpr int tc2_producers() {
  return (D == 128 ? PKV_PREFILL_TWO_PRODUCERS128 : PKV_PREFILL_TWO_PRODUCERS64) ? 2 : 1;
}
template <int D, int H>
__host__ __device__ constexpr int tc2_threads() { return 32 * (8 * H + 1 + tc2_producers<D>()); }

template <int D, int H>
struct Tc2Smem {
  // P in TMEM (no P buffers in shared memory)
  static constexpr bool kPT = row_once<D>() &&
                              (D == 128 ? PKV_PREFILL_P_TMEM != 0 : PKV_PREFILL_P_TMEM64 != 0);
  static constexpr int KSK = D == 64 ? PKV_PREFILL_KS64 : (kPT ? PKV_PREFILL_KSK128 : 2);  // K ring stages
  static constexpr int KSV = D == 64 ? PKV_PREFILL_KS64 : (kPT ? PKV_PREFILL_KSV128 : 1);  // V ring stages
  static constexpr uint32_t kSub = kTcKeys * 128;    // 128 rows x 128 B (64 dims)
  static constexpr uint32_t kTile = kSub * (D / 64); // one K or V block / one Q tile
  static constexpr uint32_t k = 0;
  static constexpr uint32_t v = k + KSK * kTile;
  static constexpr uint32_t q = v + KSV * kTile;     // two Q tiles
  static constexpr uint32_t p = q + 2 * kTile;       // two P buffers [2][128 rows][128 B]
  static constexpr uint32_t kP = 2 * kSub;
  // H = 2: the halves' row values, [2 buffers][2 tiles][2 halves][128 rows] fp32
  static constexpr uint32_t xchg = p + (kPT ? 0 : 2 * kP);
  // kOnes: a [128 keys][64] bf16 tile of ones, read by P.V as 16 extra B columns, so that
  // the tensor core also forms each row's sum of the bf16 weights (in O's extra columns)
  static constexpr bool kOnes = D == 64 && PKV_PREFILL_SUM_MMA64 != 0;
  static constexpr uint32_t ones = (xchg + (H == 2 ? 2 * 2 * 2 * kTcRows * 4 : 0) + 1023u) & ~1023u;
  static constexpr uint32_t bars = ones + (kOnes ? kSub : 0);
  // the rings, s_full/p_full/pv_done per tile, q_ready, mma_done, with H = 2 one
  // barrier per (tile, lane quadrant) where the two halves of its rows meet, then
  // s_free per tile
  static constexpr int kBars = 2 * KSK + 2 * KSV + 8 + (H == 2 ? 8 : 0) + 2;
  static constexpr uint32_t tslot = bars + kBars * 8;
  static constexpr uint32_t flag = tslot + 8;
  static constexpr uint32_t total = flag + 8;
};

template <int D, int H>
__global__ void __launch_bounds__(tc2_threads<D, H>(), 1)
    prefill_tc2_kernel(const __grid_constant__ CUtensorMap tmk,
                       const __grid_constant__ CUtensorMap tmv, const PrefillArgs a) {
  using SL = Tc2Smem<D, H>;
  constexpr int KSK = SL::KSK, KSV = SL::KSV;
  constexpr int kSoftWarps = 8 * H;        // softmax warps of both tiles
  constexpr int kTileWarps = 4 * H;        // softmax warps of one tile
  constexpr int kProducer = kSoftWarps, kMma = kSoftWarps + 1, kProducerV = kSoftWarps + 2;
  constexpr int NCH = kTcKeys / 32 / H;    // 32-column chunks of a block per thread
  constexpr bool kOnes = SL::kOnes;        // row sums from the tensor core
  constexpr int kON = D + (kOnes ? 16 : 0);  // O columns per tile (then the row sums)
  constexpr bool kPT = SL::kPT;           // P in TMEM, over S_t
  // P_t's columns within S_t: one thread a row reads the whole row before it writes,
  // so P takes the upper 64 columns (keys 0-63 then 64-127); with two threads a row,
  // each half writes its 32 columns of P over the first 32 of the 64 it has read
  constexpr uint32_t kPCol = H == 1 ? 64u : 0u, kPGroup = H == 1 ? 32u : 64u;
  constexpr bool kOnePass = kPT && PKV_PREFILL_ONE_PASS != 0;
  constexpr bool kEarlyS = !kPT && PKV_PREFILL_EARLY_S != 0 && row_once<D>();
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const bp = smem_raw + (base - raw);
  const uint32_t bars = base + SL::bars;
  constexpr int R4 = 2 * KSK + 2 * KSV;  // barriers of the two rings
  auto k_full = [&](int s) { return bars + 8u * s; };
  auto k_empty = [&](int s) { return bars + 8u * (KSK + s); };
  auto v_full = [&](int s) { return bars + 8u * (2 * KSK + s); };
  auto v_empty = [&](int s) { return bars + 8u * (2 * KSK + KSV + s); };
  auto s_full = [&](int t) { return bars + 8u * (R4 + t); };
  auto p_full = [&](int t) { return bars + 8u * (R4 + 2 + t); };
  auto pv_done = [&](int t) { return bars + 8u * (R4 + 4 + t); };
  const uint32_t q_ready = bars + 8u * (R4 + 6);
  const uint32_t mma_done = bars + 8u * (R4 + 7);
  auto pair_bar = [&](int t, int wq) { return bars + 8u * (R4 + 8 + 4 * t + wq); };
  auto s_free = [&](int t) { return bars + 8u * (SL::kBars - 2 + t); };
  volatile uint32_t *const s_tmem = reinterpret_cast<volatile uint32_t *>(bp + SL::tslot);
  volatile int *const s_flag = reinterpret_cast<volatile int *>(bp + SL::flag);

  const int tile = blockIdx.x, g = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.group;

  int L = __ldg(a.context_lens + b);
  const int q0 = __ldg(a.query_start + b);
  int n = __ldg(a.query_start + b + 1) - q0;
  if (L < 0 || L > a.cap || n < 0 || n > L) {
    if (tid == 0 && tile == 0) raise_error(PKV_DEVERR_CONTEXT_LEN);
    L = L < 0 ? 0 : (L > a.cap ? a.cap : L);
    n = n < 0 ? 0 : (n > L ? L : n);
  }
  const int rows = n * G;
  const int row0 = tile * 2 * kTcRows;
  // rows past the grid (n_b > max_query_len) would go unwritten: flag it
  if (tile == 0 && tid == 0 && (int64_t)rows > (int64_t)gridDim.x * 2 * kTcRows)
    raise_error(PKV_DEVERR_CONTEXT_LEN);
  if (row0 >= rows) return;
  // per tile: its last row, the keys it needs [0, t_end_t), its blocks
  int t_end_t[2], nblk_t[2];
#pragma unroll
  for (int t = 0; t < 2; ++t) {
    const int first = row0 + t * kTcRows;
    if (first >= rows) {
      t_end_t[t] = 0;
      nblk_t[t] = 0;
    } else {
      const int last = min(first + kTcRows, rows) - 1;
      t_end_t[t] = L - n + last / G + 1;
      nblk_t[t] = (t_end_t[t] + kTcKeys - 1) / kTcKeys;
    }
  }
  const int t_end = max(t_end_t[0], t_end_t[1]);  // keys the CTA stages
  const int nblk = max(nblk_t[0], nblk_t[1]);
  auto nblk_of = [&](int t) { return t ? nblk_t[1] : nblk_t[0]; };

  // The producers' first window of block-table entries goes out before the set-up, so
  // that its latency runs under the barrier initialisation and the TMEM allocation.  (The
  // softmax threads' query rows wait until after it: loaded before the barrier they held
  // every warp, the producers too, behind their latency: -3% on workload 3.)
  const bool is_producer = warp == kProducer || (tc2_producers<D>() == 2 && warp == kProducerV);
  const int32_t *const trow = a.block_tables + (int64_t)b * a.max_blocks;
  const int lb_last = (t_end - 1) >> a.log2_bs;
  const int tb_first = (is_producer && lane <= lb_last) ? __ldg(trow + lane) : 0;

  if (tid == 0) {
    for (int i = 0; i < SL::kBars; ++i) {
      const uint32_t bar = bars + 8u * i;
      const bool per_warp = bar == p_full(0) || bar == p_full(1) || bar == s_free(0) ||
                            bar == s_free(1);
      const bool pair = i >= R4 + 8 && i < SL::kBars - 2;  // every thread of the halves' warps
      dev::mbar_init(bar, pair ? 64u
                               : per_warp ? (uint32_t)kTileWarps
                                          : (bar == q_ready ? (uint32_t)kSoftWarps : 1u));
    }
    *s_flag = 0;
    dev::fence_mbar_init();
  }
  if constexpr (kOnes) {  // bf16 1.0 everywhere; read by the tensor cores (async proxy)
    for (int i = tid; i < (int)(SL::kSub / 16); i += tc2_threads<D, H>())
      *reinterpret_cast<uint4 *>(bp + SL::ones + i * 16) =
          make_uint4(0x3F803F80u, 0x3F803F80u, 0x3F803F80u, 0x3F803F80u);
    dev::fence_proxy_async_smem();
  }
  if (warp == 0) dev::tmem_alloc(base + SL::tslot, 512);
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  const uint32_t tmem = *s_tmem;  // S of tile t at column 128 t, O of tile t at 256 + kON t

  auto fail = [&](bool ok) {
    if (!ok) {
      raise_error(PKV_DEVERR_TIMEOUT);
      *s_flag = 1;
    }
    return ok;
  };
  int k_issued = 0, v_issued = 0;

  if (warp == kProducer || (tc2_producers<D>() == 2 && warp == kProducerV)) {
    // ---------------------------------------------------------- producer warp(s)
    const bool do_k = warp == kProducer, do_v = tc2_producers<D>() == 1 || warp == kProducerV;
    const uint64_t policy = dev::policy_evict_last();
    int kwin = 0, vwin = 0;
    int ktb = tb_first;
    int vtb = ktb;
    for (int j = 0; j <= nblk; ++j) {  // K runs one block ahead of V
      if (do_k && j < nblk) {
        const int s = j % KSK;
        if (j >= KSK && !__all_sync(0xffffffffu, dev::mbar_wait(k_empty(s), ((j / KSK) - 1) & 1))) {
          if (lane == 0) fail(false);
          break;
        }
        tc_load_block<D>(&tmk, base + SL::k + s * SL::kTile, k_full(s), j * kTcKeys,
                         min(kTcKeys, t_end - j * kTcKeys), kwin, ktb, trow, lb_last, a, g, lane,
                         policy);
        k_issued = j + 1;
      }
      if (do_v && j >= 1) {
        const int jv = j - 1, s = jv % KSV;
        if (jv >= KSV && !__all_sync(0xffffffffu, dev::mbar_wait(v_empty(s), ((jv / KSV) - 1) & 1))) {
          if (lane == 0) fail(false);
          break;
        }
        tc_load_block<D>(&tmv, base + SL::v + s * SL::kTile, v_full(s), jv * kTcKeys,
                         min(kTcKeys, t_end - jv * kTcKeys), vwin, vtb, trow, lb_last, a, g, lane,
                         policy);
        v_issued = jv + 1;
      }
    }
  } else if (warp == kMma) {
    // ------------------------------------------------- tensor-core issue (one thread)
    if (lane == 0) {
      constexpr uint32_t id_s = dev::idesc_bf16_f32(kTcRows, kTcKeys, 0);
      constexpr uint32_t id_o = dev::idesc_bf16_f32(kTcRows, kON, 1);
      bool ok = fail(dev::mbar_wait(q_ready, 0));
      int k_waited = 0;  // K blocks whose k_full this thread has seen
      auto need_k = [&](int j) {
        if (j < k_waited) return true;
        if (!fail(dev::mbar_wait(k_full(j % KSK), (j / KSK) & 1))) return false;
        k_waited = j + 1;
        dev::tc_fence_after();
        return true;
      };
      const uint64_t dq0 = dev::smem_desc(base + SL::q, 16, 1024);
      const uint64_t dk0 = dev::smem_desc(base + SL::k, 16, 1024);
      // V stage s as the MN-major B operand: the next 64 columns are V's other half
      // (head_dim 128) or, with kOnes, the tile of ones, `lbo` bytes further on
      auto dv = [&](int s) {
        const uint32_t vs = SL::v + s * SL::kTile;
        return dev::smem_desc(base + vs, kOnes ? SL::ones - vs : SL::kSub, 1024);
      };
      const uint64_t dp0 = dev::smem_desc(base + SL::p, 16, 1024);
      auto issue_s = [&](int t, int j) {
        issue_qk<D>(tmem + 128u * t, desc_add(dq0, t * SL::kTile),
                    desc_add(dk0, (j % KSK) * SL::kTile), SL::kSub, id_s);
        dev::umma_commit(s_full(t));
        // K_j is free once the last tile that reads it has its S
        if (t == 1 || j >= nblk_of(1)) dev::umma_commit(k_empty(j % KSK));
      };
      if (ok && (ok = need_k(0))) {
        issue_s(0, 0);
        if (nblk_of(1) > 0) issue_s(1, 0);
      }
      for (int j = 0; ok && j < nblk; ++j) {
        if constexpr (kEarlyS) {  // S_t(j+1) once the softmax holds S_t(j) in registers
          for (int t = 0; t < 2 && ok; ++t) {
            if (j + 1 >= nblk_of(t)) continue;
            if (!(ok = fail(dev::mbar_wait(s_free(t), j & 1)))) break;
            dev::tc_fence_after();
            if (!(ok = need_k(j + 1))) break;
            issue_s(t, j + 1);
          }
        }
        bool v_seen = false;
        for (int t = 0; t < 2 && ok; ++t) {
          if (j >= nblk_of(t)) continue;
          if (!(ok = fail(dev::mbar_wait(p_full(t), j & 1)))) break;
          dev::tc_fence_after();
          // S_t(j+1) first: the softmax can start on it while the tensor core runs PV_t(j)
          if (!kEarlyS && !kPT && j + 1 < nblk_of(t)) {
            if (!(ok = need_k(j + 1))) break;
            issue_s(t, j + 1);
          }
          if (!v_seen) {
            if (!(ok = fail(dev::mbar_wait(v_full(j % KSV), (j / KSV) & 1)))) break;
            v_seen = true;
            dev::tc_fence_after();
          }
          if constexpr (kPT) {
            issue_pv_ts(tmem + 256u + (uint32_t)(kON * t), tmem + 128u * t + kPCol, dv(j % KSV),
                        id_o, j > 0 ? 1u : 0u, kPGroup);
            dev::umma_commit(pv_done(t));
            // V_j is free once the last tile that reads it has its P.V
            if (t == 1 || j >= nblk_of(1)) dev::umma_commit(v_empty(j % KSV));
            // S_t(j+1) over S_t(j) and P_t(j), after the P.V that reads P_t(j)
            if (j + 1 < nblk_of(t)) {
              if (!(ok = need_k(j + 1))) break;
              issue_s(t, j + 1);
            }
          } else {
            issue_pv(tmem + 256u + (uint32_t)(kON * t), desc_add(dp0, t * SL::kP), dv(j % KSV),
                     SL::kSub, id_o, j > 0 ? 1u : 0u);
            dev::umma_commit(pv_done(t));
          }
        }
        if (ok && !kPT) dev::umma_commit(v_empty(j % KSV));
      }
      dev::umma_commit(mma_done);
    }
  } else {
    // ------------------------- softmax warps of tile t: row r, half hc of each block
    const int t = warp / kTileWarps;
    const int wq = warp & 3;                       // TMEM lane quadrant of this warp
    const int hc = (warp % kTileWarps) >> 2;       // which H-th of the columns
    const int r = 32 * wq + lane;
    const int gr = row0 + t * kTcRows + r;
    const bool valid = gr < rows;
    const int last_row_t = min(row0 + t * kTcRows + kTcRows, rows) - 1;
    const int qi = valid ? gr / G : (last_row_t >= 0 ? last_row_t / G : 0);
    const int h = valid ? gr - (gr / G) * G : 0;
    const int pos = L - n + qi;
    const uint32_t lane_base = (uint32_t)(32 * wq) << 16;
    const uint32_t sb = tmem + lane_base + 128u * t;
    const uint32_t ob = tmem + lane_base + 256u + (uint32_t)(kON * t);
    // The two halves of a row exchange a value through shared memory: use k writes
    // buffer k & 1 and arrives on the pair's barrier (every thread of both warps), whose
    // phase k then publishes both values.  A half is at most one phase ahead of the
    // other, so it never overwrites a buffer its partner has yet to read.  The wait is
    // bounded; if it gives up, the row keeps its own value and the error is raised.
    float *const xchg = reinterpret_cast<float *>(bp + SL::xchg);  // [buf][t][half][row]
    auto other_half = [&](float v, int use, bool &good) -> float {
      if constexpr (H == 2) {
        xchg[(((use & 1) * 2 + t) * 2 + hc) * kTcRows + r] = v;
        dev::mbar_arrive(pair_bar(t, wq));
        if (!__all_sync(0xffffffffu, dev::mbar_wait(pair_bar(t, wq), use & 1))) {
          good = false;
          return v;
        }
        return xchg[(((use & 1) * 2 + t) * 2 + (hc ^ 1)) * kTcRows + r];
      } else {
        return v;
      }
    };
    {  // this tile's query rows (zeros past the end): chunks [hc D/8/H, (hc+1) D/8/H)
      const uint4 *src = reinterpret_cast<const uint4 *>(
          a.q + ((int64_t)(q0 + qi) * a.num_q_heads + g * G + h) * D);
#pragma unroll
      for (int cc = 0; cc < D / 8 / H; ++cc) {
        const int c = hc * (D / 8 / H) + cc;
        const uint4 v = valid ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        *reinterpret_cast<uint4 *>(bp + SL::q + t * SL::kTile + (c >> 3) * SL::kSub + r * 128 +
                                   (((c & 7) ^ (r & 7)) << 4)) = v;
      }
      dev::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(q_ready);
    }
    const int nb = nblk_of(t);
    const int te = t ? t_end_t[1] : t_end_t[0];
    float m_ref = -INFINITY, lsum = 0.f;
    const bool pos_scale = a.scale_log2 > 0.f;
    bool ok = true;
    for (int j = 0; j < nb; ++j) {
      const int k0 = j * kTcKeys;
      const int lim = min(pos, te - 1) - k0;
      if (!(ok = __all_sync(0xffffffffu, dev::mbar_wait(s_full(t), j & 1)))) break;
      dev::tc_fence_after();
      // the same for both halves of a row: its rows and the block are the same
      const bool whole = __all_sync(0xffffffffu, lim >= kTcKeys - 1);
      uint32_t xrow[row_once<D>() ? NCH * 32 : 1];
      float hmax = -INFINITY;
      const bool one_pass = kOnePass && j > 0;  // the max comes with the weights below
      if constexpr (row_once<D>()) {
        row_block_load<NCH>(sb, hc * NCH, xrow);
        if constexpr (kEarlyS) {  // S_t(j) is in registers: the tensor core may overwrite it
          dev::tc_fence_before();
          __syncwarp();
          if (lane == 0) dev::mbar_arrive(s_free(t));
        }
        if (!one_pass) hmax = row_regs_max<NCH>(xrow, hc * NCH, lim, whole, pos_scale, a.scale_log2);
      } else {
        hmax = row_block_max<NCH>(sb, hc * NCH, lim, whole, pos_scale, a.scale_log2);
      }
      float bmax = hmax;
      if (!one_pass) {  // with one_pass the halves exchange their maxima after the weights
        bmax = fmaxf(hmax, other_half(hmax, j, ok));
        if (!ok) break;
      }
      // Lazy rescaling: the reference max moves only when the block raises it by more
      // than kTcRescale; then O_t (and its row-sum column) and the row sum scale by f.
      float f = 1.f;
      bool resc = false;
      if (one_pass) {
        // decided after the weights, below
      } else if (j > 0) {
        const bool need = bmax > m_ref + kTcRescale;
        resc = __any_sync(0xffffffffu, need);
        if (resc) {
          const float m_new = fmaxf(m_ref, bmax);
          f = need ? dev::ex2(m_ref - m_new) : 1.f;
          if (need) m_ref = m_new;
        }
      } else {
        m_ref = bmax;
      }
      auto rescale_o = [&]() {  // each half rescales its D/H columns of O
#pragma unroll 1
        for (int ch = hc * (D / 32 / H); ch < (hc + 1) * (D / 32 / H); ++ch) {
          uint32_t o[32];
          dev::tmem_ld32(ob + ch * 32, o);
          dev::tmem_wait_ld();
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          dev::tmem_st32(ob + ch * 32, o);
        }
        if constexpr (kOnes) {  // the row sum in O's column D (the first half's)
          if (hc == 0) {
            const uint32_t sm = tmem_ld1(ob + D);
            dev::tmem_wait_ld();
            tmem_st1(ob + D, __float_as_uint(__uint_as_float(sm) * f));
          }
        }
        dev::tmem_wait_st();
        lsum *= f;
      };
      if constexpr (kPT) {
        // P_t(j) into TMEM over S_t, in columns this thread has read.  PV_t(j-1) was
        // issued before S_t(j) by the same thread, and s_full tracks every MMA issued
        // before its commit, so O_t is stable here.
        uint32_t pk[NCH * 16];
        float ls;
        if (one_pass) {
          float bm;
          ls = row_regs_exp_pk_max<NCH, !kOnes>(xrow, hc * NCH, lim, whole, pos_scale,
                                                a.scale_log2, m_ref, pk, &bm);
          if constexpr (H == 2) {
            bm = fmaxf(bm, other_half(bm, j, ok));
            if (!ok) break;
          }
          const bool need = bm > m_ref + kTcRescale;
          resc = __any_sync(0xffffffffu, need);
          if (resc) {  // the reference moves: the weights again, against the new one, from
                       // S_t(j) read once more (the registers were spent on the first pass)
            const float m_new = fmaxf(m_ref, bm);
            f = need ? dev::ex2(m_ref - m_new) : 1.f;
            if (need) m_ref = m_new;
            row_block_load<NCH>(sb, hc * NCH, xrow);
            ls = row_regs_exp_pk<NCH, !kOnes>(xrow, hc * NCH, lim, whole, a.scale_log2, m_ref,
                                              pk);
          }
        } else {
          ls = row_regs_exp_pk<NCH, !kOnes>(xrow, hc * NCH, lim, whole, a.scale_log2, m_ref, pk);
        }
        if (resc) rescale_o();
        lsum += ls;
#pragma unroll
        for (int i = 0; i < NCH / 2; ++i)
          dev::tmem_st32(sb + kPCol + kPGroup * hc + 32u * i,
                         *reinterpret_cast<uint32_t(*)[32]>(&pk[32 * i]));
        dev::tmem_wait_st();
      } else if constexpr (kEarlyS) {
        // the block's weights first, kept in registers; then, once PV_t(j-1) has
        // completed (O_t stable, P buffer free), the rescale and the P stores
        uint32_t pk[NCH * 16];
        const float ls =
            row_regs_exp_pk<NCH, !kOnes>(xrow, hc * NCH, lim, whole, a.scale_log2, m_ref, pk);
        if (j > 0) {
          if (!(ok = __all_sync(0xffffffffu, dev::mbar_wait(pv_done(t), (j - 1) & 1)))) break;
          dev::tc_fence_after();
          if (resc) rescale_o();
        }
        lsum += ls;
        row_store_p<NCH>(pk, hc * NCH, bp, SL::p + t * SL::kP + r * 128, SL::kSub, r);
      } else {
        // O_t is stable and the P buffer free once PV_t(j-1) has completed
        if (j > 0 && !(ok = __all_sync(0xffffffffu, dev::mbar_wait(pv_done(t), (j - 1) & 1)))) break;
        if (resc) rescale_o();
        if constexpr (row_once<D>())
          lsum += row_regs_exp<NCH>(xrow, hc * NCH, bp, SL::p + t * SL::kP + r * 128, SL::kSub, r,
                                    lim, whole, a.scale_log2, m_ref);
        else
          lsum += row_block_exp<NCH, !kOnes>(sb, hc * NCH, bp, SL::p + t * SL::kP + r * 128,
                                             SL::kSub, r, lim, whole, a.scale_log2, m_ref);
      }
      const int nk = min(kTcKeys, t_end - k0);  // keys the CTA staged in this block
      if (nk < kTcKeys) {  // the CTA's last block: V rows past its keys are stale or unowned
        const int s = j % KSV;
        if (!(ok = __all_sync(0xffffffffu, dev::mbar_wait(v_full(s), (j / KSV) & 1)))) break;
        const uint32_t vt = SL::v + s * SL::kTile;
        for (int idx = hc * kTcRows + r; idx < (kTcKeys - nk) * (D / 8); idx += H * kTcRows) {
          const int row = nk + idx / (D / 8), c = idx % (D / 8);
          *reinterpret_cast<uint4 *>(bp + vt + (c >> 3) * SL::kSub + row * 128 +
                                     (((c & 7) ^ (row & 7)) << 4)) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      dev::tc_fence_before();
      dev::fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(p_full(t));
    }
    if (!ok && lane == 0) fail(false);
    // the row sum: both halves' parts (exchange number nb of the pair)
    float ltot = lsum;
    if (H == 2 && ok) ltot = lsum + other_half(lsum, nb, ok);
    if (ok && nb > 0 && __all_sync(0xffffffffu, dev::mbar_wait(pv_done(t), (nb - 1) & 1))) {
      dev::tc_fence_after();
      if constexpr (kOnes) {
        ltot = __uint_as_float(tmem_ld1(ob + D));
        dev::tmem_wait_ld();
      }
      const float inv = 1.f / ltot;
      uint4 *dst = reinterpret_cast<uint4 *>(
          a.out + ((int64_t)(q0 + qi) * a.num_q_heads + g * G + h) * D);
#pragma unroll 1
      for (int ch = hc * (D / 32 / H); ch < (hc + 1) * (D / 32 / H); ++ch) {
        uint32_t o[32];
        dev::tmem_ld32(ob + ch * 32, o);
        dev::tmem_wait_ld();
        if (valid) {
#pragma unroll
          for (int u = 0; u < 4; ++u) {
            uint32_t w4[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w4[e] = dev::pack_bf16x2(__uint_as_float(o[8 * u + 2 * e]) * inv,
                                       __uint_as_float(o[8 * u + 2 * e + 1]) * inv);
            dst[ch * 4 + u] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
          }
        }
      }
    } else if (ok && nb > 0 && lane == 0) {
      fail(false);
    }
  }

  if (tid == 0) (void)dev::mbar_wait(mma_done, 0);
  if ((warp == kProducer || (tc2_producers<D>() == 2 && warp == kProducerV)) && lane == 0 && *s_flag) {
    for (int s = 0; s < KSK; ++s) {
      const int kl = s + ((k_issued - 1 - s) / KSK) * KSK;
      if (kl >= 0 && kl < k_issued) (void)dev::mbar_wait(k_full(s), (kl / KSK) & 1);
    }
    for (int s = 0; s < KSV; ++s) {
      const int vl = s + ((v_issued - 1 - s) / KSV) * KSV;
      if (vl >= 0 && vl < v_issued) (void)dev::mbar_wait(v_full(s), (vl / KSV) & 1);
    }
  }
  dev::tc_fence_before();
  __syncthreads();
  dev::tc_fence_after();
  if (warp == 0) dev::tmem_dealloc(tmem, 512);
}

cudaError_t read_prefill_errors(uint32_t *flags, int clear) { return read_tu_errors(flags, clear); }

constexpr int tc_halves(int d) { return d == 64 ? 1 : PKV_PREFILL_TC_HALVES128; }
constexpr size_t tc_smem(int d) {
  return 1024 + (d == 64 ? TcSmem<64, tc_halves(64)>::total : TcSmem<128, tc_halves(128)>::total);
}
static_assert(tc_smem(64) <= 227 * 1024 && tc_smem(128) <= 227 * 1024, "prefill tile fits a CTA");
// Softmax threads per query row of the two-tile kernel, by head_dim.  At head_dim 128 two
// (16 softmax warps, 96 registers a thread, each half of a row in its own warp) measured
// 1% faster than one.  At 64 one: with P in TMEM two ran 4-5% slower (the kernel is held
// to 96 registers there and spills).
#ifndef PKV_PREFILL_HALVES64
#define PKV_PREFILL_HALVES64 1
#endif
#ifndef PKV_PREFILL_HALVES128
#define PKV_PREFILL_HALVES128 2
#endif
constexpr int tc2_halves(int d) { return d == 64 ? PKV_PREFILL_HALVES64 : PKV_PREFILL_HALVES128; }
constexpr size_t tc2_smem(int d) {
  return 1024 + (d == 64 ? Tc2Smem<64, tc2_halves(64)>::total : Tc2Smem<128, tc2_halves(128)>::total);
}
static_assert(tc2_smem(64) <= 227 * 1024 && tc2_smem(128) <= 227 * 1024,
              "two prefill tiles fit a CTA");

namespace {
bool g_prefill_attr[kMaxDevices][4];  // dynamic smem attribute set: [D 64/128][one/two tiles]
}  // namespace

}  // namespace pkv

using namespace pkv;

PKV_API int paged_prefill_attention(pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                    const pkv_bf16 *v_cache, const int32_t *block_tables,
                                    int32_t max_blocks_per_seq, const int32_t *context_lens,
                                    int32_t max_context_len, const int32_t *query_start,
                                    int32_t max_query_len, int32_t num_seqs, int32_t num_q_heads,
                                    const pkv_cache_desc *cache, float scale, void *stream) {
  int rc = check_decode(q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens,
                        max_context_len, num_seqs, num_q_heads, cache, "paged_prefill_attention");
  if (rc) return rc;
  if (max_query_len < 0 || max_query_len > max_context_len)
    return set_error(PKV_ERR_SHAPE, "paged_prefill_attention: need 0 <= max_query_len <= max_context_len");
  if (num_seqs == 0 || max_query_len == 0) {
    clear_error();
    return PKV_OK;
  }
  if (!out || !query_start) return set_error(PKV_ERR_NULL, "paged_prefill_attention: NULL out/query_start");
  if (!aligned16(out))
    return set_error(PKV_ERR_ALIGN, "paged_prefill_attention: out must be 16-byte aligned");
  const int G = num_q_heads / cache->num_kv_heads;
  // Two 128-row tiles per CTA (prefill_tc2_kernel) when that still makes at least two
  // waves of CTAs; otherwise one tile per CTA (prefill_tc_kernel), e.g. a few long
  // sequences, where halving the CTAs would leave SMs idle.
  const int64_t units = (int64_t)num_seqs * cache->num_kv_heads;
  const int64_t tiles2 = ((int64_t)max_query_len * G + 2 * kTcRows - 1) / (2 * kTcRows);
  int sms = 0;
  {
    std::lock_guard<std::mutex> lk(attn_mutex());
    if ((rc = device_sms(&sms))) return rc;
  }
  const bool two = tiles2 * units >= 2 * (int64_t)sms;
  const int64_t tiles = two ? tiles2 : ((int64_t)max_query_len * G + kTcRows - 1) / kTcRows;
  if (tiles > 0x7fffffffLL) return set_error(PKV_ERR_UNSUPPORTED, "paged_prefill_attention: too many query rows");
  CUtensorMap tmk, tmv;
  const int D = cache->head_dim;
  {
    std::lock_guard<std::mutex> lk(attn_mutex());
    if ((rc = maps_for(k_cache, v_cache, *cache, &tmk, &tmv))) return rc;
    int dev = 0;
    if ((rc = current_device(&dev))) return rc;
    const int vi = (D == 64 ? 0 : 2) + (two ? 1 : 0);
    if (!g_prefill_attr[dev][vi]) {
      cudaError_t e;
      if (two)
        e = D == 64 ? cudaFuncSetAttribute(prefill_tc2_kernel<64, tc2_halves(64)>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)tc2_smem(64))
                    : cudaFuncSetAttribute(prefill_tc2_kernel<128, tc2_halves(128)>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)tc2_smem(128));
      else
        e = D == 64 ? cudaFuncSetAttribute(prefill_tc_kernel<64, tc_halves(64)>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)tc_smem(64))
                    : cudaFuncSetAttribute(prefill_tc_kernel<128, tc_halves(128)>,
                                           cudaFuncAttributeMaxDynamicSharedMemorySize,
                                           (int)tc_smem(128));
      if (e != cudaSuccess) return cuda_error(e, "cudaFuncSetAttribute");
      g_prefill_attr[dev][vi] = true;
    }
  }
  PrefillArgs a;
  a.q = q;
  a.block_tables = block_tables;
  a.context_lens = context_lens;
  a.query_start = query_start;
  a.out = out;
  a.num_blocks = cache->num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.cap = (int32_t)std::min<int64_t>((int64_t)max_blocks_per_seq * cache->block_size, max_context_len);
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = cache->num_kv_heads;
  a.group = G;
  a.block_size = cache->block_size;
  a.log2_bs = ilog2(cache->block_size);
  a.box_rows = cache->block_size < kChunk ? cache->block_size : kChunk;
  a.scale_log2 = scale * kLog2e;
  dim3 grid((unsigned)tiles, (unsigned)cache->num_kv_heads, (unsigned)num_seqs);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (two && D == 64)
    prefill_tc2_kernel<64, tc2_halves(64)><<<grid, tc2_threads<64, tc2_halves(64)>(), tc2_smem(64), s>>>(tmk, tmv, a);
  else if (two)
    prefill_tc2_kernel<128, tc2_halves(128)><<<grid, tc2_threads<128, tc2_halves(128)>(), tc2_smem(128), s>>>(tmk, tmv, a);
  else if (D == 64)
    prefill_tc_kernel<64, tc_halves(64)><<<grid, tc_threads<tc_halves(64)>(), tc_smem(64), s>>>(tmk, tmv, a);
  else
    prefill_tc_kernel<128, tc_halves(128)><<<grid, tc_threads<tc_halves(128)>(), tc_smem(128), s>>>(tmk, tmv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "prefill_tc_kernel launch");
  clear_error();
  return PKV_OK;
}
