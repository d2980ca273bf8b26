// pkv_prefill.cu -- paged prefill attention: causal multi-query attention of each
// sequence's newest tokens over the paged KV cache.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <mutex>

#include "attn_device.cuh"

namespace pkv {

// ===========================================================================
// prefill_kernel: causal attention of each sequence's newest tokens over the paged cache
// ("vLLM-Style Llama Inference Engine", How it works: prefill and recomputation use
// causal attention).  Sequence b holds L_b tokens; its last n_b = query_start[b+1] -
// query_start[b] are the queries; query i sits at position L_b - n_b + i and sees keys
// t <= that position.
//
// One CTA owns one (sequence, kv head, tile of 64 query rows), a row being a (query
// token, head of the group) pair; warp w owns rows 16w .. 16w+15 of the tile and walks
// all keys up to the tile's last position, so every K/V byte staged by the producer is
// used by 64 rows.  Per 64-key stage: S = Q . K^T as mma.sync m16n8k16 (Q: A operand from
// registers; K^T: B operand from the swizzled stage via ldmatrix), online softmax per row
// in fp32 (base 2), O += P . V with P reused from the accumulator registers (as bf16 hi +
// lo) and V through ldmatrix.trans.  Keys past a row's position are masked; V rows past
// the range are zeroed in registers.  The producer warp and TMA ring are the decode
// kernel's.
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

template <int D, int STAGES>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tmk, const __grid_constant__ CUtensorMap tmv,
                   const PrefillArgs a) {
  constexpr int kTileBytes = kChunk * D * 2;
  constexpr int kStageBytes = 2 * kTileBytes;
  constexpr int KS = D / 16;  // k steps over the head dim
  constexpr int DT = D / 8;   // 8-wide output tiles over the head dim

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = dev::smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t *const base_ptr = smem_raw + (base - raw);
  const uint32_t bar_full = base + STAGES * kStageBytes;
  const uint32_t bar_empty = bar_full + STAGES * 8;
  volatile int *const s_flag =
      reinterpret_cast<volatile int *>(base_ptr + STAGES * kStageBytes + STAGES * 16);

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
  const int rows = n * G;                 // query rows of this (b, g)
  const int row0 = tile * 64;
  if (row0 >= rows) return;
  const int last_row = min(row0 + 64, rows) - 1;
  const int t_end = L - n + last_row / G + 1;  // keys the tile needs: [0, t_end)
  const int n_chunks = (t_end + kChunk - 1) / kChunk;

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
    const int rb = a.box_rows;
    const uint32_t box_bytes = (uint32_t)rb * 128u;
    const int lb_last = (t_end - 1) >> a.log2_bs;
    int win = 0;
    int tb = (lane <= lb_last) ? __ldg(trow + lane) : 0;
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
      const int k0 = c * kChunk;
      const int nk = min(kChunk, t_end - k0);
      const int nbox = (nk + rb - 1) / rb;
      const int lb_hi = (k0 + (nbox - 1) * rb) >> a.log2_bs;
      if (lb_hi >= win + 32) {
        win = k0 >> a.log2_bs;
        tb = (win + lane <= lb_last) ? __ldg(trow + win + lane) : 0;
      }
      const int key = k0 + lane * rb;
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
  } else {
    // ----------------------------------------------------------- consumer warps
    const int gid = lane >> 2, tig = lane & 3;
    // this thread's two rows: tile rows 16*warp + gid and + 8
    const int ra = row0 + 16 * warp + gid, rbw = ra + 8;
    const bool va = ra < rows, vb = rbw < rows;
    const int pa = va ? L - n + ra / G : -1, pb = vb ? L - n + rbw / G : -1;  // positions
    const bool warp_live = __any_sync(0xffffffffu, va || vb);
    // Q as the A operand: a0a1 (row a, dims 16ks+2tig..), a2a3 (row b), a4a5 / a6a7: dims + 8
    uint32_t qa[KS][4];
    {
      const uint32_t *qra = reinterpret_cast<const uint32_t *>(
          a.q + ((int64_t)(q0 + (va ? ra / G : 0)) * a.num_q_heads + g * G + (va ? ra % G : 0)) * D);
      const uint32_t *qrb = reinterpret_cast<const uint32_t *>(
          a.q + ((int64_t)(q0 + (vb ? rbw / G : 0)) * a.num_q_heads + g * G + (vb ? rbw % G : 0)) * D);
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qa[ks][0] = va ? __ldg(qra + 8 * ks + tig) : 0u;
        qa[ks][1] = vb ? __ldg(qrb + 8 * ks + tig) : 0u;
        qa[ks][2] = va ? __ldg(qra + 8 * ks + 4 + tig) : 0u;
        qa[ks][3] = vb ? __ldg(qrb + 8 * ks + 4 + tig) : 0u;
      }
    }
    float o[DT][4];
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) o[dt][0] = o[dt][1] = o[dt][2] = o[dt][3] = 0.f;
    float ma = -INFINITY, mb = -INFINITY, la = 0.f, lb = 0.f;
    const int lj = lane >> 3, lr = lane & 7;

    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % STAGES;
      if (!__all_sync(0xffffffffu, dev::mbar_wait(bar_full + 8 * s, (c / STAGES) & 1))) {
        if (lane == 0) {
          raise_error(PKV_DEVERR_TIMEOUT);
          *s_flag = 1;
        }
        break;
      }
      const int k0 = c * kChunk;
      if (warp_live) {
        const uint32_t kb = base + s * kStageBytes, vbase = kb + kTileBytes;
        // S (16 rows x 64 keys) = Q . K^T, eight 8-key n tiles
        float sc[8][4];
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
          for (int m = 0; m < 4; ++m) {  // keys 16m .. 16m+15: n tiles 2m, 2m+1
            uint32_t bk[4];
            dev::ldsm_x4(bk, kb + tile_off(16 * m + lr + ((lj >> 1) << 3), 2 * ks + (lj & 1)));
            dev::mma_bf16_16816(sc[2 * m], qa[ks], bk[0], bk[1]);
            dev::mma_bf16_16816(sc[2 * m + 1], qa[ks], bk[2], bk[3]);
          }
        }
        // causal mask and base-2 scale; row max over the quad
        float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const int key = k0 + 8 * nt + 2 * tig;
          sc[nt][0] = key <= pa ? sc[nt][0] * a.scale_log2 : -INFINITY;
          sc[nt][1] = key + 1 <= pa ? sc[nt][1] * a.scale_log2 : -INFINITY;
          sc[nt][2] = key <= pb ? sc[nt][2] * a.scale_log2 : -INFINITY;
          sc[nt][3] = key + 1 <= pb ? sc[nt][3] * a.scale_log2 : -INFINITY;
          mxa = fmaxf(mxa, fmaxf(sc[nt][0], sc[nt][1]));
          mxb = fmaxf(mxb, fmaxf(sc[nt][2], sc[nt][3]));
        }
#pragma unroll
        for (int x = 1; x < 4; x <<= 1) {
          mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, x));
          mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, x));
        }
        const float mna = fmaxf(ma, mxa), mnb = fmaxf(mb, mxb);
        // a row that has seen no key yet keeps -inf: subtract 0 then (ex2(-inf) = 0, no NaN)
        const float ua = mna == -INFINITY ? 0.f : mna, ub = mnb == -INFINITY ? 0.f : mnb;
        const float ala = dev::ex2(ma - ua), alb = dev::ex2(mb - ub);
        ma = mna;
        mb = mnb;
        la *= ala;
        lb *= alb;
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          o[dt][0] *= ala;
          o[dt][1] *= ala;
          o[dt][2] *= alb;
          o[dt][3] *= alb;
        }
        uint32_t ph[4][4], pl[4][4];  // P as A operands, per 16-key group: hi and residual
#pragma unroll
        for (int nt = 0; nt < 8; ++nt) {
          const float p0 = dev::ex2(sc[nt][0] - ua), p1 = dev::ex2(sc[nt][1] - ua);
          const float p2 = dev::ex2(sc[nt][2] - ub), p3 = dev::ex2(sc[nt][3] - ub);
          la += p0 + p1;
          lb += p2 + p3;
          const uint32_t h01 = dev::pack_bf16x2(p0, p1), h23 = dev::pack_bf16x2(p2, p3);
          const uint32_t r01 = dev::pack_bf16x2(p0 - dev::bf16lo_to_f32(h01), p1 - dev::bf16hi_to_f32(h01));
          const uint32_t r23 = dev::pack_bf16x2(p2 - dev::bf16lo_to_f32(h23), p3 - dev::bf16hi_to_f32(h23));
          const int m = nt >> 1, hi = nt & 1;  // a0a1/a2a3 from the even tile, a4a5/a6a7 odd
          ph[m][2 * hi] = h01;
          ph[m][2 * hi + 1] = h23;
          pl[m][2 * hi] = r01;
          pl[m][2 * hi + 1] = r23;
        }
        // O += P . V; V rows past the range zeroed in registers
        const int nk = t_end - k0;
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          uint32_t mlo = 0xffffffffu, mhi = 0xffffffffu;
          if (nk < 16 * m + 16) {
            const int kk = 16 * m + 2 * tig;
            mlo = (kk < nk ? 0x0000ffffu : 0u) | (kk + 1 < nk ? 0xffff0000u : 0u);
            mhi = (kk + 8 < nk ? 0x0000ffffu : 0u) | (kk + 9 < nk ? 0xffff0000u : 0u);
          }
#pragma unroll
          for (int dt = 0; dt < DT; dt += 2) {
            uint32_t bv[4];  // (keys 0-7, dims dt), (keys 8-15, dims dt), (keys 0-7, dt+1), (8-15, dt+1)
            dev::ldsm_x4_trans(bv, vbase + tile_off(16 * m + lr + ((lj & 1) << 3), dt + (lj >> 1)));
            bv[0] &= mlo;
            bv[1] &= mhi;
            bv[2] &= mlo;
            bv[3] &= mhi;
            dev::mma_bf16_16816(o[dt], ph[m], bv[0], bv[1]);
            dev::mma_bf16_16816(o[dt], pl[m], bv[0], bv[1]);
            dev::mma_bf16_16816(o[dt + 1], ph[m], bv[2], bv[3]);
            dev::mma_bf16_16816(o[dt + 1], pl[m], bv[2], bv[3]);
          }
        }
      }
      __syncwarp();
      if (lane == 0) dev::mbar_arrive(bar_empty + 8 * s);
    }
    // ---- normalise and store this thread's rows
#pragma unroll
    for (int x = 1; x < 4; x <<= 1) {
      la += __shfl_xor_sync(0xffffffffu, la, x);
      lb += __shfl_xor_sync(0xffffffffu, lb, x);
    }
    if (!*s_flag) {
      const float ia = 1.f / la, ib = 1.f / lb;
      uint32_t *oa = reinterpret_cast<uint32_t *>(
          a.out + ((int64_t)(q0 + (va ? ra / G : 0)) * a.num_q_heads + g * G + (va ? ra % G : 0)) * D);
      uint32_t *ob = reinterpret_cast<uint32_t *>(
          a.out + ((int64_t)(q0 + (vb ? rbw / G : 0)) * a.num_q_heads + g * G + (vb ? rbw % G : 0)) * D);
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        if (va) oa[4 * dt + tig] = dev::pack_bf16x2(o[dt][0] * ia, o[dt][1] * ia);
        if (vb) ob[4 * dt + tig] = dev::pack_bf16x2(o[dt][2] * ib, o[dt][3] * ib);
      }
    }
  }

  __syncthreads();
  if (tid == 0 && *s_flag) {
    for (int s = 0; s < STAGES; ++s) {
      const int c_last = s + ((n_chunks - 1 - s) / STAGES) * STAGES;
      if (c_last >= 0 && c_last < n_chunks) (void)dev::mbar_wait(bar_full + 8 * s, (c_last / STAGES) & 1);
    }
  }
}

cudaError_t read_prefill_errors(uint32_t *flags, int clear) { return read_tu_errors(flags, clear); }

namespace {
bool g_prefill_attr[kMaxDevices][2];  // dynamic smem attribute of prefill_kernel set
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
  if (reinterpret_cast<uintptr_t>(out) & 3u)
    return set_error(PKV_ERR_ALIGN, "paged_prefill_attention: out must be 4-byte aligned");
  const int G = num_q_heads / cache->num_kv_heads;
  const int64_t tiles = ((int64_t)max_query_len * G + 63) / 64;
  if (tiles > 0x7fffffffLL) return set_error(PKV_ERR_UNSUPPORTED, "paged_prefill_attention: too many query rows");
  CUtensorMap tmk, tmv;
  const int D = cache->head_dim;
  {
    std::lock_guard<std::mutex> lk(attn_mutex());
    if ((rc = maps_for(k_cache, v_cache, *cache, &tmk, &tmv))) return rc;
    int dev = 0;
    if ((rc = current_device(&dev))) return rc;
    const int vi = D == 64 ? 0 : 1;
    if (!g_prefill_attr[dev][vi]) {
      cudaError_t e = D == 64 ? cudaFuncSetAttribute(prefill_kernel<64, split_stages(64)>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     (int)split_smem(64))
                              : cudaFuncSetAttribute(prefill_kernel<128, split_stages(128)>,
                                                     cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                     (int)split_smem(128));
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
  if (D == 64)
    prefill_kernel<64, split_stages(64)><<<grid, kThreads, split_smem(64), s>>>(tmk, tmv, a);
  else
    prefill_kernel<128, split_stages(128)><<<grid, kThreads, split_smem(128), s>>>(tmk, tmv, a);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return cuda_error(e, "prefill_kernel launch");
  clear_error();
  return PKV_OK;
}
