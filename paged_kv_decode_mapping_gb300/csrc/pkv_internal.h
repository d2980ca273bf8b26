// pkv_internal.h -- helpers shared by the library's translation units (not installed).
#pragma once

#include <cuda.h>  // CUtensorMap (header only)
#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "paged_kv.h"

#define PKV_API extern "C" __attribute__((visibility("default")))

namespace pkv {

// Records a message for pkv_last_error() on this thread and returns `code`.
int set_error(int code, const char *fmt, ...) __attribute__((format(printf, 2, 3)));
// Clears this thread's message (called on every successful entry).
void clear_error();
// Turns a failed CUDA call into PKV_ERR_CUDA with its name and message.
int cuda_error(cudaError_t e, const char *what);

// Device error word of the write kernel's translation unit (read + optional clear).
cudaError_t read_write_errors(uint32_t *flags, int clear);

// The slot-mapping write, split into its host checks and its launch.
int check_write(const void *k, const void *v, const int64_t *slot_mapping, int64_t num_tokens,
                const void *k_cache, const void *v_cache, const pkv_cache_desc *cache);
int launch_write(const pkv_bf16 *k, const pkv_bf16 *v, const int64_t *slot_mapping,
                 int64_t num_tokens, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                 const pkv_cache_desc &c, cudaStream_t stream);

// The slot write with rotary embedding, split the same way.
int check_write_rope(const void *k, const void *v, const void *q, int32_t num_q_heads,
                     const int64_t *slot_mapping, const int64_t *positions, int64_t num_tokens,
                     const float *cos_sin, int64_t max_position, int32_t rotary_dim,
                     const void *k_cache, const void *v_cache, const pkv_cache_desc *cache);
int launch_write_rope(const pkv_bf16 *k, const pkv_bf16 *v, pkv_bf16 *q, int32_t num_q_heads,
                      const int64_t *slot_mapping, const int64_t *positions, int64_t num_tokens,
                      const float *cos_sin, int64_t max_position, int32_t rotary_dim,
                      int32_t neox_style, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                      const pkv_cache_desc &c, cudaStream_t stream);

inline bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---- shared by the attention kernels (decode and prefill) ----------------------
constexpr int kChunk = 64;          // keys per pipeline stage
constexpr int kConsumerWarps = 4;   // 16 keys each
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;
constexpr int kMaxGroup = 8;        // query heads per kv head (one mma N tile)
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kMaxDevices = 64;

// Partitions one cluster merges (portable cluster size), and the slots of the area in
// which a decode CTA receives its peers' results for the heads it merges: slot
// u * ceil(G / n) + j holds source rank u's result for the CTA's j-th head, and
// n * ceil(G / n) <= 14 for every cluster size n in [2, 8] and group G <= 8.
constexpr int kMaxClusterParts = 8;
constexpr int kRecvSlots = 16;

// Stages of the TMA ring and the dynamic shared memory of one decode CTA: 1 KB of
// alignment slack, the ring, its full/empty barriers, two flags and the merge barrier,
// the receive area (kRecvSlots rows of D floats, then kRecvSlots lse values), then the
// group's query rows as bf16 (read there by the CUDA-core form of the consumer warps).
constexpr int split_stages(int d) { return d == 64 ? 4 : 3; }
constexpr size_t split_ring_bytes(int d) { return (size_t)split_stages(d) * 2 * kChunk * d * 2; }
constexpr size_t split_smem(int d) {
  return 1024 + split_ring_bytes(d) + split_stages(d) * 16 + 16 + (size_t)kRecvSlots * (d + 1) * 4 +
         (size_t)kMaxGroup * d * 2;
}
// CTAs of decode_kernel one SM holds (shared memory limited: 70 KB at D=64, 105 KB at
// D=128, of the 228 KB an SM shares out with 1 KB reserved per CTA).
constexpr int split_occupancy(int d) { return d == 64 ? 3 : 2; }
static_assert(3 * (split_smem(64) + 1024) <= 228 * 1024 && 2 * (split_smem(128) + 1024) <= 228 * 1024,
              "decode CTAs per SM");

// Guards the tensor-map cache, the SM-count cache and the per-device kernel attributes.
std::mutex &attn_mutex();
// The current device (0 .. kMaxDevices-1), or a PKV_ERR_CUDA code.
int current_device(int *dev);
// SM count of the current device (cached); the caller holds attn_mutex().
int device_sms(int *sms);
// Encoded TMA maps of the two pools (cached by pointer and shape); the caller holds
// attn_mutex().
int maps_for(const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const pkv_cache_desc &c,
             CUtensorMap *tmk, CUtensorMap *tmv);
// Argument checks shared by the decode and prefill entry points.
int check_decode(const void *q, const void *k_cache, const void *v_cache, const int32_t *bt,
                 int32_t max_blocks, const int32_t *lens, int32_t max_len, int32_t num_seqs,
                 int32_t hq, const pkv_cache_desc *c, const char *fn);
int ilog2(int x);  // smallest r with 2^r >= x
// Every host check paged_decode_attention makes (shape, pointers, alignment, the
// planned workspace against `workspace_bytes`), without enqueuing anything, for a caller
// whose workspace is a fixed, 256-byte aligned buffer of `workspace_bytes`; `fn` names
// the caller in the error message.
int check_decode_attention(const pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                           const pkv_bf16 *v_cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                           const pkv_cache_desc *cache, size_t workspace_bytes, const char *fn);

// Device error words of the attention translation units (read + optional clear).
cudaError_t read_decode_errors(uint32_t *flags, int clear);
cudaError_t read_prefill_errors(uint32_t *flags, int clear);

}  // namespace pkv

// ----------------------------------------------------------------------------
// Device-side inline PTX wrappers (sm_90+ forms, built for sm_103a).
#ifdef __CUDACC__
namespace pkv {
namespace dev {

__device__ __forceinline__ uint32_t smem_addr(const void *p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(bar), "r"(parity)
      : "memory");
  return done != 0;
}

// Waits for the phase with the given parity to complete, for at most ~2 s of
// wall time.  Returns false on timeout (the caller records an error and unwinds).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 0 && globaltimer_ns() - t0 > 2000000000ull) return false;
  }
}

// L2 policy: streamed once, evict first.
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// L2 policy: read again soon (by other CTAs), evict last.
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}

// 2-D tiled TMA load of one box into shared memory, completing on `bar`.
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, int32_t x, int32_t y,
                                            uint32_t bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      ".L2::cache_hint [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_trans(uint32_t (&r)[4], uint32_t addr) {
  asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(addr));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col)
__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], uint32_t b0,
                                               uint32_t b1) {
  asm volatile(
      "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, "
      "{%8, %9}, {%0, %1, %2, %3};"
      : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
      : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Transposes an 8x8 b16 matrix held one row-pair per lane (ldmatrix fragment layout).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t x) {
  uint32_t y;
  asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(y) : "r"(x));
  return y;
}

// Hardware base-2 exponential (MUFU.EX2); ex2(-inf) = +0.
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Packs two floats into bf16x2 (round to nearest even): `lo` in bits 0..15.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}

__device__ __forceinline__ float bf16lo_to_f32(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t x) { return __uint_as_float(x & 0xFFFF0000u); }

// Atomic add with acquire-release semantics at GPU scope; returns the old value.
__device__ __forceinline__ uint32_t atomic_add_acq_rel(uint32_t *p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Plain bulk copy of `bytes` (a multiple of 16; both addresses 16-byte aligned) from
// global into shared memory, completing on `bar`.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void *src, uint32_t bytes,
                                          uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

// ---- thread-block clusters: rank, barrier, distributed shared memory stores
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
__device__ __forceinline__ uint32_t cluster_nctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
  return r;
}
// The shared::cluster address of `addr` (a shared::cta address) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
  return r;
}
// The cluster barrier in two halves: arrive without waiting (relaxed: a preceding
// fence.mbarrier_init supplies the release of barrier initialisation), wait later.
__device__ __forceinline__ void cluster_arrive_relaxed() {
  asm volatile("barrier.cluster.arrive.relaxed;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait() {
  asm volatile("barrier.cluster.wait.acquire;" ::: "memory");
}
// Stores v at shared::cluster address `addr` (in another CTA of the cluster, or this
// one) and, once written, counts its 4 bytes off the transaction count of the mbarrier
// at shared::cluster address `bar` in the same CTA (complete_tx releases at cluster
// scope).  The sender needs nothing to stay alive: the value leaves from a register.
__device__ __forceinline__ void st_async(uint32_t addr, float v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
               ::"r"(addr), "f"(v), "r"(bar)
               : "memory");
}
// The same for two floats at an 8-byte aligned `addr` (8 bytes counted).
__device__ __forceinline__ void st_async_v2(uint32_t addr, float v0, float v1, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v2.f32 [%0], {%1, %2}, [%3];"
               ::"r"(addr), "f"(v0), "f"(v1), "r"(bar)
               : "memory");
}
// mbar_wait with acquire at cluster scope: what other CTAs of the cluster wrote to this
// CTA's shared memory before completing the phase is visible after it returns true.
// Same ~2 s limit.
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity) {
  const uint64_t t0 = globaltimer_ns();
  for (uint32_t i = 0;; ++i) {
    uint32_t done;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(done)
        : "r"(bar), "r"(parity)
        : "memory");
    if (done) return true;
    if ((i & 255u) == 255u && globaltimer_ns() - t0 > 2000000000ull) return false;
  }
}

// ---- 5th-generation tensor cores: TMEM, tcgen05.mma, shared-memory matrix descriptors
// Allocate `ncols` TMEM columns (a power of two >= 32); the base address is written to
// shared memory at `slot`.  One whole warp executes it; the same warp frees them.
__device__ __forceinline__ void tmem_alloc(uint32_t slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Generic-proxy shared-memory writes become visible to the async proxy (TMA, tensor cores).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Shared-memory matrix descriptor: 128-byte swizzle, start / leading / stride byte offsets.
// K-major operand: rows of 64 bf16 (128 B), 8-row groups `sbo` apart (lbo unused).
// MN-major operand: `lbo` between 64-element blocks along M/N, `sbo` between 8-row K groups.
__device__ __forceinline__ uint64_t smem_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// Instruction descriptor, kind::f16: bf16 A and B, fp32 accumulator, A K-major, B K-major
// (b_mn = 0) or MN-major (b_mn = 1), M x N.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)b_mn << 16) | ((uint32_t)(N >> 3) << 17) |
         ((uint32_t)(M >> 4) << 24);
}
// D[tmem] (+)= A[smem] . B[smem]; issued by one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                          uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05.mma this thread issued before has completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
// 32 consecutive 32-bit TMEM columns of this thread's lane (warp w of a warpgroup owns
// lanes 32(w%4) .. +31; `taddr` carries that lane base).  Complete with tmem_wait_ld.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
        "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
        "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, "
      "%12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, "
      "%30, %31, %32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]),
      "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]),
      "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]),
      "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_ld() {
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_wait_st() {
  asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace dev
}  // namespace pkv
#endif
