/*
 * paged_kv.h -- C ABI of the paged-KV decode library (libpkv.so, GB300 / sm_103a).
 *
 * One decode step of a paged KV cache, as the pages describe it:
 *  - "mini-vLLM" LLM-Inference-Engine README, paged KV-cache paragraph: the KV
 *    cache is a fixed pool of physical blocks of block_size token slots; a
 *    per-sequence block table maps logical positions to physical blocks.
 *  - "vLLM-Style Llama Inference Engine with Tensor Parallelism", Features and
 *    scope / How it works: each step writes the new tokens' K/V into the paged
 *    cache through a slot mapping, then one-token decode runs paged attention
 *    with grouped-query heads; split-K decode is named there as the step beyond.
 *  - "llm-stack", Serving engine: the decode query is not causally masked.
 *
 * Conventions shared by every entry point
 *  - bf16 tensors are passed as pointers to their raw 16-bit patterns (pkv_bf16).
 *  - Every pointer is DEVICE memory on the current CUDA device and is owned by
 *    the caller; the library allocates nothing and keeps no pointer after the
 *    call returns.  `stream` is a cudaStream_t (NULL = the legacy default
 *    stream); all work is enqueued asynchronously on it.
 *  - Exception, for paged_kv_write, paged_decode_attention and paged_decode_step:
 *    the per-step inputs and the output -- q, out, k and v (new), slot_mapping,
 *    block_tables, context_lens -- may instead be page-locked host memory that
 *    the device addresses directly (cudaHostAlloc / cudaMallocHost, with unified
 *    addressing the host pointer is the device pointer).  The kernels then read
 *    and write it over the host link: no copy of its own precedes or follows
 *    the call.  Caches and workspace are always device memory.
 *  - Layouts are dense and row-major (C order):
 *      k_cache, v_cache : [num_blocks][num_kv_heads][block_size][head_dim]
 *      q, out           : [num_seqs][num_q_heads][head_dim]
 *      k, v (new)       : [num_tokens][num_kv_heads][head_dim]
 *      slot_mapping     : [num_tokens] int64, slot = block * block_size + offset
 *      block_tables     : [num_seqs][max_blocks_per_seq] int32 physical block ids
 *      context_lens     : [num_seqs] int32, tokens in the cache per sequence
 *                         (including any token written this step)
 *    Query head h reads kv head h / (num_q_heads / num_kv_heads).
 *  - Return value: PKV_OK (0) or a negative PKV_ERR_* code.  Argument errors are
 *    found on the host before anything is enqueued; pkv_last_error() then holds
 *    a message for the calling thread.  Bad device-side values (a block id out of
 *    range, a slot past the pool, a context length over the table's capacity)
 *    never cause an out-of-bounds access: the kernels skip or clamp them and
 *    raise a bit in a per-device error word, read with pkv_device_errors().
 */
#ifndef PAGED_KV_H
#define PAGED_KV_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t pkv_bf16; /* raw bfloat16 bits */

/* Shape of the paged KV pool. */
typedef struct pkv_cache_desc {
  int64_t num_blocks;   /* physical blocks in the pool (> 0) */
  int32_t block_size;   /* token slots per block: a power of two, 8 .. 256 */
  int32_t num_kv_heads; /* kv heads (> 0) */
  int32_t head_dim;     /* elements per head: 64 or 128 for attention; any multiple of 8 for the write */
} pkv_cache_desc;

enum {
  PKV_OK = 0,
  PKV_ERR_NULL = -1,        /* a required pointer is NULL */
  PKV_ERR_SHAPE = -2,       /* inconsistent or out-of-range sizes */
  PKV_ERR_UNSUPPORTED = -3, /* valid but not built: head_dim, block_size or group size */
  PKV_ERR_WORKSPACE = -4,   /* workspace missing or smaller than required */
  PKV_ERR_ALIGN = -5,       /* a pointer is not 16-byte aligned */
  PKV_ERR_CUDA = -6,        /* a CUDA runtime call or launch failed */
  PKV_ERR_DEVICE = -7,      /* pkv_device_errors() found a device-side error bit */
  PKV_ERR_NOSPACE = -8      /* the block pool has too few free blocks (block manager) */
};

/* Device error bits reported by pkv_device_errors(). */
enum {
  PKV_DEVERR_BLOCK_ID = 1,     /* a block table entry outside [0, num_blocks): read as block 0 */
  PKV_DEVERR_SLOT = 2,         /* a slot >= num_blocks * block_size: that token was skipped */
  PKV_DEVERR_CONTEXT_LEN = 4,  /* context_len < 0 or over the table/max_context_len: clamped */
  PKV_DEVERR_TIMEOUT = 8,      /* a pipeline wait gave up (should never happen): output invalid */
  PKV_DEVERR_POSITION = 16     /* a RoPE position outside [0, max_position): that row skipped */
};

/*
 * paged_kv_write -- the slot-mapping write ("vLLM-Style Llama Inference Engine",
 * Features and scope: slot mappings; "mini-vLLM" README: the per-sequence K/V
 * write into the block pool that page names as overhead).
 *
 * For every token i < num_tokens and kv head h, if slot_mapping[i] >= 0:
 *   k_cache[slot / BS][h][slot % BS][:] = k[i][h][:]   (bit copy; v alike).
 * Negative slots are padding and are skipped.  Two tokens with the same slot in
 * one call leave either one's value (undefined which).  head_dim must be a
 * multiple of 8 (16-byte rows); k, v, k_cache and v_cache 16-byte aligned.
 * num_tokens == 0 is a no-op.
 */
int paged_kv_write(const pkv_bf16 *k, const pkv_bf16 *v, const int64_t *slot_mapping,
                   int64_t num_tokens, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                   const pkv_cache_desc *cache, void *stream);

/*
 * paged_kv_write_rope -- the slot-mapping write with rotary position embedding fused
 * in ("llm-stack", Serving engine: RoPE is applied at absolute positions before keys
 * enter the cache; "Building ... with tiny-vLLM", CUDA kernel engineering: RoPE
 * rotates coordinate pairs by sine/cosine of position-dependent angles).
 *
 * For token i at position p = positions[i] (0 <= p < max_position), each head row x
 * of k[i] (and of q[i] when q != NULL, in place) is rotated pairwise:
 *   neox_style != 0: pairs (e, e + r/2), e < r/2 ("rotate half");
 *   neox_style == 0: pairs (2e, 2e + 1)   (interleaved);
 *   x1' = x1 * cos_sin[p][e] - x2 * cos_sin[p][r/2 + e],
 *   x2' = x2 * cos_sin[p][e] + x1 * cos_sin[p][r/2 + e],
 * in fp32 with every product and sum rounded once (no fused multiply-add), then
 * rounded to bf16 (nearest even); coordinates at or past r = rotary_dim are copied.
 * Then k' and v are written like paged_kv_write.  cos_sin is DEVICE fp32
 * [max_position][rotary_dim] (cosines first, then sines), made by the caller (e.g.
 * angle(p, e) = p * base^(-2e/r)).  q is [num_tokens][num_q_heads][head_dim].
 * rotary_dim: a positive multiple of 16, <= head_dim.  A position out of range
 * skips that token's rows and raises PKV_DEVERR_POSITION.
 */
int paged_kv_write_rope(const pkv_bf16 *k, const pkv_bf16 *v, pkv_bf16 *q, int32_t num_q_heads,
                        const int64_t *slot_mapping, const int64_t *positions,
                        int64_t num_tokens, const float *cos_sin, int64_t max_position,
                        int32_t rotary_dim, int32_t neox_style, pkv_bf16 *k_cache,
                        pkv_bf16 *v_cache, const pkv_cache_desc *cache, void *stream);

/*
 * paged_decode_plan -- the launcher's split choice ("vLLM-Style Llama Inference
 * Engine", Features and scope, where split-K decode is the named next step).
 *
 * Returns the partition size P in tokens (a multiple of 64) that
 * paged_decode_attention cuts each (sequence, kv head) into.  With few (sequence,
 * kv head) units, one CTA streams one partition and P is chosen so that the
 * partitions make about one wave of CTAs on this GPU.  With many units (at least
 * a wave of CTAs), a persistent wave of CTAs streams the partitions as work items,
 * longest first, and P = 1536 (1024 for batches over 1024 sequences).  Batches
 * over 1024 sequences, or with contexts over 39 * 1536 = 59904 tokens, take one CTA
 * per partition instead.  P is never below min(max_context_len, 512) rounded up to 64,
 * so short contexts stay whole.  0 for empty or unsupported sizes.  num_sms <= 0
 * queries the current device.  Pure host function.
 */
int32_t paged_decode_plan(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t max_context_len, int32_t num_sms);

/*
 * paged_decode_path -- which kernel arrangement paged_decode_attention (and
 * paged_decode_step) launches for these sizes on the current device:
 *   PKV_PATH_PARTITIONS: one CTA per partition; a sequence cut into several
 *     partitions is merged by the last of them to finish (through global memory);
 *   PKV_PATH_CLUSTER: few units with 2..8 partitions each: the partitions of one
 *     (sequence, kv head) form a thread-block cluster and merge through distributed
 *     shared memory;
 *   PKV_PATH_PERSISTENT: many units (at least a wave of CTAs), at most 1024
 *     sequences, contexts up to 59904 tokens: a persistent wave of CTAs streams the
 *     partitions as work items, longest first, with the merges of multi-partition
 *     sequences kept away from the end.
 * 0 for empty or unsupported sizes.  num_sms <= 0 queries the current device.  Pure
 * host function.
 */
enum { PKV_PATH_PARTITIONS = 1, PKV_PATH_CLUSTER = 2, PKV_PATH_PERSISTENT = 3 };
int32_t paged_decode_path(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t max_context_len, int32_t num_sms);

/*
 * pkv_set_decode_consumer -- the arithmetic of the consumer warps of the partition
 * decode kernel, process-wide (every later launch on any stream or device).  Both
 * forms take bf16 inputs and accumulate exact bf16 products in fp32 ("llm-stack",
 * Attention kernel); they differ only in the units that do it:
 *   PKV_CONSUMER_TENSOR (default): the group's scores and P.V as mma.sync tiles
 *     (16 keys x 8 heads), P entering P.V as a bf16 hi + lo pair;
 *   PKV_CONSUMER_FMA: fp32 FMAs on the CUDA cores (mixed bf16 x bf16 + fp32 FMAs for
 *     the scores, P in fp32 for P.V), with warp shuffles to combine and spread values.
 * It applies to the PKV_PATH_PARTITIONS and PKV_PATH_CLUSTER arrangements and to
 * paged_decode_split; the persistent arrangement always uses the tensor form.  The
 * CUDA-core form is kept so that the two can be measured against each other on the
 * same shapes; the default is the tensor form.  Returns the previous form, or
 * PKV_ERR_UNSUPPORTED for an unknown one.  Host function; not synchronised with
 * launches already queued.
 */
enum { PKV_CONSUMER_TENSOR = 0, PKV_CONSUMER_FMA = 1 };
int32_t pkv_set_decode_consumer(int32_t consumer);

/*
 * pkv_decode_ctas_per_sm -- how many CTAs of the decode kernel that `path` (PKV_PATH_*)
 * launches for this head_dim fit on one SM of the current device, as the CUDA runtime
 * computes it from the kernel's registers, threads and shared memory (the consumer form
 * set by pkv_set_decode_consumer for the partition arrangements).  paged_decode_plan
 * sizes its grids for 3 at head_dim 64 and 2 at 128; a build whose kernels no longer
 * fit that many would run a second wave.  Returns the count, or PKV_ERR_UNSUPPORTED /
 * PKV_ERR_CUDA.  Host function; sets the kernel's shared-memory attribute as a launch
 * would.
 */
int32_t pkv_decode_ctas_per_sm(int32_t head_dim, int32_t path);

/*
 * paged_decode_workspace_size -- bytes of workspace paged_decode_attention needs for
 * these sizes on the current device: a completion counter per (sequence, kv head),
 * then the partition results of paged_decode_split's layout for P =
 * paged_decode_plan(...).  0 for empty sizes.
 */
size_t paged_decode_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                                   int32_t head_dim, int32_t max_context_len);

/* Bytes of o_part + lse_part (padded to 256 B) of paged_decode_split for a partition size. */
size_t paged_decode_split_workspace_size(int32_t num_seqs, int32_t num_q_heads, int32_t head_dim,
                                         int32_t max_context_len, int32_t partition_tokens);

/*
 * paged_decode_attention -- single-token GQA decode attention over the paged
 * cache ("vLLM-Style Llama Inference Engine", How it works: one-token decode uses
 * a custom paged attention; "mini-vLLM" README, M4 test row: it must match dense
 * attention on scattered blocks).
 *
 * For each sequence b and query head h (g = h / (num_q_heads/num_kv_heads)):
 *   L = context_lens[b];  for t < L:  K_t = k_cache[block_tables[b][t/BS]][g][t%BS]
 *   s_t = scale * <q[b][h], K_t>;  p = softmax(s);  out[b][h] = bf16(sum_t p_t V_t)
 * in fp32 arithmetic on bf16 inputs, rounded to bf16 (nearest even).  No causal
 * mask.  L == 0 gives zeros.  Table entries at or past ceil(L / BS) are not read.
 * max_context_len must be >= every context_lens[b] (it sizes the grid and the
 * workspace without a device-to-host read) and <= max_blocks_per_seq * BS.
 *
 * Supported: head_dim 64 or 128; block_size a power of two in [8, 256];
 * num_q_heads / num_kv_heads (the group) from 1 to 8.  q, k_cache, v_cache and
 * workspace 16-byte aligned; out 8-byte aligned.
 *
 * One kernel launch (see paged_decode_plan): a sequence that fits one partition is
 * written directly; otherwise each partition stores its result in the workspace and
 * the last partition of that (sequence, kv head) to finish merges them (an atomic
 * ticket; no CTA waits for another).
 * `workspace` must hold paged_decode_workspace_size() bytes and must be ZERO-FILLED
 * before its first use (it holds completion counters); every call that completes
 * leaves it ready for the next one.  Calls that share a workspace must not overlap
 * on the GPU.
 */
int paged_decode_attention(pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                           const pkv_bf16 *v_cache, const int32_t *block_tables,
                           int32_t max_blocks_per_seq, const int32_t *context_lens,
                           int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                           const pkv_cache_desc *cache, float scale, void *workspace,
                           size_t workspace_bytes, void *stream);

/*
 * paged_decode_step -- one whole decode step: paged_kv_write(k, v, slot_mapping,
 * num_tokens, ...) into the caches, then paged_decode_attention over the updated
 * caches ("vLLM-Style Llama Inference Engine", How it works: each rank writes its
 * new K/V into the paged cache, then one-token decode runs paged attention).
 *
 * Arguments, layouts, workspace rules and results are those of the two calls; both
 * are checked before either is enqueued.  The attention kernel is launched as a
 * programmatic dependent of the write kernel: its set-up (reading q, context_lens
 * and block_tables) overlaps the write, and it reads the caches only after the
 * write's stores are visible.
 */
int paged_decode_step(pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                      const int64_t *slot_mapping, int64_t num_tokens, pkv_bf16 *k_cache,
                      pkv_bf16 *v_cache, const int32_t *block_tables, int32_t max_blocks_per_seq,
                      const int32_t *context_lens, int32_t max_context_len, int32_t num_seqs,
                      int32_t num_q_heads, const pkv_cache_desc *cache, float scale,
                      void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_decode_step_rope -- one whole decode step with rotary position embedding, as
 * a model's attention layer runs it ("llm-stack", Serving engine: keys are rotated at
 * their absolute positions before they enter the cache; "vLLM-Style Llama Inference
 * Engine", How it works: write the new K/V into the paged cache, then one-token
 * paged attention):
 *   1. paged_kv_write_rope(k, v, q, num_q_heads, slot_mapping, positions, num_seqs,
 *      cos_sin, max_position, rotary_dim, neox_style, k_cache, v_cache, cache):
 *      q [num_seqs][num_q_heads][head_dim] is rotated IN PLACE, k is rotated and
 *      written with v at slot_mapping[b];
 *   2. paged_decode_attention over the updated caches with the rotated q.
 * Token b is sequence b's new token (one per sequence; positions[b] is normally
 * context_lens[b] - 1).  Arguments, layouts, workspace rules and results are those of
 * the two calls; both are checked before either is enqueued.  The attention kernel is
 * a programmatic dependent of the rotary write: its set-up overlaps the write, and it
 * reads q and the caches only after the write's stores are visible.
 */
int paged_decode_step_rope(pkv_bf16 *out, pkv_bf16 *q, const pkv_bf16 *k, const pkv_bf16 *v,
                           const int64_t *slot_mapping, const int64_t *positions,
                           const float *cos_sin, int64_t max_position, int32_t rotary_dim,
                           int32_t neox_style, pkv_bf16 *k_cache, pkv_bf16 *v_cache,
                           const int32_t *block_tables, int32_t max_blocks_per_seq,
                           const int32_t *context_lens, int32_t max_context_len,
                           int32_t num_seqs, int32_t num_q_heads, const pkv_cache_desc *cache,
                           float scale, void *workspace, size_t workspace_bytes, void *stream);

/*
 * paged_prefill_attention -- causal attention of each sequence's newest tokens over
 * the paged cache: prefill, chunked prefill, or recomputation after preemption
 * ("vLLM-Style Llama Inference Engine", How it works: prefill and recomputation use
 * causal attention).
 *
 * Sequence b holds L_b = context_lens[b] tokens in the cache (their K/V already
 * written, e.g. by paged_kv_write); its last n_b = query_start[b+1] - query_start[b]
 * tokens are the queries, packed in q [num_queries][num_q_heads][head_dim] at rows
 * query_start[b] .. query_start[b+1]-1 (query_start is DEVICE int32 [num_seqs + 1],
 * nondecreasing).  Query i of sequence b sits at position p = L_b - n_b + i and
 *   out[row][h] = bf16( sum_{t <= p} softmax_t(scale * <q[row][h], K_t>) V_t )
 * with K_t, V_t read through block_tables as in paged_decode_attention (same head
 * mapping, sizes and alignment rules; out is 16-byte aligned).  max_query_len >= every
 * n_b sizes the grid; a sequence with more queries raises PKV_DEVERR_CONTEXT_LEN and
 * its rows past max_query_len are not written.  Every out row of a query is written;
 * nothing else.
 */
int paged_prefill_attention(pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                            const pkv_bf16 *v_cache, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *context_lens,
                            int32_t max_context_len, const int32_t *query_start,
                            int32_t max_query_len, int32_t num_seqs, int32_t num_q_heads,
                            const pkv_cache_desc *cache, float scale, void *stream);

/*
 * paged_decode_split -- flash-decoding partition kernel (split-K over the keys;
 * the FlashAttention-2 online-softmax algebra that the first page references).
 *
 * Partition r of sequence b covers tokens [r*P, min((r+1)*P, L)) with
 * P = partition_tokens (a positive multiple of 64).  For each (b, h, r) with a
 * non-empty range it writes
 *   o_part  [num_seqs][num_q_heads][n_parts][head_dim] fp32 : the range's
 *                                  softmax-normalised output sum_t p_t V_t,
 *   lse_part[num_seqs][num_q_heads][n_parts]           fp32 : ln sum_t exp(s_t),
 * where n_parts = ceil(max_context_len / P).  Entries of empty ranges
 * (r*P >= L) are not written.  Same preconditions as paged_decode_attention.
 */
int paged_decode_split(float *o_part, float *lse_part, const pkv_bf16 *q,
                       const pkv_bf16 *k_cache, const pkv_bf16 *v_cache,
                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                       const int32_t *context_lens, int32_t max_context_len, int32_t num_seqs,
                       int32_t num_q_heads, const pkv_cache_desc *cache, float scale,
                       int32_t partition_tokens, void *stream);

/*
 * paged_decode_combine -- log-sum-exp merge of the partitions written by
 * paged_decode_split (same layouts, same partition_tokens and max_context_len):
 *   M = max_r lse_r,  w_r = exp(lse_r - M),  out = bf16(sum_r w_r o_r / sum_r w_r)
 * over the ceil(L / P) non-empty ranges of each sequence; L == 0 gives zeros.
 */
int paged_decode_combine(pkv_bf16 *out, const float *o_part, const float *lse_part,
                         const int32_t *context_lens, int32_t max_context_len, int32_t num_seqs,
                         int32_t num_q_heads, int32_t head_dim, int32_t partition_tokens,
                         void *stream);

/*
 * paged_decode_attention_noalloc -- paged_decode_attention for callers that cannot
 * allocate device memory.  (No counterpart in the paper: this is a library service.)
 *
 * Who needs it: code that may not call cudaMalloc or any allocator -- a host
 * application or plugin framework that owns all device memory and gives out none,
 * a latency-critical loop where an allocation (which can synchronise the device and
 * take unbounded time) is not allowed, or a caller with no allocator of its own.
 * Such callers cannot pass the workspace that paged_decode_attention needs when it
 * splits long contexts.
 *
 * Same arguments and result as paged_decode_attention, without the workspace: the
 * partition workspace lives in a fixed array of PKV_NOALLOC_SCRATCH_BYTES compiled
 * into the library (every GPU that loads the library holds it until the process
 * exits).  The call allocates nothing.
 *  - Sizes whose plan needs more than PKV_NOALLOC_SCRATCH_BYTES of workspace
 *    (paged_decode_workspace_size) are rejected with PKV_ERR_WORKSPACE and a message;
 *    use paged_decode_attention with your own workspace for those.
 *  - Every argument check of paged_decode_attention runs first: a refused call
 *    returns its PKV_ERR_* code with nothing enqueued and the array untouched.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) and caches it; make that first call outside any CUDA
 *    stream capture.
 *  - All calls share the one array, which keeps whatever the previous call left in
 *    it.  The part that must start at zero (the completion counters) is cleared by
 *    each call on its stream before the kernel runs.  Calls that overlap on the GPU
 *    (on different streams, or from different threads without ordering) race on
 *    the array and give wrong results: order them on one stream.
 */
#define PKV_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)
int paged_decode_attention_noalloc(pkv_bf16 *out, const pkv_bf16 *q, const pkv_bf16 *k_cache,
                                   const pkv_bf16 *v_cache, const int32_t *block_tables,
                                   int32_t max_blocks_per_seq, const int32_t *context_lens,
                                   int32_t max_context_len, int32_t num_seqs, int32_t num_q_heads,
                                   const pkv_cache_desc *cache, float scale, void *stream);

/*
 * Block manager -- the host-side allocator that produces block tables and slot
 * mappings ("mini-vLLM" README, architecture diagram and M4 row: a Block Manager
 * allocates physical blocks and keeps per-sequence block tables, with LIFO preemption
 * under memory pressure; "vLLM-Style Llama Inference Engine", How it works: the
 * scheduler allocates blocks and finished requests release them).  HOST memory and
 * host code only; thread-safe.  Blocks are handed out from a LIFO free list (block 0
 * first on a fresh pool); a sequence of L tokens owns ceil(L / block_size) blocks.
 * Functions return PKV_OK or a negative PKV_ERR_* code (PKV_ERR_NOSPACE when the pool
 * cannot satisfy a request; nothing changes then).
 */
typedef struct pkv_block_manager pkv_block_manager;

/* A pool of num_blocks blocks of block_size slots; NULL on bad sizes (see pkv_last_error). */
pkv_block_manager *pkv_bm_create(int64_t num_blocks, int32_t block_size);
void pkv_bm_destroy(pkv_block_manager *m);
/* Free blocks now (>= 0), or a negative error code. */
int64_t pkv_bm_num_free_blocks(pkv_block_manager *m);
/* Admit sequence seq_id holding num_tokens tokens (e.g. a prompt): allocates its blocks. */
int pkv_bm_add_sequence(pkv_block_manager *m, int64_t seq_id, int64_t num_tokens);
/* Append one token to each listed sequence (a sequence may appear several times): writes
 * the token's slot (block * block_size + offset) to slot_mapping[i], allocating a block
 * when a sequence's last block is full.  All or nothing. */
int pkv_bm_append_slots(pkv_block_manager *m, const int64_t *seq_ids, int32_t n,
                        int64_t *slot_mapping);
/* A finished sequence releases its blocks. */
int pkv_bm_free_sequence(pkv_block_manager *m, int64_t seq_id);
/* Preempt the most recently admitted sequence (LIFO): release its blocks, report its id. */
int pkv_bm_preempt_lifo(pkv_block_manager *m, int64_t *seq_id);
/* Block tables [n][max_blocks_per_seq] (unused entries -1) and context lengths [n] of the
 * listed sequences, ready to copy to the device for paged_decode_attention. */
int pkv_bm_block_tables(pkv_block_manager *m, const int64_t *seq_ids, int32_t n,
                        int32_t max_blocks_per_seq, int32_t *block_tables,
                        int32_t *context_lens);

/*
 * pkv_device_errors -- synchronises the current device, then ORs the device error
 * words of every kernel family into *flags (PKV_DEVERR_* bits; 0 = none seen since
 * the last clear).  clear != 0 resets them.  Returns PKV_OK, or PKV_ERR_CUDA if
 * the synchronisation or copy failed.  `flags` is HOST memory.
 */
int pkv_device_errors(uint32_t *flags, int clear);

/* Message for the last error returned on the calling thread ("" if none). */
const char *pkv_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* PAGED_KV_H */
