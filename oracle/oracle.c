/*
 * oracle.c -- TEST INFRASTRUCTURE ONLY.  A plain, slow, obviously correct CPU
 * definition of paged-KV decode, in fp64.  Only the tests, the smoke check and
 * the benchmark's CPU-baseline leg may load it; the library never does.  It
 * shares no code, header, table or helper with the CUDA path.
 *
 * What it follows:
 *  - "mini-vLLM" LLM-Inference-Engine README, paged KV-cache paragraph: a fixed
 *    pool of physical blocks of block_size token slots, and a per-sequence block
 *    table that maps logical positions to physical storage.  Hence the gather:
 *    logical position t of sequence b lives in physical block
 *    block_tables[b][t / block_size] at slot t % block_size.
 *  - "vLLM-Style Llama Inference Engine with Tensor Parallelism", Features and
 *    scope: paged KV caching with block tables and slot mappings, grouped-query
 *    attention, one-token decode.  Hence the slot-mapping write and the GQA map.
 *  - "llm-stack", Serving engine (KV cache bullet): the single decode query is
 *    NOT causally masked -- it attends to every cached key.
 *  - "llm-stack", Attention kernel: bf16 inputs; here every product and sum is
 *    taken in fp64 instead, so the oracle is the exact definition up to fp64
 *    rounding.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *  - cache layout [num_blocks][num_kv_heads][block_size][head_dim], bf16;
 *  - slot = physical_block * block_size + offset; negative slots are skipped;
 *  - query head h reads kv head h / (num_q_heads / num_kv_heads);
 *  - scores s_t = scale * <q, k_t>, softmax over all t < context_len, output
 *    sum_t p_t v_t; context_len == 0 gives a zero output;
 *  - a split into token ranges (flash-decoding) reports, per range, the range's
 *    normalised output and its log-sum-exp; ranges merge with weights
 *    exp(lse_r - max lse) (FlashAttention-2 online-softmax algebra, the
 *    reference the first page lists).
 *
 * bf16 values travel as their raw 16-bit patterns (uint16_t).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_OK 0
#define ORACLE_ERR_ARG (-1)
#define ORACLE_ERR_BLOCK (-2)
#define ORACLE_ERR_LEN (-3)
#define ORACLE_ERR_SLOT (-4)
#define ORACLE_ERR_NOMEM (-5)

/* ---- bf16 <-> double, from the IEEE-754 binary16-brain layout ----------------
 * bf16 is the top 16 bits of an IEEE binary32: 1 sign, 8 exponent, 7 fraction
 * bits.  Widening is exact: put the 16 bits on top of a zero low half. */
double oracle_bf16_to_double(uint16_t bits) {
  uint32_t u = ((uint32_t)bits) << 16;
  float f;
  memcpy(&f, &u, sizeof f);
  return (double)f;
}

/* Round a double to the nearest bf16, ties to even, straight from the value
 * (no detour through binary32, so there is no double rounding).  Normal bf16
 * numbers are m * 2^(E-7) with 128 <= m < 256 and -126 <= E <= 127; below 2^-126
 * the grid is the subnormal spacing 2^-133. */
uint16_t oracle_double_to_bf16(double x) {
  if (isnan(x)) return (uint16_t)0x7FC0;
  int neg = signbit(x) ? 1 : 0;
  double a = fabs(x);
  uint16_t sign = (uint16_t)(neg << 15);
  if (a == 0.0) return sign;
  if (isinf(a)) return (uint16_t)(sign | 0x7F80);
  int e2;
  (void)frexp(a, &e2); /* a = f * 2^e2, 0.5 <= f < 1, so floor(log2 a) = e2 - 1 */
  int E = e2 - 1;
  if (E < -126) E = -126;                 /* subnormal range shares the 2^-133 grid */
  double quantum = ldexp(1.0, E - 7);
  double r = a / quantum;                 /* exact: division by a power of two */
  double n = floor(r);
  double frac = r - n;
  if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) != 0.0)) n += 1.0;
  double y = n * quantum;                 /* exactly representable in bf16 (or 2^128) */
  if (y >= ldexp(1.0, 128)) return (uint16_t)(sign | 0x7F80);
  float f = (float)y;                     /* exact: every bf16 value is a binary32 value */
  uint32_t u;
  memcpy(&u, &f, sizeof u);
  return (uint16_t)(sign | (uint16_t)((u >> 16) & 0x7FFF));
}

/* ---- the slot-mapping write --------------------------------------------------
 * For every token i and kv head h: if slot_mapping[i] >= 0, copy the bits of
 * k[i][h][:] and v[i][h][:] into the cache at block slot/BS, offset slot%BS.
 * Tokens are applied in index order. */
int oracle_kv_write(const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                    int64_t num_tokens, uint16_t *k_cache, uint16_t *v_cache,
                    int64_t num_blocks, int32_t num_kv_heads, int32_t block_size,
                    int32_t head_dim) {
  if (num_tokens < 0 || num_blocks <= 0 || num_kv_heads <= 0 || block_size <= 0 || head_dim <= 0)
    return ORACLE_ERR_ARG;
  for (int64_t i = 0; i < num_tokens; ++i) {
    int64_t slot = slot_mapping[i];
    if (slot < 0) continue;
    int64_t block = slot / block_size;
    int64_t offset = slot % block_size;
    if (block >= num_blocks) return ORACLE_ERR_SLOT;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      int64_t dst = ((block * num_kv_heads + h) * block_size + offset) * head_dim;
      int64_t src = (i * num_kv_heads + h) * (int64_t)head_dim;
      for (int32_t d = 0; d < head_dim; ++d) {
        k_cache[dst + d] = k[src + d];
        v_cache[dst + d] = v[src + d];
      }
    }
  }
  return ORACLE_OK;
}

/* ---- the gather through the block table --------------------------------------
 * Dense copies Kd[t][d], Vd[t][d] (t < len) of the keys and values of sequence b,
 * kv head g. */
static int gather_dense(double *Kd, double *Vd, const uint16_t *k_cache, const uint16_t *v_cache,
                        const int32_t *table_row, int32_t len, int64_t num_blocks,
                        int32_t num_kv_heads, int32_t block_size, int32_t head_dim, int32_t g) {
  for (int32_t t = 0; t < len; ++t) {
    int64_t phys = table_row[t / block_size];
    int64_t offset = t % block_size;
    if (phys < 0 || phys >= num_blocks) return ORACLE_ERR_BLOCK;
    int64_t base = ((phys * num_kv_heads + g) * block_size + offset) * head_dim;
    for (int32_t d = 0; d < head_dim; ++d) {
      Kd[(int64_t)t * head_dim + d] = oracle_bf16_to_double(k_cache[base + d]);
      Vd[(int64_t)t * head_dim + d] = oracle_bf16_to_double(v_cache[base + d]);
    }
  }
  return ORACLE_OK;
}

/* Softmax attention of one query over dense keys/values on the token range
 * [t0, t1): writes the normalised output o[d] and the range's log-sum-exp of the
 * scaled scores.  An empty range gives o = 0 and lse = -inf. */
static void attend_range(double *o, double *lse, const double *qd, const double *Kd,
                         const double *Vd, int32_t t0, int32_t t1, int32_t head_dim,
                         double scale, double *s) {
  for (int32_t d = 0; d < head_dim; ++d) o[d] = 0.0;
  if (t1 <= t0) {
    *lse = -INFINITY;
    return;
  }
  double m = -INFINITY;
  for (int32_t t = t0; t < t1; ++t) {
    double dot = 0.0;
    for (int32_t d = 0; d < head_dim; ++d) dot += qd[d] * Kd[(int64_t)t * head_dim + d];
    s[t - t0] = scale * dot;
    if (s[t - t0] > m) m = s[t - t0];
  }
  double z = 0.0;
  for (int32_t t = t0; t < t1; ++t) {
    double w = exp(s[t - t0] - m);
    s[t - t0] = w;
    z += w;
  }
  for (int32_t t = t0; t < t1; ++t) {
    double p = s[t - t0] / z;
    for (int32_t d = 0; d < head_dim; ++d) o[d] += p * Vd[(int64_t)t * head_dim + d];
  }
  *lse = m + log(z);
}

/* Common argument checks of the decode functions. */
static int check_decode_args(const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                             int32_t num_kv_heads, int64_t num_blocks, int32_t block_size,
                             int32_t head_dim, int32_t max_blocks_per_seq) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || num_blocks <= 0 ||
      block_size <= 0 || head_dim <= 0 || max_blocks_per_seq <= 0)
    return ORACLE_ERR_ARG;
  if (num_q_heads % num_kv_heads != 0) return ORACLE_ERR_ARG;
  for (int32_t b = 0; b < num_seqs; ++b) {
    if (context_lens[b] < 0 || (int64_t)context_lens[b] > (int64_t)max_blocks_per_seq * block_size)
      return ORACLE_ERR_LEN;
  }
  return ORACLE_OK;
}

/* Attention output for a list of (sequence, query head) rows; rows[2r] = b,
 * rows[2r+1] = h.  out[r][d] (fp64).  The full decode is the list of all rows. */
int oracle_decode_rows(double *out, const int32_t *rows, int32_t num_rows, const uint16_t *q,
                       const uint16_t *k_cache, const uint16_t *v_cache,
                       const int32_t *block_tables, int32_t max_blocks_per_seq,
                       const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                       int32_t num_kv_heads, int64_t num_blocks, int32_t block_size,
                       int32_t head_dim, double scale, int32_t num_threads) {
  int rc = check_decode_args(context_lens, num_seqs, num_q_heads, num_kv_heads, num_blocks,
                             block_size, head_dim, max_blocks_per_seq);
  if (rc) return rc;
  int32_t group = num_q_heads / num_kv_heads;
  int err = ORACLE_OK;
#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
  for (int32_t r = 0; r < num_rows; ++r) {
    int32_t b = rows[2 * r], h = rows[2 * r + 1];
    double *o = out + (int64_t)r * head_dim;
    if (b < 0 || b >= num_seqs || h < 0 || h >= num_q_heads) {
#ifdef _OPENMP
#pragma omp critical
#endif
      err = ORACLE_ERR_ARG;
      continue;
    }
    int32_t len = context_lens[b];
    int32_t g = h / group;
    double *Kd = (double *)malloc(sizeof(double) * ((size_t)len * head_dim + 1));
    double *Vd = (double *)malloc(sizeof(double) * ((size_t)len * head_dim + 1));
    double *s = (double *)malloc(sizeof(double) * ((size_t)len + 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
    if (!Kd || !Vd || !s || !qd) {
#ifdef _OPENMP
#pragma omp critical
#endif
      err = ORACLE_ERR_NOMEM;
    } else {
      int grc = gather_dense(Kd, Vd, k_cache, v_cache,
                             block_tables + (int64_t)b * max_blocks_per_seq, len, num_blocks,
                             num_kv_heads, block_size, head_dim, g);
      if (grc) {
#ifdef _OPENMP
#pragma omp critical
#endif
        err = grc;
      } else {
        for (int32_t d = 0; d < head_dim; ++d)
          qd[d] = oracle_bf16_to_double(q[((int64_t)b * num_q_heads + h) * head_dim + d]);
        double lse;
        attend_range(o, &lse, qd, Kd, Vd, 0, len, head_dim, scale, s);
      }
    }
    free(Kd);
    free(Vd);
    free(s);
    free(qd);
  }
  return err;
}

/* Full decode: out[b][h][d] (fp64) for every sequence b and query head h. */
int oracle_decode_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                            const uint16_t *v_cache, const int32_t *block_tables,
                            int32_t max_blocks_per_seq, const int32_t *context_lens,
                            int32_t num_seqs, int32_t num_q_heads, int32_t num_kv_heads,
                            int64_t num_blocks, int32_t block_size, int32_t head_dim,
                            double scale, int32_t num_threads) {
  if (num_seqs < 0 || num_q_heads <= 0) return ORACLE_ERR_ARG;
  int64_t n = (int64_t)num_seqs * num_q_heads;
  int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)(2 * n + 2));
  if (!rows) return ORACLE_ERR_NOMEM;
  for (int64_t r = 0; r < n; ++r) {
    rows[2 * r] = (int32_t)(r / num_q_heads);
    rows[2 * r + 1] = (int32_t)(r % num_q_heads);
  }
  int rc = oracle_decode_rows(out, rows, (int32_t)n, q, k_cache, v_cache, block_tables,
                              max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                              num_kv_heads, num_blocks, block_size, head_dim, scale, num_threads);
  free(rows);
  return rc;
}

/* Flash-decoding partitions of one row: for r = 0 .. num_parts-1 the token range
 * [r*P, min((r+1)*P, len)) gives o_part[r][d] (normalised) and lse_part[r]. */
int oracle_decode_partitions(double *o_part, double *lse_part, int32_t num_parts,
                             int32_t partition_tokens, int32_t b, int32_t h, const uint16_t *q,
                             const uint16_t *k_cache, const uint16_t *v_cache,
                             const int32_t *block_tables, int32_t max_blocks_per_seq,
                             const int32_t *context_lens, int32_t num_seqs, int32_t num_q_heads,
                             int32_t num_kv_heads, int64_t num_blocks, int32_t block_size,
                             int32_t head_dim, double scale) {
  int rc = check_decode_args(context_lens, num_seqs, num_q_heads, num_kv_heads, num_blocks,
                             block_size, head_dim, max_blocks_per_seq);
  if (rc) return rc;
  if (partition_tokens <= 0 || num_parts < 0 || b < 0 || b >= num_seqs || h < 0 ||
      h >= num_q_heads)
    return ORACLE_ERR_ARG;
  int32_t group = num_q_heads / num_kv_heads;
  int32_t len = context_lens[b], g = h / group;
  double *Kd = (double *)malloc(sizeof(double) * ((size_t)len * head_dim + 1));
  double *Vd = (double *)malloc(sizeof(double) * ((size_t)len * head_dim + 1));
  double *s = (double *)malloc(sizeof(double) * ((size_t)partition_tokens + 1));
  double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
  if (!Kd || !Vd || !s || !qd) {
    rc = ORACLE_ERR_NOMEM;
  } else {
    rc = gather_dense(Kd, Vd, k_cache, v_cache, block_tables + (int64_t)b * max_blocks_per_seq,
                      len, num_blocks, num_kv_heads, block_size, head_dim, g);
    if (!rc) {
      for (int32_t d = 0; d < head_dim; ++d)
        qd[d] = oracle_bf16_to_double(q[((int64_t)b * num_q_heads + h) * head_dim + d]);
      for (int32_t r = 0; r < num_parts; ++r) {
        int64_t t0 = (int64_t)r * partition_tokens;
        int64_t t1 = t0 + partition_tokens;
        if (t0 > len) t0 = len;
        if (t1 > len) t1 = len;
        attend_range(o_part + (int64_t)r * head_dim, lse_part + r, qd, Kd, Vd, (int32_t)t0,
                     (int32_t)t1, head_dim, scale, s);
      }
    }
  }
  free(Kd);
  free(Vd);
  free(s);
  free(qd);
  return rc;
}

/* Merge per-range results: M = max lse_r, w_r = exp(lse_r - M),
 * out = sum_r w_r o_r / sum_r w_r.  Ranges with lse = -inf weigh nothing; if all
 * ranges are empty the output is zero. */
int oracle_lse_combine(double *out, const double *o_part, const double *lse_part,
                       int32_t num_parts, int32_t head_dim) {
  if (num_parts < 0 || head_dim <= 0) return ORACLE_ERR_ARG;
  double M = -INFINITY;
  for (int32_t r = 0; r < num_parts; ++r)
    if (lse_part[r] > M) M = lse_part[r];
  for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
  if (M == -INFINITY) return ORACLE_OK;
  double den = 0.0;
  for (int32_t r = 0; r < num_parts; ++r) {
    double w = exp(lse_part[r] - M);
    den += w;
    for (int32_t d = 0; d < head_dim; ++d) out[d] += w * o_part[(int64_t)r * head_dim + d];
  }
  for (int32_t d = 0; d < head_dim; ++d) out[d] /= den;
  return ORACLE_OK;
}

/* ---- rotary position embedding, fused into the write ---------------------------
 * "Building ... with tiny-vLLM", CUDA kernel engineering: RoPE rotates pairs of
 * coordinates by position-dependent angles (sine/cosine); "llm-stack", Serving engine:
 * RoPE is applied at absolute positions before keys enter the cache, and the Model
 * section names the two pairings (its "RoPE pairing permutation").
 * Pairs: neox_style != 0 ("rotate half"): (i, i + r/2) for i < r/2; else interleaved
 * (2i, 2i + 1).  Angle table: cos_sin[pos][0 .. r/2) = cos, [r/2 .. r) = sin of pair i
 * (fp32, given by the caller).  Coordinates at or past rotary_dim are copied.
 * The rotated bf16 value is decided by floating point, so it is computed in the
 * precision the kernel uses: fp32 products and sums, each rounded once (no fused
 * multiply-add), then rounded to bf16 (nearest even):
 *   x1' = x1*c - x2*s,   x2' = x2*c + x1*s.                                        */
static void rope_row(uint16_t *dst, const uint16_t *src, const float *cs, int32_t head_dim,
                     int32_t rotary_dim, int neox) {
  const int32_t half = rotary_dim / 2;
  for (int32_t d = 0; d < head_dim; ++d) dst[d] = src[d];
  for (int32_t i = 0; i < half; ++i) {
    const int32_t a = neox ? i : 2 * i, b = neox ? i + half : 2 * i + 1;
    const float x1 = (float)oracle_bf16_to_double(src[a]);
    const float x2 = (float)oracle_bf16_to_double(src[b]);
    const float c = cs[i], s = cs[half + i];
    volatile float p1 = x1 * c, p2 = x2 * s, p3 = x2 * c, p4 = x1 * s;
    const float r1 = p1 - p2, r2 = p3 + p4;
    dst[a] = oracle_double_to_bf16((double)r1);
    dst[b] = oracle_double_to_bf16((double)r2);
  }
}

/* Rotate k (and q, in place, when q != NULL) at positions[i], then write k and v at
 * slot_mapping[i] like oracle_kv_write.  q is [num_tokens][num_q_heads][head_dim]. */
int oracle_kv_write_rope(const uint16_t *k, const uint16_t *v, uint16_t *q, int32_t num_q_heads,
                         const int64_t *slot_mapping, const int64_t *positions,
                         int64_t num_tokens, const float *cos_sin, int64_t max_position,
                         int32_t rotary_dim, int32_t neox_style, uint16_t *k_cache,
                         uint16_t *v_cache, int64_t num_blocks, int32_t num_kv_heads,
                         int32_t block_size, int32_t head_dim) {
  if (num_tokens < 0 || rotary_dim <= 0 || rotary_dim > head_dim || rotary_dim % 2 != 0)
    return ORACLE_ERR_ARG;
  uint16_t *krot = (uint16_t *)malloc(sizeof(uint16_t) * ((size_t)num_tokens * num_kv_heads * head_dim + 1));
  uint16_t *row = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)head_dim);
  if (!krot || !row) {
    free(krot);
    free(row);
    return ORACLE_ERR_NOMEM;
  }
  int rc = ORACLE_OK;
  for (int64_t i = 0; i < num_tokens && rc == ORACLE_OK; ++i) {
    const int64_t pos = positions[i];
    if (pos < 0 || pos >= max_position) {
      rc = ORACLE_ERR_ARG;
      break;
    }
    const float *cs = cos_sin + pos * rotary_dim;
    for (int32_t h = 0; h < num_kv_heads; ++h) {
      const int64_t o = (i * num_kv_heads + h) * (int64_t)head_dim;
      rope_row(krot + o, k + o, cs, head_dim, rotary_dim, neox_style);
    }
    if (q) {
      for (int32_t h = 0; h < num_q_heads; ++h) {
        uint16_t *qr = q + (i * num_q_heads + h) * (int64_t)head_dim;
        rope_row(row, qr, cs, head_dim, rotary_dim, neox_style);
        for (int32_t d = 0; d < head_dim; ++d) qr[d] = row[d];
      }
    }
  }
  if (rc == ORACLE_OK)
    rc = oracle_kv_write(krot, v, slot_mapping, num_tokens, k_cache, v_cache, num_blocks,
                         num_kv_heads, block_size, head_dim);
  free(krot);
  free(row);
  return rc;
}

/* ---- paged prefill / recompute attention ------------------------------------------
 * "vLLM-Style Llama Inference Engine", How it works: prefill and recomputation use
 * causal attention.  Over the paged cache: sequence b holds L_b = context_lens[b]
 * tokens, of which the last n_b = query_start[b+1] - query_start[b] are this chunk's
 * queries; query i of the chunk sits at position p = L_b - n_b + i and attends to keys
 * t <= p (causal).  q and out are packed [num_queries][num_q_heads][head_dim] with
 * sequence b's queries at rows query_start[b] .. query_start[b+1]-1.  fp64.
 * The (sequence, kv head) pairs are independent and are shared out over threads
 * (OpenMP; num_threads <= 0: all); each pair's arithmetic is the same either way. */
int oracle_prefill_attention(double *out, const uint16_t *q, const uint16_t *k_cache,
                             const uint16_t *v_cache, const int32_t *block_tables,
                             int32_t max_blocks_per_seq, const int32_t *context_lens,
                             const int32_t *query_start, int32_t num_seqs, int32_t num_q_heads,
                             int32_t num_kv_heads, int64_t num_blocks, int32_t block_size,
                             int32_t head_dim, double scale, int32_t num_threads) {
  int rc = check_decode_args(context_lens, num_seqs, num_q_heads, num_kv_heads, num_blocks,
                             block_size, head_dim, max_blocks_per_seq);
  if (rc) return rc;
  for (int32_t b = 0; b < num_seqs; ++b) {
    const int32_t n = query_start[b + 1] - query_start[b];
    if (n < 0 || n > context_lens[b]) return ORACLE_ERR_LEN;
  }
  const int32_t group = num_q_heads / num_kv_heads;
  const int64_t pairs = (int64_t)num_seqs * num_kv_heads;
  int err = ORACLE_OK;
#ifdef _OPENMP
  if (num_threads <= 0) num_threads = omp_get_max_threads();
#pragma omp parallel for schedule(dynamic, 1) num_threads(num_threads)
#endif
  for (int64_t pg = 0; pg < pairs; ++pg) {
    const int32_t b = (int32_t)(pg / num_kv_heads), g = (int32_t)(pg % num_kv_heads);
    const int32_t len = context_lens[b];
    const int32_t n = query_start[b + 1] - query_start[b];
    double *Kd = (double *)malloc(sizeof(double) * ((size_t)len * head_dim + 1));
    double *Vd = (double *)malloc(sizeof(double) * ((size_t)len * head_dim + 1));
    double *s = (double *)malloc(sizeof(double) * ((size_t)len + 1));
    double *qd = (double *)malloc(sizeof(double) * (size_t)head_dim);
    int prc = ORACLE_OK;
    if (!Kd || !Vd || !s || !qd) prc = ORACLE_ERR_NOMEM;
    if (!prc)
      prc = gather_dense(Kd, Vd, k_cache, v_cache, block_tables + (int64_t)b * max_blocks_per_seq,
                         len, num_blocks, num_kv_heads, block_size, head_dim, g);
    for (int32_t i = 0; i < n && !prc; ++i) {
      const int32_t pos = len - n + i;
      for (int32_t j = 0; j < group; ++j) {
        const int32_t h = g * group + j;
        const int64_t row = ((int64_t)(query_start[b] + i) * num_q_heads + h) * head_dim;
        for (int32_t d = 0; d < head_dim; ++d) qd[d] = oracle_bf16_to_double(q[row + d]);
        double lse;
        attend_range(out + row, &lse, qd, Kd, Vd, 0, pos + 1, head_dim, scale, s);
      }
    }
    free(Kd);
    free(Vd);
    free(s);
    free(qd);
    if (prc) {
#ifdef _OPENMP
#pragma omp critical
#endif
      err = prc;
    }
  }
  return err;
}
