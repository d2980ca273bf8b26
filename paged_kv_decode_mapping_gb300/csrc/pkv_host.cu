// pkv_host.cu -- host pieces shared by the attention entry points: the per-thread
// error message, device queries, the cache of encoded TMA tensor maps of the KV pools
// (2-D box {64 dims, rows} for head_dim 64, 3-D {64, 1, rows} for head_dim 128; 128-byte
// swizzle), the argument checks of the attention calls, and the device error API.
#include <cuda.h>  // CUtensorMap and its enums (header only; the entry point is fetched at run time)
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdarg>
#include <cstdio>
#include <mutex>

#include "pkv_internal.h"

namespace pkv {

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

std::mutex &attn_mutex() {
  static std::mutex mu;
  return mu;
}

namespace {

int g_sms[kMaxDevices];  // SM count per device (0 = not queried)

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

}  // namespace

int current_device(int *dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e != cudaSuccess) return cuda_error(e, "cudaGetDevice");
  if (*dev < 0 || *dev >= kMaxDevices) return set_error(PKV_ERR_CUDA, "device index %d", *dev);
  return PKV_OK;
}

int device_sms(int *sms) {
  int dev = 0;
  int rc = current_device(&dev);
  if (rc) return rc;
  if (!g_sms[dev]) {
    int n = 0;
    cudaError_t e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return cuda_error(e, "cudaDeviceGetAttribute");
    g_sms[dev] = n;
  }
  *sms = g_sms[dev];
  return PKV_OK;
}

namespace {

// A small cache of encoded tensor maps, keyed by (pointer, pool shape).
struct MapEntry {
  const void *ptr;
  int64_t nb;
  int32_t hkv, bs, d;
  CUtensorMap map;
};
MapEntry g_maps[16];
int g_maps_next = 0;

}  // namespace

static int tensor_map(const void *cache_ptr, const pkv_cache_desc &c, CUtensorMap *out) {
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

static bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
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

int maps_for(const pkv_bf16 *k_cache, const pkv_bf16 *v_cache, const pkv_cache_desc &c,
             CUtensorMap *tmk, CUtensorMap *tmv) {
  int rc = tensor_map(k_cache, c, tmk);
  if (!rc) rc = tensor_map(v_cache, c, tmv);
  return rc;
}

}  // namespace pkv

using namespace pkv;

PKV_API int pkv_device_errors(uint32_t *flags, int clear) {
  if (!flags) return set_error(PKV_ERR_NULL, "pkv_device_errors: flags is NULL");
  *flags = 0;
  cudaError_t e = cudaDeviceSynchronize();
  if (e != cudaSuccess) return cuda_error(e, "cudaDeviceSynchronize");
  if ((e = read_decode_errors(flags, clear)) != cudaSuccess) return cuda_error(e, "decode error word");
  if ((e = read_prefill_errors(flags, clear)) != cudaSuccess) return cuda_error(e, "prefill error word");
  if ((e = read_write_errors(flags, clear)) != cudaSuccess) return cuda_error(e, "write error word");
  clear_error();
  return PKV_OK;
}

PKV_API const char *pkv_last_error(void) { return g_msg; }
