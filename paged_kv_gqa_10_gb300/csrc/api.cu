// C ABI of libpgqa: argument validation (host-checkable errors return before any
// launch), TMA descriptor encoding through the driver entry point (cached by
// address and shape), device-property caches, and dispatch to the kernel files.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "host.h"

namespace pgqa {
namespace {

constexpr int kMaxDevices = 64;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

struct MapKey {
  const void* base;
  int dtype, rank, swizzle, pad;
  uint64_t dims[3];
  uint64_t pitch[2];
  uint32_t box[3];
  uint32_t pad2;
};

struct MapEntry {
  MapKey key;
  CUtensorMap map;
  bool used;
};

constexpr int kMapCache = 64;
std::mutex g_map_mu;
MapEntry g_maps[kMapCache];
int g_map_next = 0;

bool encode_cached(CUtensorMap* out, const MapKey& key) {
  {
    std::lock_guard<std::mutex> lock(g_map_mu);
    for (int i = 0; i < kMapCache; ++i)
      if (g_maps[i].used && memcmp(&g_maps[i].key, &key, sizeof key) == 0) {
        *out = g_maps[i].map;
        return true;
      }
  }
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (fn == nullptr) return false;
  cuuint64_t dims[3], strides[2];
  cuuint32_t box[3], estr[3] = {1, 1, 1};
  for (int i = 0; i < key.rank; ++i) {
    dims[i] = key.dims[i];
    box[i] = key.box[i];
  }
  for (int i = 0; i + 1 < key.rank; ++i) strides[i] = key.pitch[i];
  CUtensorMap m;
  const CUresult r = fn(&m, static_cast<CUtensorMapDataType>(key.dtype), key.rank,
                        const_cast<void*>(key.base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE,
                        static_cast<CUtensorMapSwizzle>(key.swizzle),
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return false;
  std::lock_guard<std::mutex> lock(g_map_mu);
  g_maps[g_map_next].key = key;
  g_maps[g_map_next].map = m;
  g_maps[g_map_next].used = true;
  g_map_next = (g_map_next + 1) % kMapCache;
  *out = m;
  return true;
}

int current_device() {
  int dev = -1;
  return cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < kMaxDevices ? dev : -1;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

}  // namespace

bool tensor_map_2d(CUtensorMap* out, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                   uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle) {
  MapKey k;
  memset(&k, 0, sizeof k);
  k.base = base;
  k.dtype = dtype;
  k.rank = 2;
  k.swizzle = swizzle;
  k.dims[0] = inner;
  k.dims[1] = rows;
  k.pitch[0] = row_bytes;
  k.box[0] = box_inner;
  k.box[1] = box_rows;
  return encode_cached(out, k);
}

bool tensor_map_3d(CUtensorMap* out, const void* base, CUtensorMapDataType dtype, uint64_t d0,
                   uint64_t d1, uint64_t d2, uint64_t pitch1, uint64_t pitch2, uint32_t box0,
                   uint32_t box1, uint32_t box2, CUtensorMapSwizzle swizzle) {
  MapKey k;
  memset(&k, 0, sizeof k);
  k.base = base;
  k.dtype = dtype;
  k.rank = 3;
  k.swizzle = swizzle;
  k.dims[0] = d0;
  k.dims[1] = d1;
  k.dims[2] = d2;
  k.pitch[0] = pitch1;
  k.pitch[1] = pitch2;
  k.box[0] = box0;
  k.box[1] = box1;
  k.box[2] = box2;
  return encode_cached(out, k);
}

int num_sms_current_device() {
  static int cache[kMaxDevices] = {0};
  const int dev = current_device();
  if (dev < 0) return 0;
  if (cache[dev] == 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    cache[dev] = n;
  }
  return cache[dev];
}

bool smem_attr_ready(const void* kernel, int bytes) {
  struct Entry {
    const void* kernel;
    int dev;
  };
  static std::mutex mu;
  static Entry done[256];
  static int n_done = 0;
  const int dev = current_device();
  if (dev < 0) return false;
  std::lock_guard<std::mutex> lock(mu);
  for (int i = 0; i < n_done; ++i)
    if (done[i].kernel == kernel && done[i].dev == dev) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) !=
      cudaSuccess)
    return false;
  if (n_done < 256) done[n_done++] = Entry{kernel, dev};
  return true;
}

pgqa_status_t decode_validate(const void* out, const void* q, const void* k_cache,
                              const void* v_cache, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                              int block_size, float scale, int cache_dtype, const float* k_scale,
                              const float* v_scale, int max_context_len, const void* key,
                              const void* value) {
  if (num_seqs < 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 ||
      block_size <= 0 || max_context_len < 0 || max_blocks_per_seq < 0 || !isfinite(scale))
    return PGQA_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PGQA_EINVAL;
  if (cache_dtype == PGQA_DTYPE_E4M3) {
    if (k_scale == nullptr || v_scale == nullptr) return PGQA_EINVAL;
  } else if (cache_dtype == PGQA_DTYPE_BF16) {
    if (k_scale != nullptr || v_scale != nullptr) return PGQA_EINVAL;
  } else {
    return PGQA_EUNSUPPORTED;
  }
  const int group = num_q_heads / num_kv_heads;
  if (group > 8 || (block_size != 8 && block_size != 16 && block_size != 32))
    return PGQA_EUNSUPPORTED;
  if (head_dim != 128 && head_dim != 64) return PGQA_EUNSUPPORTED;
  if (static_cast<int64_t>(num_blocks) * num_kv_heads * block_size > INT32_MAX)
    return PGQA_EUNSUPPORTED;
  if (num_seqs == 0) return PGQA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !context_lens) return PGQA_EINVAL;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return PGQA_EINVAL;
  if ((key == nullptr) != (value == nullptr) || !aligned(key, 16) || !aligned(value, 16))
    return PGQA_EINVAL;
  return PGQA_OK;
}


}  // namespace pgqa

using pgqa::aligned;

extern "C" {

int pgqa_abi_version(void) { return PGQA_ABI_VERSION; }

void pgqa_set_decode_wait_limit_ns(uint64_t ns) { pgqa::set_decode_wait_limit_ns(ns); }

const char* pgqa_status_string(pgqa_status_t s) {
  switch (s) {
    case PGQA_OK: return "ok";
    case PGQA_EINVAL: return "invalid argument";
    case PGQA_EUNSUPPORTED: return "unsupported configuration";
    case PGQA_ENOWORKSPACE: return "workspace too small";
    case PGQA_ECUDA: return "CUDA runtime error";
    case PGQA_EBADINDEX: return "block id or slot out of range";
    case PGQA_ETIMEOUT: return "bounded wait in a kernel gave up";
    default: return "unknown status";
  }
}

int64_t pgqa_kv_cache_bytes(int num_layers, int64_t tokens, int num_kv_heads, int head_dim,
                            int cache_dtype) {
  if (num_layers < 0 || tokens < 0 || num_kv_heads < 0 || head_dim < 0) return -1;
  int64_t elem;
  if (cache_dtype == PGQA_DTYPE_BF16)
    elem = 2;
  else if (cache_dtype == PGQA_DTYPE_E4M3)
    elem = 1;
  else
    return -1;
  return 2 * static_cast<int64_t>(num_layers) * tokens * num_kv_heads * head_dim * elem;
}

pgqa_status_t pgqa_kv_cache_write(const void* key, const void* value,
                                  const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                  int head_dim, void* k_cache, void* v_cache, int num_blocks,
                                  int block_size, int cache_dtype, const float* k_scale,
                                  const float* v_scale, int* dev_status, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0 || block_size <= 0)
    return PGQA_EINVAL;
  if (head_dim % 8 != 0) return PGQA_EUNSUPPORTED;
  if (cache_dtype == PGQA_DTYPE_E4M3) {
    if (k_scale == nullptr || v_scale == nullptr) return PGQA_EINVAL;
  } else if (cache_dtype == PGQA_DTYPE_BF16) {
    if (k_scale != nullptr || v_scale != nullptr) return PGQA_EINVAL;
  } else {
    return PGQA_EUNSUPPORTED;
  }
  if (num_tokens == 0) return PGQA_OK;
  if (!key || !value || !slot_mapping || !k_cache || !v_cache) return PGQA_EINVAL;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return PGQA_EINVAL;
  return pgqa::launch_kv_cache_write(key, value, slot_mapping, num_tokens, num_kv_heads, head_dim,
                                     k_cache, v_cache, num_blocks, block_size, cache_dtype,
                                     k_scale, v_scale, dev_status,
                                     static_cast<cudaStream_t>(stream));
}

pgqa_status_t pgqa_paged_kv_gather(const void* k_cache, const void* v_cache, int cache_dtype,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs, int num_kv_heads,
                                   int head_dim, int num_blocks, int block_size,
                                   int max_context_len, void* k_out, void* v_out,
                                   int* dev_status, void* stream) {
  if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0 || block_size <= 0 ||
      max_context_len < 0 || max_blocks_per_seq < 0)
    return PGQA_EINVAL;
  if (cache_dtype != PGQA_DTYPE_BF16 && cache_dtype != PGQA_DTYPE_E4M3) return PGQA_EUNSUPPORTED;
  const int elem = cache_dtype == PGQA_DTYPE_BF16 ? 2 : 1;
  if ((head_dim * elem) % 16 != 0) return PGQA_EUNSUPPORTED;
  if (num_seqs == 0 || max_context_len == 0) return PGQA_OK;
  if (!k_cache || !v_cache || !block_tables || !context_lens || !k_out || !v_out)
    return PGQA_EINVAL;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(k_out, 16) || !aligned(v_out, 16))
    return PGQA_EINVAL;
  return pgqa::launch_kv_gather(k_cache, v_cache, cache_dtype, block_tables, max_blocks_per_seq,
                                context_lens, num_seqs, num_kv_heads, head_dim, num_blocks,
                                block_size, max_context_len, k_out, v_out, dev_status,
                                static_cast<cudaStream_t>(stream));
}

int pgqa_decode_grid_size(int num_sms, int head_dim, int cache_dtype) {
  if (num_sms <= 0 || (head_dim != 64 && head_dim != 128) ||
      (cache_dtype != PGQA_DTYPE_BF16 && cache_dtype != PGQA_DTYPE_E4M3))
    return PGQA_EINVAL;
  return pgqa::decode_plan(1, 1, head_dim, cache_dtype, num_sms).grid;
}

size_t pgqa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int max_context_len) {
  (void)num_q_heads;
  (void)max_context_len;
  if (num_seqs <= 0 || num_kv_heads <= 0 || head_dim <= 0) return 0;
  const int sms = pgqa::num_sms_current_device();
  const size_t a =
      pgqa::decode_plan(num_seqs, num_kv_heads, head_dim, PGQA_DTYPE_BF16, sms).bytes;
  const size_t b =
      pgqa::decode_plan(num_seqs, num_kv_heads, head_dim, PGQA_DTYPE_E4M3, sms).bytes;
  return a > b ? a : b;
}


// Shared by the decode entry points (window 0: the whole context; key/value null: no
// fused append).
static pgqa_status_t decode_call(void* out, float* lse, const void* q, const void* k_cache,
                                 const void* v_cache, const int32_t* block_tables,
                                 int max_blocks_per_seq, const int32_t* context_lens,
                                 int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int num_blocks, int block_size, float scale, int window,
                                 int cache_dtype, const float* k_scale, const float* v_scale,
                                 int max_context_len, void* workspace, size_t workspace_bytes,
                                 int* dev_status, void* stream, const void* key = nullptr,
                                 const void* value = nullptr) {
  const pgqa_status_t rc = pgqa::decode_validate(
      out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
      num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, cache_dtype, k_scale,
      v_scale, max_context_len, key, value);
  if (rc != PGQA_OK || num_seqs == 0) return rc;
  const int sms = pgqa::num_sms_current_device();
  if (sms <= 0) return PGQA_ECUDA;
  const pgqa::DecodePlan plan =
      pgqa::decode_plan(num_seqs, num_kv_heads, head_dim, cache_dtype, sms);
  if (workspace == nullptr || workspace_bytes < plan.bytes) return PGQA_ENOWORKSPACE;
  if (!aligned(workspace, 256)) return PGQA_EINVAL;
  pgqa::DecodeArgs a;
  a.out = out;
  a.lse = lse;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.scale = scale;
  a.cache_dtype = cache_dtype;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.max_context_len = max_context_len;
  a.window = window;
  a.q_len = 1;
  a.new_key = key;
  a.new_value = value;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.dev_status = dev_status;
  a.stream = static_cast<cudaStream_t>(stream);
  return pgqa::launch_paged_decode(a, plan);
}

pgqa_status_t pgqa_paged_attention_decode(void* out, float* lse, const void* q,
                                          const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* context_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int num_blocks, int block_size, float scale,
                                          int cache_dtype, const float* k_scale,
                                          const float* v_scale, int max_context_len,
                                          void* workspace, size_t workspace_bytes,
                                          int* dev_status, void* stream) {
  return decode_call(out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks,
                     block_size, scale, 0, cache_dtype, k_scale, v_scale, max_context_len,
                     workspace, workspace_bytes, dev_status, stream);
}

pgqa_status_t pgqa_paged_attention_decode_window(
    void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, int block_size,
    float scale, int window, int cache_dtype, const float* k_scale, const float* v_scale,
    int max_context_len, void* workspace, size_t workspace_bytes, int* dev_status, void* stream) {
  if (window <= 0) return PGQA_EINVAL;
  return decode_call(out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks,
                     block_size, scale, window, cache_dtype, k_scale, v_scale, max_context_len,
                     workspace, workspace_bytes, dev_status, stream);
}

pgqa_status_t pgqa_paged_attention_decode_append(
    void* out, float* lse, const void* q, const void* key, const void* value, void* k_cache,
    void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int num_blocks, int block_size, float scale, int cache_dtype, const float* k_scale,
    const float* v_scale, int max_context_len, void* workspace, size_t workspace_bytes,
    int* dev_status, void* stream) {
  if (num_seqs > 0 && (key == nullptr || value == nullptr)) return PGQA_EINVAL;
  return decode_call(out, lse, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                     context_lens, num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks,
                     block_size, scale, 0, cache_dtype, k_scale, v_scale, max_context_len,
                     workspace, workspace_bytes, dev_status, stream, key, value);
}

size_t pgqa_decode_multi_workspace_size(int num_seqs, int q_len, int num_q_heads,
                                        int num_kv_heads, int head_dim) {
  if (num_seqs <= 0 || q_len <= 0 || num_q_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
      num_q_heads % num_kv_heads != 0)
    return 0;
  const int nt = pgqa::decode_row_tiles(q_len, num_q_heads / num_kv_heads);
  if (nt == 0) return pgqa::kPrefillWorkspaceBytes;  // the prefill kernel runs these
  const int sms = pgqa::num_sms_current_device();
  const size_t a =
      pgqa::decode_plan(num_seqs, num_kv_heads, head_dim, PGQA_DTYPE_BF16, sms, nt).bytes;
  const size_t b =
      pgqa::decode_plan(num_seqs, num_kv_heads, head_dim, PGQA_DTYPE_E4M3, sms, nt).bytes;
  return a > b ? a : b;
}

pgqa_status_t pgqa_paged_attention_decode_multi(
    void* out, float* lse, const void* q, int q_len, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, int block_size,
    float scale, int cache_dtype, const float* k_scale, const float* v_scale, int max_context_len,
    void* workspace, size_t workspace_bytes, int* dev_status, void* stream) {
  if (q_len < 1 || q_len > PGQA_MAX_DECODE_TOKENS) return q_len < 1 ? PGQA_EINVAL
                                                                      : PGQA_EUNSUPPORTED;
  const pgqa_status_t rc = pgqa::decode_validate(
      out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
      num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, cache_dtype, k_scale,
      v_scale, max_context_len, nullptr, nullptr);
  if (rc != PGQA_OK || num_seqs == 0) return rc;
  const int nt = pgqa::decode_row_tiles(q_len, num_q_heads / num_kv_heads);
  if (nt == 0) {
    // more query rows per (sequence, kv-head) than the decode kernel holds: the
    // prefill kernel, in its grouped-rows layout, with q_len new tokens per sequence
    if (block_size != 16) return PGQA_EUNSUPPORTED;
    if (!(scale > 0.f)) return PGQA_EINVAL;
    if (workspace == nullptr || workspace_bytes < pgqa::kPrefillWorkspaceBytes)
      return PGQA_ENOWORKSPACE;
    if (!aligned(workspace, 16)) return PGQA_EINVAL;
    if (num_seqs > pgqa::prefill_max_seqs() || max_context_len > (1 << 26))
      return PGQA_EUNSUPPORTED;
    pgqa::PrefillArgs a;
    a.out = out;
    a.lse = lse;
    a.q = q;
    a.k_cache = k_cache;
    a.v_cache = v_cache;
    a.block_tables = block_tables;
    a.max_blocks_per_seq = max_blocks_per_seq;
    a.cu_seqlens = nullptr;  // q_len tokens per sequence, in order
    a.seq_lens_k = context_lens;
    a.max_seqlen_k = max_context_len;
    a.workspace = workspace;
    a.num_tokens = num_seqs * q_len;
    a.num_seqs = num_seqs;
    a.max_seqlen = q_len;
    a.num_q_heads = num_q_heads;
    a.num_kv_heads = num_kv_heads;
    a.head_dim = head_dim;
    a.num_blocks = num_blocks;
    a.block_size = block_size;
    a.scale = scale;
    a.cache_dtype = cache_dtype;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    a.dev_status = dev_status;
    a.stream = static_cast<cudaStream_t>(stream);
    return pgqa::launch_paged_prefill(a);
  }
  const int sms = pgqa::num_sms_current_device();
  if (sms <= 0) return PGQA_ECUDA;
  const pgqa::DecodePlan plan =
      pgqa::decode_plan(num_seqs, num_kv_heads, head_dim, cache_dtype, sms, nt);
  if (workspace == nullptr || workspace_bytes < plan.bytes) return PGQA_ENOWORKSPACE;
  if (!aligned(workspace, 256)) return PGQA_EINVAL;
  pgqa::DecodeArgs a;
  a.out = out;
  a.lse = lse;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.context_lens = context_lens;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.scale = scale;
  a.cache_dtype = cache_dtype;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.max_context_len = max_context_len;
  a.window = 0;
  a.q_len = q_len;
  a.new_key = nullptr;
  a.new_value = nullptr;
  a.workspace = workspace;
  a.workspace_bytes = workspace_bytes;
  a.dev_status = dev_status;
  a.stream = static_cast<cudaStream_t>(stream);
  return pgqa::launch_paged_decode(a, plan);
}

size_t pgqa_prefill_workspace_size(int num_seqs, int num_q_heads, int max_seqlen) {
  (void)num_seqs;
  (void)num_q_heads;
  (void)max_seqlen;
  return pgqa::kPrefillWorkspaceBytes;
}

// Shared by the prefill entry points (seq_lens_k null: no cached prefix).
static pgqa_status_t prefill_call(void* out, float* lse, const void* q, int num_tokens,
                                  const void* k_cache, const void* v_cache,
                                  const int32_t* block_tables, int max_blocks_per_seq,
                                  const int32_t* cu_seqlens, const int32_t* seq_lens_k,
                                  int num_seqs, int max_seqlen, int max_seqlen_k,
                                  int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                                  int block_size, float scale, int cache_dtype,
                                  const float* k_scale, const float* v_scale, void* workspace,
                                  size_t workspace_bytes, int* dev_status, void* stream) {
  if (num_seqs < 0 || max_seqlen < 0 || max_seqlen_k < 0 || num_tokens < 0 || num_q_heads <= 0 ||
      num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0 || block_size <= 0 ||
      max_blocks_per_seq < 0 || !isfinite(scale) || !(scale > 0.f))
    return PGQA_EINVAL;
  if (num_q_heads % num_kv_heads != 0) return PGQA_EINVAL;
  if (cache_dtype == PGQA_DTYPE_E4M3) {
    if (k_scale == nullptr || v_scale == nullptr) return PGQA_EINVAL;
    if (!aligned(k_scale, 4) || !aligned(v_scale, 4)) return PGQA_EINVAL;
  } else if (cache_dtype == PGQA_DTYPE_BF16) {
    if (k_scale != nullptr || v_scale != nullptr) return PGQA_EINVAL;
  } else {
    return PGQA_EUNSUPPORTED;
  }
  if (head_dim != 128 && head_dim != 64) return PGQA_EUNSUPPORTED;
  if (block_size != 16) return PGQA_EUNSUPPORTED;
  if (static_cast<int64_t>(num_blocks) * num_kv_heads * 16 > INT32_MAX) return PGQA_EUNSUPPORTED;
  if (num_seqs > pgqa::prefill_max_seqs() || max_seqlen > pgqa::prefill_max_seqlen() ||
      max_seqlen_k > (1 << 26))
    return PGQA_EUNSUPPORTED;
  if (num_seqs == 0 || max_seqlen == 0 || num_tokens == 0) return PGQA_OK;
  if (workspace == nullptr || workspace_bytes < pgqa::kPrefillWorkspaceBytes)
    return PGQA_ENOWORKSPACE;
  if (!aligned(workspace, 16)) return PGQA_EINVAL;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !cu_seqlens) return PGQA_EINVAL;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return PGQA_EINVAL;
  pgqa::PrefillArgs a;
  a.out = out;
  a.lse = lse;
  a.q = q;
  a.k_cache = k_cache;
  a.v_cache = v_cache;
  a.block_tables = block_tables;
  a.max_blocks_per_seq = max_blocks_per_seq;
  a.cu_seqlens = cu_seqlens;
  a.seq_lens_k = seq_lens_k;
  a.max_seqlen_k = max_seqlen_k;
  a.workspace = workspace;
  a.num_tokens = num_tokens;
  a.num_seqs = num_seqs;
  a.max_seqlen = max_seqlen;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.head_dim = head_dim;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.scale = scale;
  a.cache_dtype = cache_dtype;
  a.k_scale = k_scale;
  a.v_scale = v_scale;
  a.dev_status = dev_status;
  a.stream = static_cast<cudaStream_t>(stream);
  return pgqa::launch_paged_prefill(a);
}

pgqa_status_t pgqa_paged_prefill_varlen(void* out, float* lse, const void* q, int num_tokens,
                                        const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, int max_blocks_per_seq,
                                        const int32_t* cu_seqlens, int num_seqs, int max_seqlen,
                                        int num_q_heads, int num_kv_heads, int head_dim,
                                        int num_blocks, int block_size, float scale,
                                        void* workspace, size_t workspace_bytes,
                                        int* dev_status, void* stream) {
  return prefill_call(out, lse, q, num_tokens, k_cache, v_cache, block_tables,
                      max_blocks_per_seq, cu_seqlens, nullptr, num_seqs, max_seqlen, max_seqlen,
                      num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale,
                      PGQA_DTYPE_BF16, nullptr, nullptr, workspace, workspace_bytes, dev_status,
                      stream);
}

pgqa_status_t pgqa_paged_prefill_varlen_kv(void* out, float* lse, const void* q, int num_tokens,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_tables, int max_blocks_per_seq,
                                           const int32_t* cu_seqlens_q, const int32_t* seq_lens_k,
                                           int num_seqs, int max_seqlen_q, int max_seqlen_k,
                                           int num_q_heads, int num_kv_heads, int head_dim,
                                           int num_blocks, int block_size, float scale,
                                           void* workspace, size_t workspace_bytes,
                                           int* dev_status, void* stream) {
  if (seq_lens_k == nullptr && num_seqs > 0) return PGQA_EINVAL;
  return prefill_call(out, lse, q, num_tokens, k_cache, v_cache, block_tables,
                      max_blocks_per_seq, cu_seqlens_q, seq_lens_k, num_seqs, max_seqlen_q,
                      max_seqlen_k, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size,
                      scale, PGQA_DTYPE_BF16, nullptr, nullptr, workspace, workspace_bytes,
                      dev_status, stream);
}

pgqa_status_t pgqa_paged_prefill_varlen_e4m3(
    void* out, float* lse, const void* q, int num_tokens, const void* k_cache,
    const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, int num_seqs, int max_seqlen_q,
    int max_seqlen_k, int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
    int block_size, float scale, const float* k_scale, const float* v_scale, void* workspace,
    size_t workspace_bytes, int* dev_status, void* stream) {
  if (k_scale == nullptr || v_scale == nullptr) return PGQA_EINVAL;
  return prefill_call(out, lse, q, num_tokens, k_cache, v_cache, block_tables,
                      max_blocks_per_seq, cu_seqlens_q, seq_lens_k, num_seqs, max_seqlen_q,
                      seq_lens_k ? max_seqlen_k : max_seqlen_q, num_q_heads, num_kv_heads,
                      head_dim, num_blocks, block_size, scale, PGQA_DTYPE_E4M3, k_scale, v_scale,
                      workspace, workspace_bytes, dev_status, stream);
}

}  // extern "C"
