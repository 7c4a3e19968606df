// Paged decode for callers that cannot allocate device memory.
//
// Some callers of this library have no way to obtain device scratch memory: a
// serving engine that sizes its paged KV pool to fill the GPU's free memory at
// start-up (so any later cudaMalloc fails), or a plugin hosted inside another
// framework whose device memory belongs to that framework's allocator (so the
// plugin has no allocator to ask). pgqa_paged_attention_decode_noalloc serves
// them: it is the same decode as pgqa_paged_attention_decode, but its split-K
// scratch lives in a fixed array owned by this library.
//
//  - The scratch is a file-scope device array of PGQA_NOALLOC_SCRATCH_BYTES. The CUDA
//    runtime loads this file's module, and with it the array, on a device when the
//    array is first looked up there (lazy module loading, the default), or at context
//    creation when modules load eagerly; from then on the device holds it until the
//    process exits. The decode kernels' module is loaded the same way.
//  - Per-device set-up: host code cannot use the array's name as a device address (on
//    the host it names a host-side stand-in), so the device address is looked up with
//    cudaGetSymbolAddress once per device, with that device current, and the decode
//    kernels are loaded and given their shared-memory limit. The first call on a
//    device does this; a call with num_seqs == 0 does only this and launches nothing,
//    so a caller can make it before it fills the device's free memory and before any
//    stream capture. Later calls allocate nothing.
//  - Every call shares the array, which keeps the previous call's contents. The
//    split-merge ticket counters must start at zero, so each call clears them with
//    cudaMemsetAsync on its stream before the kernel runs. Calls that overlap on
//    the GPU (different streams, or different host threads) race on the array.
//  - Arguments are checked on the host before anything is enqueued: a call that
//    returns an error has queued no clear and no kernel.
//  - Nothing here calls cudaMalloc, cudaFree or any allocating routine.
#include <cuda_runtime.h>

#include <mutex>

#include "host.h"

namespace pgqa {
namespace {

constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_decode_scratch[PGQA_NOALLOC_SCRATCH_BYTES];

std::mutex g_scratch_mu;
void* g_scratch_addr[kMaxDevices] = {nullptr};

// Device address of g_decode_scratch on the current device, looked up once per device
// together with loading the decode kernels there.
pgqa_status_t scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PGQA_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return PGQA_ECUDA;
    if (!decode_prepare()) return PGQA_ECUDA;
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return PGQA_OK;
}

}  // namespace
}  // namespace pgqa

extern "C" pgqa_status_t pgqa_paged_attention_decode_noalloc(
    void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
    int block_size, float scale, int cache_dtype, const float* k_scale, const float* v_scale,
    int max_context_len, int* dev_status, void* stream) {
  const pgqa_status_t valid = pgqa::decode_validate(
      out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, context_lens, num_seqs,
      num_q_heads, num_kv_heads, head_dim, num_blocks, block_size, scale, cache_dtype, k_scale,
      v_scale, max_context_len, nullptr, nullptr);
  if (valid != PGQA_OK) return valid;
  void* scratch = nullptr;
  if (num_seqs == 0) return pgqa::scratch_address(&scratch);  // the per-device set-up only
  const int sms = pgqa::num_sms_current_device();
  if (sms <= 0) return PGQA_ECUDA;
  const pgqa::DecodePlan plan =
      pgqa::decode_plan(num_seqs, num_kv_heads, head_dim, cache_dtype, sms);
  if (plan.bytes > PGQA_NOALLOC_SCRATCH_BYTES) return PGQA_ENOWORKSPACE;
  const pgqa_status_t rc = pgqa::scratch_address(&scratch);
  if (rc != PGQA_OK) return rc;
  // the ticket counters occupy [0, lse_off)
  if (cudaMemsetAsync(scratch, 0, plan.lse_off, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return PGQA_ECUDA;
  return pgqa_paged_attention_decode(out, lse, q, k_cache, v_cache, block_tables,
                                     max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                                     num_kv_heads, head_dim, num_blocks, block_size, scale,
                                     cache_dtype, k_scale, v_scale, max_context_len, scratch,
                                     PGQA_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
