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
//  - The scratch is a file-scope device array of PGQA_NOALLOC_SCRATCH_BYTES. Every
//    GPU that loads the library holds it until the process exits.
//  - Host code cannot use the array's name as a device address (on the host it
//    names a host-side stand-in), so the device address is looked up with
//    cudaGetSymbolAddress once per device, with that device current, on the first
//    call made on that device. Make that first call before any stream capture.
//  - Every call shares the array, which keeps the previous call's contents. The
//    split-merge ticket counters must start at zero, so each call clears them with
//    cudaMemsetAsync on its stream before the kernel runs. Calls that overlap on
//    the GPU (different streams, or different host threads) race on the array.
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

// Device address of g_decode_scratch on the current device (looked up once).
pgqa_status_t scratch_address(void** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PGQA_ECUDA;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (g_scratch_addr[dev] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_decode_scratch) != cudaSuccess || p == nullptr)
      return PGQA_ECUDA;
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
  if (num_seqs < 0 || num_kv_heads <= 0 || head_dim <= 0 || block_size <= 0 ||
      max_context_len < 0)
    return PGQA_EINVAL;
  size_t need = 0;
  size_t counter_bytes = 0;
  if (num_seqs > 0) {
    const int sms = pgqa::num_sms_current_device();
    if (sms <= 0) return PGQA_ECUDA;
    const pgqa::DecodePlan plan =
        pgqa::decode_plan(num_seqs, num_kv_heads, head_dim, cache_dtype, sms);
    need = plan.bytes;
    counter_bytes = plan.lse_off;  // the ticket counters occupy [0, lse_off)
  }
  if (need > PGQA_NOALLOC_SCRATCH_BYTES) return PGQA_ENOWORKSPACE;
  void* scratch = nullptr;
  if (need > 0) {
    const pgqa_status_t rc = pgqa::scratch_address(&scratch);
    if (rc != PGQA_OK) return rc;
    if (cudaMemsetAsync(scratch, 0, counter_bytes, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
      return PGQA_ECUDA;
  }
  return pgqa_paged_attention_decode(out, lse, q, k_cache, v_cache, block_tables,
                                     max_blocks_per_seq, context_lens, num_seqs, num_q_heads,
                                     num_kv_heads, head_dim, num_blocks, block_size, scale,
                                     cache_dtype, k_scale, v_scale, max_context_len, scratch,
                                     need > 0 ? PGQA_NOALLOC_SCRATCH_BYTES : 0, dev_status,
                                     stream);
}
