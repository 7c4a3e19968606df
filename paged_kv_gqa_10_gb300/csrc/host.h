// Host-side plumbing shared by the translation units of libpgqa: TMA descriptor
// encoding (through the driver entry point, cached by address and shape), device
// properties, and the launchers each kernel file exports to the C ABI layer.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/pgqa.h"

namespace pgqa {

// Row-major 2-D view [rows][inner] of `base` with a row pitch of row_bytes, tiled
// in boxes of box_inner x box_rows elements. Returns false if the driver refuses.
bool tensor_map_2d(CUtensorMap* out, const void* base, CUtensorMapDataType dtype, uint64_t inner,
                   uint64_t rows, uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows,
                   CUtensorMapSwizzle swizzle);

// 3-D view [d2][d1][d0] with pitches (bytes) for dims 1 and 2.
bool tensor_map_3d(CUtensorMap* out, const void* base, CUtensorMapDataType dtype, uint64_t d0,
                   uint64_t d1, uint64_t d2, uint64_t pitch1, uint64_t pitch2, uint32_t box0,
                   uint32_t box1, uint32_t box2, CUtensorMapSwizzle swizzle);

// Multiprocessor count of the current device (cached per device); 0 on error.
int num_sms_current_device();

// Raises a kernel's dynamic shared memory limit to `bytes` on the current device
// (once per device and kernel). Returns false if the runtime refuses.
bool smem_attr_ready(const void* kernel, int bytes);

// Launches `kernel` with programmatic stream serialization: it may be scheduled while
// the stream's previous kernel runs, and waits for it in grid_dependency_wait().
template <typename... Params, typename... Args>
cudaError_t launch_after_previous(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                                  cudaStream_t stream, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<Args&&>(args)...);
}

// ----------------------------------------------------------- launchers

pgqa_status_t launch_kv_cache_write(const void* key, const void* value,
                                    const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                    int head_dim, void* k_cache, void* v_cache, int num_blocks,
                                    int block_size, int cache_dtype, const float* k_scale,
                                    const float* v_scale, int* dev_status, cudaStream_t stream);

pgqa_status_t launch_kv_gather(const void* k_cache, const void* v_cache, int cache_dtype,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int num_kv_heads,
                               int head_dim, int num_blocks, int block_size, int max_context_len,
                               void* k_out, void* v_out, int* dev_status, cudaStream_t stream);

struct DecodeArgs {
  void* out;
  float* lse;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* context_lens;
  int num_seqs, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size;
  float scale;
  int cache_dtype;
  const float* k_scale;
  const float* v_scale;
  int max_context_len;
  int window;  // > 0: only the last `window` keys of each context are attended
  int q_len;   // new tokens per sequence (1: decode; more: multi-token decode, q is
               // [num_seqs][q_len][num_q_heads][head_dim] and token t sees keys
               // 0 .. L - q_len + t)
  // fused append (both null: none): the new token's K/V rows [num_seqs][Hkv][D] bf16,
  // written at position context_len - 1 of each sequence before it is attended
  const void* new_key;
  const void* new_value;
  void* workspace;
  size_t workspace_bytes;
  int* dev_status;
  cudaStream_t stream;
};

// Grid and workspace layout of paged decode: `grid` CTAs, each owning an equal
// share of all pages; the workspace holds one ticket counter per (sequence,
// kv-head) and two partial-result slots per CTA.
struct DecodePlan {
  int grid;
  int row_tiles;  // 8-row tiles of query rows per unit: 1, or 4 (the row-split form)
  size_t counters_off, lse_off, o_off, bytes;
};
// 8-row tiles the decode kernel holds for q_len x group query rows per unit: 1 (up to 8
// rows, one tile per warp, warps splitting the pages), 4 (up to 32 rows, the row-split
// form: one tile per consumer warp, every warp reading every page), or 0 when the decode
// kernel does not take that many
int decode_row_tiles(int q_len, int group);
int decode_ctas_per_sm(int head_dim, int cache_dtype, int row_tiles = 1);
DecodePlan decode_plan(int num_seqs, int num_kv_heads, int head_dim, int cache_dtype,
                       int num_sms, int row_tiles = 1);

pgqa_status_t launch_paged_decode(const DecodeArgs& a, const DecodePlan& plan);

// Host-side checks of a decode call's arguments, everything but the workspace (the
// decode entry points return this status before anything is enqueued). key / value:
// the fused append's new rows, both null without it.
pgqa_status_t decode_validate(const void* out, const void* q, const void* k_cache,
                              const void* v_cache, const int32_t* block_tables,
                              int max_blocks_per_seq, const int32_t* context_lens, int num_seqs,
                              int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
                              int block_size, float scale, int cache_dtype, const float* k_scale,
                              const float* v_scale, int max_context_len, const void* key,
                              const void* value);

// Limit of the decode kernels' bounded waits while they stream (the default 2 s, or
// what pgqa_set_decode_wait_limit_ns set); read at each launch.
unsigned long long decode_wait_limit_ns();
void set_decode_wait_limit_ns(unsigned long long ns);

// Loads the decode kernels on the current device and sets their shared-memory limits
// (what a first decode launch would otherwise do). False if the runtime refuses.
bool decode_prepare();

struct PrefillArgs {
  void* out;
  float* lse;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* block_tables;
  int max_blocks_per_seq;
  const int32_t* cu_seqlens;  // null: every sequence has max_seqlen new tokens, in order
  const int32_t* seq_lens_k;  // cached tokens per sequence, or null (no cached prefix)
  int max_seqlen_k;
  void* workspace;  // >= prefill_workspace_bytes(), zero before first use
  int num_tokens;
  int num_seqs, max_seqlen, num_q_heads, num_kv_heads, head_dim, num_blocks, block_size;
  float scale;
  int cache_dtype;        // PGQA_DTYPE_BF16 or PGQA_DTYPE_E4M3
  const float* k_scale;   // [num_kv_heads], E4M3 only
  const float* v_scale;
  int* dev_status;
  cudaStream_t stream;
};

pgqa_status_t launch_paged_prefill(const PrefillArgs& a);
// ticket counters (256 B) + the item tables (sorted sequences, per-level counts
// and offsets) of up to 4096 sequences and 2048 tile pairs
constexpr size_t kPrefillWorkspaceBytes = 256 + (4096 + 2 * 2048) * 4;
int prefill_max_seqs();    // sequences per prefill call
int prefill_max_seqlen();  // tokens of the longest sequence

}  // namespace pgqa
