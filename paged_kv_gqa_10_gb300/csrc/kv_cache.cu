// KV-cache scatter (new K/V rows into their slots, optionally quantised to E4M3)
// and the page gather used to test block-table addressing.
//
// kv_cache_write follows the in-place cache update of "LLM inference surgery
// log" (xdnf.cn) sec. 3.1: the pool is pre-allocated and each new token's K/V is
// written into the row its slot names (slot = physical block * block_size + row,
// the page-table addressing of the rkmt.cn article, sec. 3.1).
//
// Both kernels are pure HBM streams: one thread moves 16 bytes of input (8 bf16
// elements), consecutive threads cover consecutive bytes of one (token, head)
// row, so every warp reads and writes whole 32-byte sectors.
#include "host.h"
#include "ptx.cuh"

namespace pgqa {
namespace {

template <bool kFp8>
__global__ void __launch_bounds__(256) kv_cache_write_kernel(
    const uint4* __restrict__ key, const uint4* __restrict__ value,
    const int64_t* __restrict__ slot_mapping, int num_tokens, int num_kv_heads, int head_dim,
    void* __restrict__ k_cache, void* __restrict__ v_cache, int num_blocks, int block_size,
    const float* __restrict__ k_scale, const float* __restrict__ v_scale, int* dev_status) {
  grid_launch_dependents();  // a following attention kernel may get its CTAs in place now
  grid_dependency_wait();    // the stream's previous kernel (inputs, cache readers) is done
  const int vecs = head_dim / 8;  // 16-byte input vectors per (token, head) row
  const int64_t total = static_cast<int64_t>(num_tokens) * num_kv_heads * vecs;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(i % vecs);
    const int64_t th = i / vecs;
    const int h = static_cast<int>(th % num_kv_heads);
    const int64_t t = th / num_kv_heads;
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    const int64_t block = slot / block_size;
    const int row = static_cast<int>(slot % block_size);
    if (block >= num_blocks) {
      record_status(dev_status, PGQA_EBADINDEX);
      continue;
    }
    // element offset of (block, h, row, 8v) in [NB][Hkv][bs][D]
    const size_t dst = ((static_cast<size_t>(block) * num_kv_heads + h) * block_size + row) *
                           static_cast<size_t>(head_dim) + static_cast<size_t>(v) * 8;
    const uint4 kx = __ldg(key + i);
    const uint4 vx = __ldg(value + i);
    if constexpr (!kFp8) {
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(k_cache) + dst) = kx;
      *reinterpret_cast<uint4*>(static_cast<uint16_t*>(v_cache) + dst) = vx;
    } else {
      const float ks = __ldg(k_scale + h), vs = __ldg(v_scale + h);
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(k_cache) + dst) = e4m3_quant8(kx, ks);
      *reinterpret_cast<uint2*>(static_cast<uint8_t*>(v_cache) + dst) = e4m3_quant8(vx, vs);
    }
  }
}

// The same scatter with the index arithmetic in 32 bits and shifts: kVecs 16-byte input
// vectors per row (head_dim 128 or 64), fewer than 2^31 (token, head) rows, and a
// block size that is a power of two (bs_shift = log2 of it). The general form above
// spends most of its issue slots on 64-bit divisions; this one is a plain stream.
template <bool kFp8, int kVecs>
__global__ void __launch_bounds__(256) kv_cache_write_rows_kernel(
    const uint4* __restrict__ key, const uint4* __restrict__ value,
    const int64_t* __restrict__ slot_mapping, int num_tokens, int num_kv_heads,
    void* __restrict__ k_cache, void* __restrict__ v_cache, int num_blocks, int bs_shift,
    const float* __restrict__ k_scale, const float* __restrict__ v_scale, int* dev_status) {
  static_assert(kVecs == 8 || kVecs == 16, "head_dim 64 or 128");
  constexpr int kVecShift = kVecs == 16 ? 4 : 3;
  grid_launch_dependents();
  grid_dependency_wait();
  const uint32_t hkv = static_cast<uint32_t>(num_kv_heads);
  const int64_t total = (static_cast<int64_t>(num_tokens) * num_kv_heads) << kVecShift;
  const int64_t bs_mask = (int64_t{1} << bs_shift) - 1;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const uint32_t row = static_cast<uint32_t>(i >> kVecShift);  // (token, head)
    const uint32_t v = static_cast<uint32_t>(i) & (kVecs - 1);
    const uint32_t t = row / hkv, h = row - t * hkv;
    const int64_t slot = __ldg(slot_mapping + t);
    if (slot < 0) continue;
    const int64_t block = slot >> bs_shift;
    if (block >= num_blocks) {
      record_status(dev_status, PGQA_EBADINDEX);
      continue;
    }
    // 16-byte vector of (block, h, row, 8v) in [NB][Hkv][bs][D]
    const size_t dst = (((static_cast<size_t>(block) * hkv + h) << bs_shift) + (slot & bs_mask))
                           * kVecs + v;
    const uint4 kx = __ldg(key + i);
    const uint4 vx = __ldg(value + i);
    if constexpr (!kFp8) {
      reinterpret_cast<uint4*>(k_cache)[dst] = kx;
      reinterpret_cast<uint4*>(v_cache)[dst] = vx;
    } else {
      const float ks = __ldg(k_scale + h), vs = __ldg(v_scale + h);
      reinterpret_cast<uint2*>(k_cache)[dst] = e4m3_quant8(kx, ks);
      reinterpret_cast<uint2*>(v_cache)[dst] = e4m3_quant8(vx, vs);
    }
  }
}

// out[b][h][j][:] = cache[block_tables[b][j / bs]][h][j % bs][:] for j < L_b, else 0.
// Each thread moves one 16-byte vector; `vecs` vectors per row.
__global__ void __launch_bounds__(256) kv_gather_kernel(
    const uint4* __restrict__ k_cache, const uint4* __restrict__ v_cache,
    const int32_t* __restrict__ block_tables, int max_blocks_per_seq,
    const int32_t* __restrict__ context_lens, int num_seqs, int num_kv_heads, int vecs,
    int num_blocks, int block_size, int max_context_len, uint4* __restrict__ k_out,
    uint4* __restrict__ v_out, int* dev_status) {
  const int64_t total =
      static_cast<int64_t>(num_seqs) * num_kv_heads * max_context_len * vecs;
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int v = static_cast<int>(i % vecs);
    int64_t r = i / vecs;
    const int j = static_cast<int>(r % max_context_len);
    r /= max_context_len;
    const int h = static_cast<int>(r % num_kv_heads);
    const int b = static_cast<int>(r / num_kv_heads);
    const int L = __ldg(context_lens + b);
    uint4 kx = make_uint4(0, 0, 0, 0), vx = kx;
    if (j < L) {
      const int lpn = j / block_size;
      const int32_t pbn =
          lpn < max_blocks_per_seq ? __ldg(block_tables + static_cast<int64_t>(b) * max_blocks_per_seq + lpn) : -1;
      if (pbn < 0 || pbn >= num_blocks || L > max_context_len) {
        record_status(dev_status, PGQA_EBADINDEX);
      } else {
        const size_t src =
            ((static_cast<size_t>(pbn) * num_kv_heads + h) * block_size + j % block_size) * vecs + v;
        kx = __ldg(k_cache + src);
        vx = __ldg(v_cache + src);
      }
    }
    k_out[i] = kx;
    v_out[i] = vx;
  }
}

int grid_for(int64_t work, int threads) {
  int64_t blocks = (work + threads - 1) / threads;
  const int sms = num_sms_current_device();
  const int64_t cap = static_cast<int64_t>(sms > 0 ? sms : 148) * 32;
  if (blocks > cap) blocks = cap;
  return static_cast<int>(blocks < 1 ? 1 : blocks);
}

}  // namespace

pgqa_status_t launch_kv_cache_write(const void* key, const void* value,
                                    const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                    int head_dim, void* k_cache, void* v_cache, int num_blocks,
                                    int block_size, int cache_dtype, const float* k_scale,
                                    const float* v_scale, int* dev_status, cudaStream_t stream) {
  const int64_t work = static_cast<int64_t>(num_tokens) * num_kv_heads * (head_dim / 8);
  if (work == 0) return PGQA_OK;
  const int grid = grid_for(work, 256);
  const bool pow2 = (block_size & (block_size - 1)) == 0;
  const bool rows32 = static_cast<int64_t>(num_tokens) * num_kv_heads < (int64_t{1} << 31);
  if (pow2 && rows32 && (head_dim == 128 || head_dim == 64)) {
    int bs_shift = 0;
    while ((1 << bs_shift) < block_size) ++bs_shift;
    const bool fp8 = cache_dtype == PGQA_DTYPE_E4M3;
    auto kern = head_dim == 128 ? (fp8 ? kv_cache_write_rows_kernel<true, 16>
                                       : kv_cache_write_rows_kernel<false, 16>)
                                : (fp8 ? kv_cache_write_rows_kernel<true, 8>
                                       : kv_cache_write_rows_kernel<false, 8>);
    const cudaError_t e = launch_after_previous(
        kern, dim3(grid), dim3(256), 0, stream, static_cast<const uint4*>(key),
        static_cast<const uint4*>(value), slot_mapping, num_tokens, num_kv_heads, k_cache,
        v_cache, num_blocks, bs_shift, k_scale, v_scale, dev_status);
    if (e != cudaSuccess) return PGQA_ECUDA;
    return cudaPeekAtLastError() == cudaSuccess ? PGQA_OK : PGQA_ECUDA;
  }
  // programmatic launch: the CTAs may be placed while the previous kernel finishes
  const cudaError_t e = launch_after_previous(
      cache_dtype == PGQA_DTYPE_BF16 ? kv_cache_write_kernel<false> : kv_cache_write_kernel<true>,
      dim3(grid), dim3(256), 0, stream, static_cast<const uint4*>(key),
      static_cast<const uint4*>(value), slot_mapping, num_tokens, num_kv_heads, head_dim, k_cache,
      v_cache, num_blocks, block_size, k_scale, v_scale, dev_status);
  if (e != cudaSuccess) return PGQA_ECUDA;
  return cudaPeekAtLastError() == cudaSuccess ? PGQA_OK : PGQA_ECUDA;
}

pgqa_status_t launch_kv_gather(const void* k_cache, const void* v_cache, int cache_dtype,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int num_seqs, int num_kv_heads,
                               int head_dim, int num_blocks, int block_size, int max_context_len,
                               void* k_out, void* v_out, int* dev_status, cudaStream_t stream) {
  const int elem = cache_dtype == PGQA_DTYPE_BF16 ? 2 : 1;
  const int vecs = head_dim * elem / 16;
  const int64_t work = static_cast<int64_t>(num_seqs) * num_kv_heads * max_context_len * vecs;
  if (work == 0) return PGQA_OK;
  kv_gather_kernel<<<grid_for(work, 256), 256, 0, stream>>>(
      static_cast<const uint4*>(k_cache), static_cast<const uint4*>(v_cache), block_tables,
      max_blocks_per_seq, context_lens, num_seqs, num_kv_heads, vecs, num_blocks, block_size,
      max_context_len, static_cast<uint4*>(k_out), static_cast<uint4*>(v_out), dev_status);
  return cudaPeekAtLastError() == cudaSuccess ? PGQA_OK : PGQA_ECUDA;
}

}  // namespace pgqa
