// Causal variable-length prefill over the paged KV cache, on the tcgen05 tensor
// cores (sm_103a).
//
// Computes, for every sequence i (tokens cu_seqlens[i] .. cu_seqlens[i+1]-1), query
// head hq and position p, softmax(scale * q_p K^T) V over keys 0..p of sequence i,
// read through its block table, and lse = ln sum exp(score): the varlen, causal
// call of the rkmt.cn article (sec. 2.4) over the paged cache of its sec. 3.1, with
// the attention steps of "LLaMA structure and inference performance" (sec. 3.1) and
// repeat_kv as the index map kv_head = hq / G (sec. 2.1).
//
// One CTA computes one 128-query tile of one query head (FlashAttention-style
// online softmax over 128-key tiles, never materialising the full score matrix):
//  - warp 4 (TMA): Q tile once; then K and V tiles of 128 keys, each gathered as 8
//    pages of 16 rows with 2-D tensor-map loads (128-byte swizzle) into a 2-stage
//    ring. Pages past the sequence end are loaded from past the end of the cache
//    view, which TMA fills with zeros.
//  - warp 5 (MMA, one thread): S_j = Q K_j^T into one of two TMEM buffers
//    (tcgen05.mma, M = N = 128, K-major operands), issued one tile ahead; then
//    O += P_j V_j into TMEM (V MN-major), signalling completion via tcgen05.commit.
//  - warps 0-3 (softmax; thread = query row = TMEM lane): read S_j from TMEM, apply
//    the causal mask, keep a running max, rescale O in TMEM only when the max grew
//    by more than 2^8 (exact either way: P and l use the same reference max), write
//    P = 2^(s - m) as bf16 into shared memory in the MMA's swizzled layout; finally
//    O / l -> bf16 out and lse.
//  - Causal tile skipping: query tile t visits key tiles 0..t only; only tile t
//    carries the diagonal mask.
// All waits are bounded (a wait that gives up records PGQA_ETIMEOUT).
#include <cuda_bf16.h>

#include "host.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pgqa {
namespace {

constexpr int kBlockM = 128;  // query rows per CTA
constexpr int kBlockN = 128;  // keys per tile
constexpr int kThreads = 192;
constexpr int kWarpTma = 4, kWarpMma = 5;
constexpr uint32_t kTmemCols = 512;  // S buffers at columns 0 and 128, O at 256
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units

template <int D>
struct PCfg {
  static constexpr int kSub = D / 64;          // 128-byte (64-element) column blocks
  static constexpr int kTile = 128 * D * 2;    // [128 rows][D] bf16
  static constexpr int kQ = 0;
  static constexpr int kKV = kTile;            // stage s: K at kKV + 2 s kTile, V after it
  static constexpr int kP = kKV + 4 * kTile;   // [128 rows][128 keys] bf16
  static constexpr int kBar = kP + 128 * 128 * 2;
  static constexpr int kUsed = kBar + 128;
  // at least 120 KB, so that a single CTA (which owns all 512 TMEM columns) fits per SM
  static constexpr int kSmem = (1024 + kUsed) > 122880 ? (1024 + kUsed) : 122880;
};

struct PrefillParams {
  __nv_bfloat16* out;
  float* lse;
  const int32_t* cu_seqlens;
  const int32_t* block_tables;
  int* dev_status;
  int max_blocks_per_seq;
  int num_seqs, num_tokens, max_seqlen;
  int num_q_heads, num_kv_heads, group;
  int num_blocks;
  int n_qtiles;
  int oob_row;  // a row index past the end of the cache view (TMA fills zeros)
  float scale_log2;
};

__device__ __forceinline__ void named_bar_sync(int id, int n) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(n) : "memory");
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) paged_prefill_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  using C = PCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kQ;
  uint8_t* sP = smem + C::kP;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* kv_full = bars + 1;   // [2]
  uint64_t* kv_empty = bars + 3;  // [2]
  uint64_t* s_full = bars + 5;    // [2]
  uint64_t* p_full = bars + 7;
  uint64_t* o_full = bars + 8;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 9);
  int* flags = reinterpret_cast<int*>(bars + 10);  // [0] bad block id, [1] timeout

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int seq = blockIdx.x % p.num_seqs;
  const int hq = blockIdx.x / p.num_seqs;
  const int t = p.n_qtiles - 1 - static_cast<int>(blockIdx.y);  // longest tiles first
  const int start = __ldg(p.cu_seqlens + seq);
  const int L = __ldg(p.cu_seqlens + seq + 1) - start;
  if (t == p.n_qtiles - 1 && tid == 0) {
    const bool bad_len = L < 0 || L > p.max_seqlen || (L + 15) / 16 > p.max_blocks_per_seq ||
                         start < 0 || start + L > p.num_tokens ||
                         (seq == p.num_seqs - 1 && start + L != p.num_tokens);
    if (bad_len) record_status(p.dev_status, PGQA_EINVAL);
  }
  if (L <= 0 || t * kBlockM >= L) return;
  if (L > p.max_seqlen || (L + 15) / 16 > p.max_blocks_per_seq || start < 0 ||
      start + L > p.num_tokens)
    return;  // reported above; nothing sensible to compute
  const int h = hq / p.group;
  const int nkt = t + 1;                       // key tiles 0..t (causal skipping)
  const int rows = min(kBlockM, L - t * kBlockM);

  if (tid == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
      mbar_init(&s_full[s], 1);
    }
    mbar_init(p_full, 4 * 32);
    mbar_init(o_full, 1);
    flags[0] = flags[1] = 0;
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------- TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
      mbar_arrive_expect_tx(q_full, C::kTile);
#pragma unroll
      for (int sub = 0; sub < C::kSub; ++sub)
        tma_load_3d(sQ + sub * 16384, &qmap, q_full, sub * 64, hq, start + t * kBlockM);
    }
    const int32_t* bt = p.block_tables + static_cast<size_t>(seq) * p.max_blocks_per_seq;
    bool ok = true;
    for (int j = 0; j < nkt && ok; ++j) {
      const int st = j & 1, use = j >> 1;
      int y = p.oob_row;
      if (lane < 8) {
        const int lp = j * 8 + lane;  // logical page
        if (lp * 16 < L) {
          const int32_t pbn = __ldg(bt + lp);
          if (pbn < 0 || pbn >= p.num_blocks)
            flags[0] = 1;
          else
            y = (pbn * p.num_kv_heads + h) * 16;
        }
      }
      if (lane == 0) {
        if (use > 0 && !mbar_wait(&kv_empty[st], (use - 1) & 1)) {
          record_status(p.dev_status, PGQA_ETIMEOUT);
          flags[1] = 1;
          ok = false;
        } else {
          mbar_arrive_expect_tx(&kv_full[st], 2 * C::kTile);
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (ok && lane < 8) {
        uint8_t* sK = smem + C::kKV + st * 2 * C::kTile;
        uint8_t* sV = sK + C::kTile;
#pragma unroll
        for (int sub = 0; sub < C::kSub; ++sub) {
          tma_load_2d(sK + sub * 16384 + lane * 2048, &kmap, &kv_full[st], sub * 64, y);
          tma_load_2d(sV + sub * 16384 + lane * 2048, &vmap, &kv_full[st], sub * 64, y);
        }
      }
      __syncwarp();
    }
    named_bar_sync(1, 5 * 32);  // bad-index flag published to the softmax warps
    if (lane == 0) {
      // no TMA write may land after the CTA exits: wait for the last fill of each stage
      if (!mbar_wait(q_full, 0)) record_status(p.dev_status, PGQA_ETIMEOUT);
      for (int st = 0; st < 2 && st < nkt; ++st) {
        const int last_j = st + ((nkt - 1 - st) / 2) * 2;
        if (!mbar_wait(&kv_full[st], (last_j >> 1) & 1)) record_status(p.dev_status, PGQA_ETIMEOUT);
      }
    }
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, kBlockN, false);
      const uint32_t id_o = idesc_bf16_f32(128, D, true);
      const uint32_t q_addr = smem_u32(sQ), p_addr = smem_u32(sP);
      bool ok = mbar_wait(q_full, 0);
      tc_fence_after();
      auto issue_s = [&](int j) -> bool {
        const int st = j & 1;
        if (!mbar_wait(&kv_full[st], (j >> 1) & 1)) return false;
        tc_fence_after();
        const uint32_t k_addr = smem_u32(smem + C::kKV + st * 2 * C::kTile);
        const uint32_t d_tmem = tmem + static_cast<uint32_t>(st * 128);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_f16_ss(d_tmem, smem_desc_sw128(q_addr + off, 16, 1024),
                      smem_desc_sw128(k_addr + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[st]);
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; j < nkt && ok; ++j) {
        if (j + 1 < nkt && !issue_s(j + 1)) {
          ok = false;
          break;
        }
        if (!mbar_wait(p_full, j & 1)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const int st = j & 1;
        const uint32_t v_addr = smem_u32(smem + C::kKV + st * 2 * C::kTile + C::kTile);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_f16_ss(tmem + 256, smem_desc_sw128(p_addr + poff, 16, 1024),
                      smem_desc_sw128(v_addr + kk * 2048, 16384, 1024), id_o,
                      (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(o_full);
        umma_commit(&kv_empty[st]);
      }
      if (!ok) {
        record_status(p.dev_status, PGQA_ETIMEOUT);
        flags[1] = 1;
      }
    }
  } else {
    // ------------------------------------------------------------- softmax rows
    const int r = warp * 32 + lane;          // query row in the tile = TMEM lane
    const int qpos = t * kBlockM + r;        // position in the sequence
    const int lim = min(qpos, L - 1);        // last key this row attends
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(warp * 32) << 16);
    float m_ref = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int st = j & 1;
      // tcgen05.ld / st are warp-collective: every decision before them is warp-uniform
      if (!__all_sync(0xffffffffu, mbar_wait(&s_full[st], (j >> 1) & 1))) {
        ok = false;
        break;
      }
      tc_fence_after();
      float s[kBlockN];
#pragma unroll
      for (int c = 0; c < kBlockN / 32; ++c) {
        uint32_t rr[32];
        tmem_ld32(lane_base + st * 128 + c * 32, rr);
#pragma unroll
        for (int k = 0; k < 32; ++k) s[c * 32 + k] = __uint_as_float(rr[k]);
      }
      const int kbase = j * kBlockN;
      float mx = -INFINITY;
#pragma unroll
      for (int k = 0; k < kBlockN; ++k) {
        const float v = kbase + k <= lim ? s[k] * p.scale_log2 : -INFINITY;
        s[k] = v;
        mx = fmaxf(mx, v);
      }
      if (j > 0) {  // P_{j-1} V_{j-1} done: O is stable and the P buffer is free
        if (!__all_sync(0xffffffffu, mbar_wait(o_full, (j - 1) & 1))) {
          ok = false;
          break;
        }
        tc_fence_after();
      }
      const bool grow = mx > m_ref + kRescaleThreshold;
      const float alpha = grow ? ex2(m_ref - mx) : 1.f;  // 0 while m_ref = -inf
      if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld32(lane_base + 256 + c * 32, o);
#pragma unroll
          for (int k = 0; k < 32; ++k) o[k] = __float_as_uint(__uint_as_float(o[k]) * alpha);
          tmem_st32(lane_base + 256 + c * 32, o);
        }
        tmem_wait_st();
      }
      if (grow) {
        l *= alpha;
        m_ref = mx;
      }
      // P = 2^(s - m_ref) as bf16, row r of the K-major, 128-byte-swizzled A operand
      float sum = 0.f;
#pragma unroll
      for (int c16 = 0; c16 < kBlockN / 8; ++c16) {
        float e[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          e[k] = ex2(s[c16 * 8 + k] - m_ref);
          sum += e[k];
        }
        const uint4 pk = make_uint4(pack_bf16(e[0], e[1]), pack_bf16(e[2], e[3]),
                                    pack_bf16(e[4], e[5]), pack_bf16(e[6], e[7]));
        *reinterpret_cast<uint4*>(sP + (c16 >> 3) * 16384 + swz128(r, c16 & 7)) = pk;
      }
      l += sum;
      // V rows past the sequence end may hold anything (NaN included): zero them so
      // that P = 0 there contributes exactly nothing
      if (kbase + r >= L) {
        uint8_t* sV = smem + C::kKV + st * 2 * C::kTile + C::kTile;
#pragma unroll
        for (int sub = 0; sub < C::kSub; ++sub) {
          uint4* row = reinterpret_cast<uint4*>(sV + sub * 16384 + r * 128);
#pragma unroll
          for (int c = 0; c < 8; ++c) row[c] = make_uint4(0, 0, 0, 0);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(p_full);
    }
    named_bar_sync(1, 5 * 32);
    if (ok && !__all_sync(0xffffffffu, mbar_wait(o_full, (nkt - 1) & 1))) ok = false;
    tc_fence_after();
    if (!ok) {
      record_status(p.dev_status, PGQA_ETIMEOUT);
      flags[1] = 1;
    }
    const bool bad = flags[0] != 0 || !ok;
    if (flags[0] != 0 && r == 0) record_status(p.dev_status, PGQA_EBADINDEX);
    // every lane loads (warp-collective); only rows inside the sequence are stored
    const bool store = r < rows;
    const size_t orow = static_cast<size_t>(start + (store ? qpos : 0)) * p.num_q_heads + hq;
    uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
    const float inv = 1.f / l;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      if (ok) {
        tmem_ld32(lane_base + 256 + c * 32, o);
      } else {
#pragma unroll
        for (int k = 0; k < 32; ++k) o[k] = 0u;
      }
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        uint4 v = make_uint4(0, 0, 0, 0);
        if (!bad) {
          const float* f = reinterpret_cast<const float*>(o) + k * 8;
          v = make_uint4(pack_bf16(f[0] * inv, f[1] * inv), pack_bf16(f[2] * inv, f[3] * inv),
                         pack_bf16(f[4] * inv, f[5] * inv), pack_bf16(f[6] * inv, f[7] * inv));
        }
        if (store) dst[c * 4 + k] = v;
      }
    }
    if (store && p.lse) p.lse[orow] = bad ? -INFINITY : (m_ref + log2f(l)) * kLn2;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kWarpMma) tmem_dealloc(tmem, kTmemCols);
}

template <int D>
pgqa_status_t launch_prefill_variant(const PrefillArgs& a) {
  using C = PCfg<D>;
  const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * 16;
  CUtensorMap qmap, kmap, vmap;
  if (!tensor_map_3d(&qmap, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, a.num_q_heads,
                     a.num_tokens, static_cast<uint64_t>(D) * 2,
                     static_cast<uint64_t>(a.num_q_heads) * D * 2, 64, 1, kBlockM,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tensor_map_2d(&kmap, a.k_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, rows, D * 2, 64, 16,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tensor_map_2d(&vmap, a.v_cache, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, rows, D * 2, 64, 16,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return PGQA_ECUDA;
  if (!smem_attr_ready(reinterpret_cast<const void*>(paged_prefill_kernel<D>), C::kSmem))
    return PGQA_ECUDA;
  PrefillParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.cu_seqlens = a.cu_seqlens;
  p.block_tables = a.block_tables;
  p.dev_status = a.dev_status;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_tokens = a.num_tokens;
  p.max_seqlen = a.max_seqlen;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.n_qtiles = (a.max_seqlen + kBlockM - 1) / kBlockM;
  p.oob_row = static_cast<int>(rows);
  p.scale_log2 = a.scale * kLog2e;
  dim3 grid(a.num_seqs * a.num_q_heads, p.n_qtiles);
  paged_prefill_kernel<D><<<grid, kThreads, C::kSmem, a.stream>>>(qmap, kmap, vmap, p);
  return cudaPeekAtLastError() == cudaSuccess ? PGQA_OK : PGQA_ECUDA;
}

}  // namespace

pgqa_status_t launch_paged_prefill(const PrefillArgs& a) {
  if (a.head_dim == 128) return launch_prefill_variant<128>(a);
  if (a.head_dim == 64) return launch_prefill_variant<64>(a);
  return PGQA_EUNSUPPORTED;
}

}  // namespace pgqa
