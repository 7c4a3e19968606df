// Causal variable-length prefill over the paged KV cache, on the tcgen05 tensor
// cores (sm_103a).
//
// Computes, for every sequence i (tokens cu_seqlens[i] .. cu_seqlens[i+1]-1), query
// head hq and position p, softmax(scale * q_p K^T) V over keys 0..p of sequence i,
// read through its block table, and lse = ln sum exp(score): the varlen, causal
// call of the rkmt.cn article (sec. 2.4) over the paged cache of its sec. 3.1, with
// the attention steps of "LLaMA structure and inference performance" (sec. 3.1) and
// repeat_kv as the index map kv_head = hq / G (sec. 2.1). FlashAttention-style
// online softmax over 128-key tiles; the full score matrix is never formed.
//
// Work and warp roles
//  - A work item is a pair of consecutive 128-query tiles (A = 2m, B = 2m + 1) of
//    one query head. A persistent grid (one CTA per SM) walks the items longest
//    first, round-robin. Causal tile skipping: tile t visits key tiles 0..t; B
//    exists only if the sequence reaches it.
//  - warp 8 (TMA): checks the item's block ids, loads Q_A and Q_B once, then for
//    each key tile K (2-stage ring) and V (1 stage), each gathered as 8 pages of 16
//    rows with 2-D tensor-map loads (128-byte swizzle). Pages past the sequence end
//    are loaded from past the end of the cache view, which TMA fills with zeros.
//  - warp 9 (MMA, one thread): tcgen05.mma, M = N = 128, f32 accumulators in TMEM:
//    S_X = Q_X K^T for X = A, B and O_X += P_X V (V MN-major). The tile pair
//    ping-pongs: while one tile's softmax runs, the tensor core computes the other
//    tile's S and PV.
//  - warps 0-3 / 4-7 (softmax of tile A / B; thread = query row = TMEM lane): two
//    passes over S in TMEM (max, then exp2), causal mask, O rescaled in TMEM only
//    when the running max grows by more than 2^8 (exact either way: P and l use the
//    same reference max), P = 2^(s - m) as bf16 in shared memory in the MMA's
//    swizzled layout; at the end O / l -> bf16 out and lse.
// All waits are bounded (a wait that gives up records PGQA_ETIMEOUT).
#include <cuda_bf16.h>

#include "host.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pgqa {
namespace {

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // keys per tile
constexpr int kThreads = 320;
constexpr int kWarpTma = 8, kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;  // S_A 0, S_B 128, O_A 256, O_B 384
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units

template <int D>
struct PCfg {
  static constexpr int kSub = D / 64;        // 128-byte (64-element) column blocks
  static constexpr int kTile = 128 * D * 2;  // [128 rows][D] bf16
  static constexpr int kQ = 0;               // Q_A, Q_B
  static constexpr int kK = 2 * kTile;       // K stages 0, 1
  static constexpr int kV = 4 * kTile;       // V
  static constexpr int kP = 5 * kTile;       // P_A, P_B: [128 rows][128 keys] bf16 each
  static constexpr int kBar = kP + 2 * 128 * 128 * 2;
  static constexpr int kSmem = 1024 + kBar + 256;
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
  int n_pairs;      // tile pairs of the longest sequence
  int num_items;    // n_pairs * num_seqs * num_q_heads
  int oob_row;      // a row index past the end of the cache view (TMA fills zeros)
  float scale_log2;
};

// One work item: a pair of query tiles of one (sequence, head).
struct Item {
  int seq, hq, m, start, L;
  bool valid, active_b;
  int nkt;  // key tiles the pair visits
};

__device__ __forceinline__ Item decode_item(const PrefillParams& p, int k) {
  Item it;
  const int sh = p.num_seqs * p.num_q_heads;
  it.m = p.n_pairs - 1 - k / sh;  // longest work first
  const int r = k % sh;
  it.seq = r % p.num_seqs;
  it.hq = r / p.num_seqs;
  it.start = __ldg(p.cu_seqlens + it.seq);
  it.L = __ldg(p.cu_seqlens + it.seq + 1) - it.start;
  const bool len_ok = it.L > 0 && it.L <= p.max_seqlen &&
                      (it.L + 15) / 16 <= p.max_blocks_per_seq && it.start >= 0 &&
                      it.start + it.L <= p.num_tokens;
  it.valid = len_ok && 2 * it.m * kBlockM < it.L;
  it.active_b = (2 * it.m + 1) * kBlockM < it.L;
  it.nkt = it.active_b ? 2 * it.m + 2 : 2 * it.m + 1;
  return it;
}

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
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;   // [2]
  uint64_t* k_empty = bars + 4;  // [2]
  uint64_t* v_full = bars + 6;
  uint64_t* v_empty = bars + 7;
  uint64_t* s_full = bars + 8;   // [2] per tile
  uint64_t* p_full = bars + 10;  // [2]
  uint64_t* o_full = bars + 12;  // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 14);
  int* bad_item = reinterpret_cast<int*>(bars + 15);  // [2], by item parity

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, ncta = gridDim.x;

  // length errors: reported once per sequence, by CTA 0
  if (c == 0) {
    for (int s = tid; s < p.num_seqs; s += kThreads) {
      const int st = __ldg(p.cu_seqlens + s), L = __ldg(p.cu_seqlens + s + 1) - st;
      const bool bad = L < 0 || L > p.max_seqlen || (L + 15) / 16 > p.max_blocks_per_seq ||
                       st < 0 || st + L > p.num_tokens ||
                       (s == p.num_seqs - 1 && st + L != p.num_tokens);
      if (bad) record_status(p.dev_status, PGQA_EINVAL);
    }
  }

  if (tid == 0) {
    mbar_init(q_full, 1);
    // Q buffers are reused once the item's last S MMAs are done (one commit) and all
    // 8 softmax warps have taken the item (one arrival each), so q_full can never
    // run two phases ahead of a softmax warp's wait
    mbar_init(q_empty, 1 + 8);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&k_full[s], 1);
      mbar_init(&k_empty[s], 1);
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4 * 32);
      mbar_init(&o_full[s], 1);
    }
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
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
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    int it = 0, gk = 0, gv = 0;
    bool ok = true;
    for (int k = c; k < p.num_items && ok; k += ncta) {
      const Item w = decode_item(p, k);
      if (!w.valid) continue;
      const int h = w.hq / p.group;
      const int32_t* bt = p.block_tables + static_cast<size_t>(w.seq) * p.max_blocks_per_seq;
      const int npages = (min(w.L, w.nkt * kBlockN) + 15) / 16;
      // block ids of the item, checked before its Q is published
      bool bad = false;
      for (int pg = lane; pg < npages; pg += 32) {
        const int32_t pbn = __ldg(bt + pg);
        bad |= pbn < 0 || pbn >= p.num_blocks;
      }
      bad = __any_sync(0xffffffffu, bad);
      if (lane == 0) {
        if (it > 0 && !mbar_wait(q_empty, (it - 1) & 1)) {
          ok = false;
        } else {
          bad_item[it & 1] = bad;
          if (bad) record_status(p.dev_status, PGQA_EBADINDEX);
          mbar_arrive_expect_tx(q_full, (w.active_b ? 2 : 1) * C::kTile);
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub) {
            tma_load_3d(smem + C::kQ + sub * 16384, &qmap, q_full, sub * 64, w.hq,
                        w.start + 2 * w.m * kBlockM);
            if (w.active_b)
              tma_load_3d(smem + C::kQ + C::kTile + sub * 16384, &qmap, q_full, sub * 64, w.hq,
                          w.start + (2 * w.m + 1) * kBlockM);
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (int j = 0; j < w.nkt && ok; ++j) {
        int y = p.oob_row;
        if (lane < 8) {
          const int lp = j * 8 + lane;  // logical page
          if (lp * 16 < w.L) {
            const int32_t pbn = __ldg(bt + lp);
            if (pbn >= 0 && pbn < p.num_blocks) y = (pbn * p.num_kv_heads + h) * 16;
          }
        }
        // K tile j -> stage gk & 1
        const int ks = gk & 1;
        if (lane == 0) {
          if (gk >= 2 && !mbar_wait(&k_empty[ks], ((gk >> 1) - 1) & 1))
            ok = false;
          else
            mbar_arrive_expect_tx(&k_full[ks], C::kTile);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane < 8) {
          uint8_t* sK = smem + C::kK + ks * C::kTile;
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub)
            tma_load_2d(sK + sub * 16384 + lane * 2048, &kmap, &k_full[ks], sub * 64, y);
        }
        ++gk;
        // V tile j -> the single V stage
        if (lane == 0) {
          if (gv >= 1 && !mbar_wait(v_empty, (gv - 1) & 1))
            ok = false;
          else
            mbar_arrive_expect_tx(v_full, C::kTile);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane < 8) {
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub)
            tma_load_2d(smem + C::kV + sub * 16384 + lane * 2048, &vmap, v_full, sub * 64, y);
        }
        ++gv;
        __syncwarp();
      }
      ++it;
    }
    if (lane == 0) {
      if (!ok) record_status(p.dev_status, PGQA_ETIMEOUT);
      // no TMA write may land after the CTA exits: wait for the last fill of each buffer
      bool done = true;
      if (it > 0) done &= mbar_wait(q_full, (it - 1) & 1);
      for (int s = 0; s < 2 && s < gk; ++s) {
        const int last = s + ((gk - 1 - s) / 2) * 2;
        done &= mbar_wait(&k_full[s], (last >> 1) & 1);
      }
      if (gv > 0) done &= mbar_wait(v_full, (gv - 1) & 1);
      if (!done) record_status(p.dev_status, PGQA_ETIMEOUT);
    }
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, kBlockN, false);
      const uint32_t id_o = idesc_bf16_f32(128, D, true);
      const uint32_t q_addr = smem_u32(smem + C::kQ), v_addr = smem_u32(smem + C::kV);
      const uint32_t p_addr = smem_u32(smem + C::kP);
      int it = 0, gk = 0, gv = 0, np[2] = {0, 0};
      bool ok = true;
      // S_X = Q_X K^T for the K tile in stage ks
      auto issue_s = [&](int X, int ks) {
        const uint32_t k_addr = smem_u32(smem + C::kK + ks * C::kTile);
        const uint32_t qx = q_addr + X * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_f16_ss(tmem + X * 128, smem_desc_sw128(qx + off, 16, 1024),
                      smem_desc_sw128(k_addr + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        umma_commit(&s_full[X]);
      };
      // O_X (+)= P_X V
      auto issue_pv = [&](int X, bool accumulate) {
        const uint32_t px = p_addr + X * (128 * 128 * 2);
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk) {
          const uint32_t poff = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_f16_ss(tmem + 256 + X * 128, smem_desc_sw128(px + poff, 16, 1024),
                      smem_desc_sw128(v_addr + kk * 2048, 16384, 1024), id_o,
                      (accumulate || kk > 0) ? 1u : 0u);
        }
        umma_commit(&o_full[X]);
      };
      for (int k = c; k < p.num_items && ok; k += ncta) {
        const Item w = decode_item(p, k);
        if (!w.valid) continue;
        const int nkt_a = 2 * w.m + 1;
        if (!(ok = mbar_wait(q_full, it & 1))) break;
        tc_fence_after();
        if (!(ok = mbar_wait(&k_full[gk & 1], (gk >> 1) & 1))) break;
        tc_fence_after();
        issue_s(0, gk & 1);
        if (w.active_b) issue_s(1, gk & 1);
        umma_commit(&k_empty[gk & 1]);
        ++gk;
        if (w.nkt == 1) umma_commit(q_empty);
        for (int j = 0; j < w.nkt; ++j) {
          const bool more = j + 1 < w.nkt;
          if (!(ok = mbar_wait(v_full, gv & 1))) break;
          tc_fence_after();
          if (j < nkt_a) {
            if (!(ok = mbar_wait(&p_full[0], np[0] & 1))) break;
            ++np[0];
            tc_fence_after();
            issue_pv(0, j > 0);
          }
          if (more) {
            if (!(ok = mbar_wait(&k_full[gk & 1], (gk >> 1) & 1))) break;
            tc_fence_after();
            if (j + 1 < nkt_a) issue_s(0, gk & 1);
          }
          if (w.active_b) {
            if (!(ok = mbar_wait(&p_full[1], np[1] & 1))) break;
            ++np[1];
            tc_fence_after();
            issue_pv(1, j > 0);
          }
          umma_commit(v_empty);
          ++gv;
          if (more) {
            if (w.active_b) issue_s(1, gk & 1);
            umma_commit(&k_empty[gk & 1]);
            ++gk;
            if (j + 1 == w.nkt - 1) umma_commit(q_empty);
          }
        }
        ++it;
      }
      if (!ok) record_status(p.dev_status, PGQA_ETIMEOUT);
    }
  } else {
    // ================================================================ softmax rows
    const int X = warp >> 2;                      // 0: tile A, 1: tile B
    const int wq = warp & 3;                      // TMEM lane quadrant
    const int r = wq * 32 + lane;                 // query row in the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t s_col = X * 128, o_col = 256 + X * 128;
    uint8_t* sP = smem + C::kP + X * (128 * 128 * 2);
    int it = 0, gv = 0, tcnt = 0;
    bool ok = true;
    for (int k = c; k < p.num_items && ok; k += ncta) {
      const Item w = decode_item(p, k);
      if (!w.valid) continue;
      const int gv0 = gv;
      gv += w.nkt;
      const int my_it = it++;
      // the item's bad-block flag was published with its Q; every softmax warp takes
      // every item, including the warps of tile B when B does not exist
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(q_full, my_it & 1)))) break;
      const bool bad = bad_item[my_it & 1] != 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(q_empty);
      if (X == 1 && !w.active_b) continue;
      const int tq = 2 * w.m + X;                 // this tile's index in the sequence
      const int qpos = tq * kBlockM + r;          // this row's position in the sequence
      const int lim = min(qpos, w.L - 1);         // last key this row attends
      const int nkt_x = tq + 1;
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < nkt_x; ++j) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[X], tcnt & 1)))) break;
        tc_fence_after();
        const int kbase = j * kBlockN;
        // pass 1: the row's max over this key tile
        float mx = -INFINITY;
#pragma unroll
        for (int cc = 0; cc < kBlockN / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(lane_base + s_col + cc * 32, rr);
#pragma unroll
          for (int q = 0; q < 32; ++q) {
            const float v =
                kbase + cc * 32 + q <= lim ? __uint_as_float(rr[q]) * p.scale_log2 : -INFINITY;
            mx = fmaxf(mx, v);
          }
        }
        if (j > 0) {  // P_X V of the previous tile done: O_X stable and P_X free
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&o_full[X], (tcnt - 1) & 1)))) break;
          tc_fence_after();
        }
        const bool grow = mx > m_ref + kRescaleThreshold;
        const float alpha = grow ? ex2(m_ref - mx) : 1.f;  // 0 while m_ref = -inf
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_base + o_col + cc * 32, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tmem_st32(lane_base + o_col + cc * 32, o);
          }
          tmem_wait_st();
        }
        if (grow) {
          l *= alpha;
          m_ref = mx;
        }
        // pass 2: P = 2^(s * scale - m_ref) as bf16 into row r of the K-major,
        // 128-byte-swizzled A operand
        float sum = 0.f;
#pragma unroll
        for (int cc = 0; cc < kBlockN / 32; ++cc) {
          uint32_t rr[32];
          tmem_ld32(lane_base + s_col + cc * 32, rr);
          uint32_t pk[16];
#pragma unroll
          for (int q = 0; q < 32; q += 2) {
            const float e0 = kbase + cc * 32 + q <= lim
                                 ? ex2(fmaf(__uint_as_float(rr[q]), p.scale_log2, -m_ref))
                                 : 0.f;
            const float e1 = kbase + cc * 32 + q + 1 <= lim
                                 ? ex2(fmaf(__uint_as_float(rr[q + 1]), p.scale_log2, -m_ref))
                                 : 0.f;
            sum += e0 + e1;
            pk[q >> 1] = pack_bf16(e0, e1);
          }
#pragma unroll
          for (int c4 = 0; c4 < 4; ++c4) {
            const int c16 = cc * 4 + c4;  // 16-byte chunk of the 256-byte row
            *reinterpret_cast<uint4*>(sP + (c16 >> 3) * 16384 + swz128(r, c16 & 7)) =
                make_uint4(pk[c4 * 4], pk[c4 * 4 + 1], pk[c4 * 4 + 2], pk[c4 * 4 + 3]);
          }
        }
        l += sum;
        // V rows past the sequence end may hold anything (NaN included): zero them so
        // that P = 0 there contributes exactly nothing. Only the last key tile of the
        // item reaches past the end, and only this tile's softmax uses it.
        if (kbase + kBlockN > w.L) {
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(v_full, (gv0 + j) & 1)))) break;
          if (kbase + r >= w.L) {
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub) {
              uint4* row = reinterpret_cast<uint4*>(smem + C::kV + sub * 16384 + r * 128);
#pragma unroll
              for (int q = 0; q < 8; ++q) row[q] = make_uint4(0, 0, 0, 0);
            }
          }
        }
        fence_proxy_async_smem();
        tc_fence_before();
        mbar_arrive(&p_full[X]);
        ++tcnt;
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, lse
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&o_full[X], (tcnt - 1) & 1)))) break;
      tc_fence_after();
      const bool store = qpos < w.L;
      const size_t orow =
          static_cast<size_t>(w.start + (store ? qpos : 0)) * p.num_q_heads + w.hq;
      uint4* dst = reinterpret_cast<uint4*>(p.out + orow * D);
      const float inv = 1.f / l;
#pragma unroll
      for (int cc = 0; cc < D / 32; ++cc) {
        uint32_t o[32];
        tmem_ld32(lane_base + o_col + cc * 32, o);  // every lane: warp-collective
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (!bad) {
            const float* f = reinterpret_cast<const float*>(o) + q * 8;
            v = make_uint4(pack_bf16(f[0] * inv, f[1] * inv), pack_bf16(f[2] * inv, f[3] * inv),
                           pack_bf16(f[4] * inv, f[5] * inv), pack_bf16(f[6] * inv, f[7] * inv));
          }
          if (store) dst[cc * 4 + q] = v;
        }
      }
      if (store && p.lse) p.lse[orow] = bad ? -INFINITY : (m_ref + log2f(l)) * kLn2;
      tc_fence_before();
    }
    if (!ok && lane == 0) record_status(p.dev_status, PGQA_ETIMEOUT);
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
  const int sms = num_sms_current_device();
  if (sms <= 0) return PGQA_ECUDA;
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
  const int n_qtiles = (a.max_seqlen + kBlockM - 1) / kBlockM;
  p.n_pairs = (n_qtiles + 1) / 2;
  const long long items = static_cast<long long>(p.n_pairs) * a.num_seqs * a.num_q_heads;
  if (items > INT32_MAX) return PGQA_EUNSUPPORTED;
  p.num_items = static_cast<int>(items);
  p.oob_row = static_cast<int>(rows);
  p.scale_log2 = a.scale * kLog2e;
  const int grid = static_cast<int>(items < sms ? items : sms);
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
