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
// Work and scheduling
//  - A work item is a pair of consecutive 128-query tiles (A = 2m, B = 2m + 1) of
//    one query head; tile t visits key tiles 0..t (causal tile skipping) and B
//    exists only if the sequence reaches it.
//  - Every CTA builds the same dense list of the batch's items, longest first:
//    items of pair index m (descending), then sequences ordered by their number of
//    tile pairs (a stable counting sort in shared memory), then heads (so the heads
//    sharing a kv-head run side by side and share K/V in L2). A persistent grid (one
//    CTA per SM) takes items from this list with an atomic ticket counter, so the
//    load balances itself whatever the length mix; the last CTA to finish resets the
//    counter for the next call.
// Warp roles
//  - warp 8 (TMA): takes tickets (one ahead), checks the item's block ids, loads
//    Q_A and Q_B once, then for each key tile K and V (one stage each), each gathered
//    as 8 pages of 16 rows with 2-D tensor-map loads (128-byte swizzle). Pages past
//    the sequence end are loaded from past the end of the cache view, which TMA
//    fills with zeros.
//  - warp 9 (MMA, one thread): tcgen05.mma, M = N = 128, f32 accumulators in TMEM:
//    S_X = Q_X K^T for X = A, B and O_X += P_X V (V MN-major). The tile pair
//    ping-pongs: while one tile's softmax runs, the tensor core computes the other
//    tile's S and PV.
//  - warps 0-3 / 4-7 (softmax of tile A / B; thread = query row = TMEM lane): two
//    passes over the row's scores in TMEM (max, then exp2; 64 columns per load), the
//    causal mask applied on the diagonal tile only, P = 2^(s - m) as bf16 into
//    shared memory in the MMA's swizzled layout, O rescaled in TMEM only when the
//    running max grows by more than 2^8 (exact either way: P and l use the same
//    reference max); at the end O / l -> bf16 out and lse.
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
constexpr int kMaxSeqs = 4096;            // sequences per call
constexpr int kMaxLevels = 2048;          // tile pairs of the longest sequence

template <int D>
struct PCfg {
  static constexpr int kSub = D / 64;        // 128-byte (64-element) column blocks
  static constexpr int kTile = 128 * D * 2;  // [128 rows][D] bf16
  static constexpr int kQ = 0;               // Q_A, Q_B
  static constexpr int kK = 2 * kTile;       // K
  static constexpr int kV = 3 * kTile;       // V
  static constexpr int kP = 4 * kTile;       // P_A, P_B: [128 rows][128 keys] bf16 each
  static constexpr int kSeq = kP + 2 * 128 * 128 * 2;       // int [kMaxSeqs]: sorted sequences
  static constexpr int kLvlCnt = kSeq + kMaxSeqs * 4;       // int [kMaxLevels]: seqs with > m pairs
  static constexpr int kLvlOff = kLvlCnt + kMaxLevels * 4;  // int [kMaxLevels]: items before m
  static constexpr int kBar = kLvlOff + kMaxLevels * 4;
  static constexpr int kSmem = 1024 + kBar + 256;
};

struct PrefillParams {
  __nv_bfloat16* out;
  float* lse;
  const int32_t* cu_seqlens;
  const int32_t* block_tables;
  int* dev_status;
  int* ticket;  // [2] workspace: next ticket, finished CTAs (zero between calls)
  int max_blocks_per_seq;
  int num_seqs, num_tokens, max_seqlen;
  int num_q_heads, num_kv_heads, group;
  int num_blocks;
  int n_levels;  // tile pairs of the longest allowed sequence
  int oob_row;   // a row index past the end of the cache view (TMA fills zeros)
  float scale_log2;
};

__device__ __forceinline__ bool seq_ok(const PrefillParams& p, int s, int* start, int* len) {
  const int st = __ldg(p.cu_seqlens + s), L = __ldg(p.cu_seqlens + s + 1) - st;
  *start = st;
  *len = L;
  return L > 0 && L <= p.max_seqlen && (L + 15) / 16 <= p.max_blocks_per_seq && st >= 0 &&
         st + L <= p.num_tokens;
}

// Tile pairs of sequence s (0 for an empty or invalid one).
__device__ __forceinline__ int pairs_of(const PrefillParams& p, int s) {
  int st, L;
  if (!seq_ok(p, s, &st, &L)) return 0;
  return ((L + kBlockM - 1) / kBlockM + 1) / 2;
}

// One work item: a pair of query tiles of one (sequence, head).
struct Item {
  int seq, hq, m, start, L, nkt;
  bool active_b;
};

// Maps ticket t of the dense item list to its item. `lvl` is the caller's level
// cursor (the tickets a CTA receives only grow, so it only moves down).
__device__ __forceinline__ Item item_of(const PrefillParams& p, const int* sorted,
                                        const int* lvl_cnt, const int* lvl_off, int t,
                                        int& lvl) {
  while (lvl > 0 && t >= lvl_off[lvl] + lvl_cnt[lvl] * p.num_q_heads) --lvl;
  Item w;
  w.m = lvl;
  const int j = t - lvl_off[lvl];
  w.seq = sorted[j / p.num_q_heads];
  w.hq = j % p.num_q_heads;
  int st, L;
  seq_ok(p, w.seq, &st, &L);
  w.start = st;
  w.L = L;
  w.active_b = (2 * w.m + 1) * kBlockM < L;
  w.nkt = w.active_b ? 2 * w.m + 2 : 2 * w.m + 1;
  return w;
}

__device__ __forceinline__ uint64_t f2(float lo, float hi) {
  uint64_t r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ void unf2(uint64_t v, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
// (a.x * b.x + c.x, a.y * b.y + c.y) in one packed instruction
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1) paged_prefill_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const PrefillParams p) {
  using C = PCfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  int* sorted = reinterpret_cast<int*>(smem + C::kSeq);
  int* lvl_cnt = reinterpret_cast<int*>(smem + C::kLvlCnt);
  int* lvl_off = reinterpret_cast<int*>(smem + C::kLvlOff);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* k_full = bars + 2;
  uint64_t* k_empty = bars + 3;
  uint64_t* v_full = bars + 4;
  uint64_t* v_empty = bars + 5;
  uint64_t* s_full = bars + 6;   // [2] per tile
  uint64_t* p_full = bars + 8;   // [2]
  uint64_t* o_full = bars + 10;  // [2]
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(bars + 12);
  int* slot = reinterpret_cast<int*>(bars + 13);  // [2] ticket, [2] bad flag, by item parity
  int* misc = slot + 4;                           // [0] total items

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, ncta = gridDim.x;
  const int S = p.num_seqs, NL = p.n_levels;

  // length errors: reported once per sequence, by CTA 0
  if (c == 0) {
    for (int s = tid; s < S; s += kThreads) {
      int st, L;
      const bool ok = seq_ok(p, s, &st, &L) || L == 0;
      if (!ok || (s == S - 1 && st + L != p.num_tokens)) record_status(p.dev_status, PGQA_EINVAL);
    }
  }

  // ---- the dense item list: histogram of tile pairs per sequence (P area as scratch)
  int* hist = reinterpret_cast<int*>(smem + C::kP);
  for (int i = tid; i < NL; i += kThreads) hist[i] = 0;
  __syncthreads();
  for (int s = tid; s < S; s += kThreads) {
    const int np = pairs_of(p, s);
    if (np > 0) atomicAdd(&hist[np - 1], 1);
  }
  __syncthreads();
  if (warp == 0) {
    // lvl_cnt[m] = sequences with more than m pairs (a suffix sum over the histogram)
    int carry = 0;
    for (int base = ((NL - 1) / 32) * 32; base >= 0; base -= 32) {
      const int m = base + 31 - lane;  // descending within the chunk
      int v = m < NL ? hist[m] : 0;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
      }
      if (m < NL) lvl_cnt[m] = carry + v;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
    __syncwarp();
    // scatter cursor of pair count v: after the sequences with more than v pairs
    int* cursor = hist;
    for (int v = 1 + lane; v <= NL; v += 32) cursor[v - 1] = v < NL ? lvl_cnt[v] : 0;
    __syncwarp();
    // stable scatter: sequence index order within equal pair counts
    for (int base = 0; base < S; base += 32) {
      const int s = base + lane;
      const int v = s < S ? pairs_of(p, s) : 0;
      const unsigned grp = __match_any_sync(0xffffffffu, v);
      const int rank = __popc(grp & ((1u << lane) - 1));
      int pos = 0;
      if (v > 0) pos = cursor[v - 1] + rank;
      __syncwarp();
      if (v > 0) {
        sorted[pos] = s;
        if (rank == 0) cursor[v - 1] += __popc(grp);
      }
      __syncwarp();
    }
    // items before level m: levels are visited from NL - 1 down to 0
    if (lane == 0) {
      int off = 0;
      for (int m = NL - 1; m >= 0; --m) {
        lvl_off[m] = off;
        off += lvl_cnt[m] * p.num_q_heads;
      }
      misc[0] = off;
    }
  }
  if (tid == 0) {
    mbar_init(q_full, 1);
    // Q buffers are reused once the item's last S MMAs are done (one commit) and all
    // 8 softmax warps have taken the item (one arrival each), so q_full can never
    // run two phases ahead of a softmax warp's wait
    mbar_init(q_empty, 1 + 8);
    mbar_init(k_full, 1);
    mbar_init(k_empty, 1);
    mbar_init(v_full, 1);
    mbar_init(v_empty, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4 * 32);
      mbar_init(&o_full[s], 1);
    }
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
  const int total = misc[0];

  if (warp == kWarpTma) {
    // ================================================================ TMA producer
    if (lane == 0) {
      tma_prefetch_desc(&qmap);
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    int it = 0, gk = 0, gv = 0, lvl = NL - 1;
    bool ok = true;
    int t = 0;
    if (lane == 0) t = atomicAdd(p.ticket, 1);
    t = __shfl_sync(0xffffffffu, t, 0);
    for (;;) {
      const bool last = t >= total;
      int t_next = 0;
      if (lane == 0 && !last) t_next = atomicAdd(p.ticket, 1);  // one ahead
      Item w;
      bool bad = false;
      if (!last) {
        w = item_of(p, sorted, lvl_cnt, lvl_off, t, lvl);
        const int32_t* bt = p.block_tables + static_cast<size_t>(w.seq) * p.max_blocks_per_seq;
        const int npages = (min(w.L, w.nkt * kBlockN) + 15) / 16;
        for (int pg = lane; pg < npages; pg += 32) {  // block ids checked before Q is out
          const int32_t pbn = __ldg(bt + pg);
          bad |= pbn < 0 || pbn >= p.num_blocks;
        }
        bad = __any_sync(0xffffffffu, bad);
      }
      if (lane == 0) {
        if (it > 0 && !mbar_wait(q_empty, (it - 1) & 1)) {
          ok = false;
        } else {
          slot[it & 1] = last ? -1 : t;
          slot[2 + (it & 1)] = bad;
          if (bad) record_status(p.dev_status, PGQA_EBADINDEX);
          if (last) {
            mbar_arrive(q_full);  // publishes the end of the list
          } else {
            mbar_arrive_expect_tx(q_full, (w.active_b ? 2 : 1) * C::kTile);
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub) {
              tma_load_3d(smem + C::kQ + sub * 16384, &qmap, q_full, sub * 64, w.hq,
                          w.start + 2 * w.m * kBlockM);
              if (w.active_b)
                tma_load_3d(smem + C::kQ + C::kTile + sub * 16384, &qmap, q_full, sub * 64,
                            w.hq, w.start + (2 * w.m + 1) * kBlockM);
            }
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++it;
      if (last || !ok) break;
      const int h = w.hq / p.group;
      const int32_t* bt = p.block_tables + static_cast<size_t>(w.seq) * p.max_blocks_per_seq;
      for (int j = 0; j < w.nkt && ok; ++j) {
        int y = p.oob_row;
        if (lane < 8) {
          const int lp = j * 8 + lane;  // logical page
          if (lp * 16 < w.L) {
            const int32_t pbn = __ldg(bt + lp);
            if (pbn >= 0 && pbn < p.num_blocks) y = (pbn * p.num_kv_heads + h) * 16;
          }
        }
        if (lane == 0) {  // K tile j (its previous tile's S MMAs are done)
          if (gk >= 1 && !mbar_wait(k_empty, (gk - 1) & 1))
            ok = false;
          else
            mbar_arrive_expect_tx(k_full, C::kTile);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane < 8) {
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub)
            tma_load_2d(smem + C::kK + sub * 16384 + lane * 2048, &kmap, k_full, sub * 64, y);
        }
        ++gk;
        if (lane == 0) {  // V tile j (its previous tile's PV MMAs are done)
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
      t = __shfl_sync(0xffffffffu, t_next, 0);
    }
    if (lane == 0) {
      if (!ok) record_status(p.dev_status, PGQA_ETIMEOUT);
      // no TMA write may land after the CTA exits: wait for the last fill of each buffer
      bool done = mbar_wait(q_full, (it - 1) & 1);
      if (gk > 0) done &= mbar_wait(k_full, (gk - 1) & 1);
      if (gv > 0) done &= mbar_wait(v_full, (gv - 1) & 1);
      if (!done) record_status(p.dev_status, PGQA_ETIMEOUT);
    }
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issuer
    if (lane == 0) {
      const uint32_t id_s = idesc_bf16_f32(128, kBlockN, false);
      const uint32_t id_o = idesc_bf16_f32(128, D, true);
      const uint32_t q_addr = smem_u32(smem + C::kQ), k_addr = smem_u32(smem + C::kK);
      const uint32_t v_addr = smem_u32(smem + C::kV), p_addr = smem_u32(smem + C::kP);
      int it = 0, gk = 0, gv = 0, np[2] = {0, 0}, lvl = NL - 1;
      bool ok = true;
      // S_X = Q_X K^T
      auto issue_s = [&](int X) {
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
      for (;;) {
        if (!(ok = mbar_wait(q_full, it & 1))) break;
        const int t = slot[it & 1];
        ++it;
        if (t < 0) break;
        tc_fence_after();
        const Item w = item_of(p, sorted, lvl_cnt, lvl_off, t, lvl);
        const int nkt_a = 2 * w.m + 1;
        if (!(ok = mbar_wait(k_full, gk & 1))) break;
        tc_fence_after();
        issue_s(0);
        if (w.active_b) issue_s(1);
        umma_commit(k_empty);
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
            if (!(ok = mbar_wait(k_full, gk & 1))) break;
            tc_fence_after();
            if (j + 1 < nkt_a) issue_s(0);
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
            if (w.active_b) issue_s(1);
            umma_commit(k_empty);
            ++gk;
            if (j + 1 == w.nkt - 1) umma_commit(q_empty);
          }
        }
        if (!ok) break;
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
    const float sc = p.scale_log2;  // > 0 (checked on the host)
    const uint64_t sc2 = f2(sc, sc);
    int it = 0, gv = 0, tcnt = 0, lvl = NL - 1;
    bool ok = true;
    for (;;) {
      // the item's ticket and bad-block flag were published with its Q; every softmax
      // warp takes every item, including the warps of tile B when B does not exist
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(q_full, it & 1)))) break;
      const int t = slot[it & 1];
      const bool bad = slot[2 + (it & 1)] != 0;
      ++it;
      if (t < 0) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(q_empty);
      const Item w = item_of(p, sorted, lvl_cnt, lvl_off, t, lvl);
      const int gv0 = gv;
      gv += w.nkt;
      if (X == 1 && !w.active_b) continue;
      const int tq = 2 * w.m + X;                 // this tile's index in the sequence
      const int qpos = tq * kBlockM + r;          // this row's position in the sequence
      const int lim = min(qpos, w.L - 1);         // last key this row attends
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j <= tq; ++j) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[X], tcnt & 1)))) break;
        tc_fence_after();
        const int kbase = j * kBlockN;
        const bool diag = j == tq;  // the only tile with masked keys
        // pass 1: the row's max (of the raw scores; scale > 0)
        float mx = -INFINITY;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[64];
          tmem_ld64(lane_base + s_col + half * 64, sr);
          if (!diag) {
#pragma unroll
            for (int q = 0; q < 64; q += 2)
              mx = max3(mx, __uint_as_float(sr[q]), __uint_as_float(sr[q + 1]));
          } else {
#pragma unroll
            for (int q = 0; q < 64; ++q)
              mx = fmaxf(mx, kbase + half * 64 + q <= lim ? __uint_as_float(sr[q]) : -INFINITY);
          }
        }
        mx *= sc;
        if (j > 0) {  // P_X V of the previous tile done: O_X stable and P_X free
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&o_full[X], (tcnt - 1) & 1)))) break;
          tc_fence_after();
        }
        const bool grow = mx > m_ref + kRescaleThreshold;
        const float alpha = grow ? ex2(m_ref - mx) : 1.f;  // 0 while m_ref = -inf
        if (grow) {
          l *= alpha;
          m_ref = mx;
        }
        // pass 2: P = 2^(s * scale - m_ref) as bf16 into row r of the K-major,
        // 128-byte-swizzled A operand (masked keys give exactly 0)
        const uint64_t neg_m2 = f2(-m_ref, -m_ref);
        float sum0 = 0.f, sum1 = 0.f;
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t sr[64];
          tmem_ld64(lane_base + s_col + half * 64, sr);
#pragma unroll
          for (int c8 = 0; c8 < 8; ++c8) {
            uint32_t pk[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const int i0 = c8 * 8 + 2 * q;
              float a0, a1;
              unf2(fma2(f2(__uint_as_float(sr[i0]), __uint_as_float(sr[i0 + 1])), sc2, neg_m2),
                   a0, a1);
              float e0 = ex2(a0), e1 = ex2(a1);
              if (diag) {
                if (kbase + half * 64 + i0 > lim) e0 = 0.f;
                if (kbase + half * 64 + i0 + 1 > lim) e1 = 0.f;
              }
              sum0 += e0;
              sum1 += e1;
              pk[q] = pack_bf16(e0, e1);
            }
            const int c16 = half * 8 + c8;  // 16-byte chunk of the 256-byte row
            *reinterpret_cast<uint4*>(sP + (c16 >> 3) * 16384 + swz128(r, c16 & 7)) =
                make_uint4(pk[0], pk[1], pk[2], pk[3]);
          }
        }
        l += sum0 + sum1;
        // rescale O_X when some row's max grew (warp-collective TMEM access)
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int cc = 0; cc < D / 32; ++cc) {
            uint32_t o[32];
            tmem_ld32(lane_base + o_col + cc * 32, o);
#pragma unroll
            for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tmem_st32(lane_base + o_col + cc * 32, o);
          }
          tmem_wait_st();
        }
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
      for (int half = 0; half < D / 64; ++half) {
        uint32_t o[64];
        tmem_ld64(lane_base + o_col + half * 64, o);  // every lane: warp-collective
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          uint4 v = make_uint4(0, 0, 0, 0);
          if (!bad) {
            const float* f = reinterpret_cast<const float*>(o) + q * 8;
            v = make_uint4(pack_bf16(f[0] * inv, f[1] * inv), pack_bf16(f[2] * inv, f[3] * inv),
                           pack_bf16(f[4] * inv, f[5] * inv), pack_bf16(f[6] * inv, f[7] * inv));
          }
          if (store) dst[half * 8 + q] = v;
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
  if (tid == 0) {
    // the last CTA to finish resets the ticket counter for the next call
    __threadfence();
    if (atomicInc(reinterpret_cast<unsigned*>(p.ticket + 1), static_cast<unsigned>(ncta - 1)) ==
        static_cast<unsigned>(ncta - 1))
      atomicExch(p.ticket, 0);
  }
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
  p.ticket = static_cast<int*>(a.workspace);
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_tokens = a.num_tokens;
  p.max_seqlen = a.max_seqlen;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.n_levels = ((a.max_seqlen + kBlockM - 1) / kBlockM + 1) / 2;
  p.oob_row = static_cast<int>(rows);
  p.scale_log2 = a.scale * kLog2e;
  const long long items = static_cast<long long>(p.n_levels) * a.num_seqs * a.num_q_heads;
  const int grid = static_cast<int>(items < sms ? items : sms);
  paged_prefill_kernel<D><<<grid, kThreads, C::kSmem, a.stream>>>(qmap, kmap, vmap, p);
  return cudaPeekAtLastError() == cudaSuccess ? PGQA_OK : PGQA_ECUDA;
}

}  // namespace

int prefill_max_seqs() { return kMaxSeqs; }
int prefill_max_seqlen() { return kMaxLevels * 2 * kBlockM; }

pgqa_status_t launch_paged_prefill(const PrefillArgs& a) {
  if (a.head_dim == 128) return launch_prefill_variant<128>(a);
  if (a.head_dim == 64) return launch_prefill_variant<64>(a);
  return PGQA_EUNSUPPORTED;
}

}  // namespace pgqa
