// Causal variable-length prefill over the paged KV cache, on the tcgen05 tensor
// cores (sm_103a).
//
// Computes, for every sequence i (new tokens cu_seqlens[i] .. cu_seqlens[i+1]-1),
// query head hq and chunk position p, softmax(scale * q_p K^T) V over keys
// 0..Lk-Lq+p of sequence i, read through its block table, and lse = ln sum
// exp(score): the varlen, causal call of the rkmt.cn article (sec. 2.4), with
// separate query and key lengths (the chunk is the last Lq of the Lk cached tokens,
// bottom-right alignment; Lk = Lq without a cached prefix), over the paged cache of
// its sec. 3.1, with the attention steps of "LLaMA structure and inference
// performance" (sec. 3.1) and repeat_kv as the index map kv_head = hq / G (sec. 2.1).
// FlashAttention-style online softmax over 128-key tiles; the full score matrix is
// never formed.
//
// Work and scheduling
//  - A work item is one 128-query tile t of a sequence for a pair of query heads of
//    one kv-head group (A = head h, B = head h + 1; B absent for the last head of an
//    odd-sized group). Both tiles visit the key tiles up to the one holding the
//    tile's last query position (causal tile skipping) over the same K/V, in lockstep.
//  - Every CTA builds the same dense list of the batch's items, longest first:
//    items of tile index t (descending), then sequences ordered by their number of
//    tiles (a stable counting sort in shared memory), then head pairs (so the heads
//    sharing a kv-head run side by side and share K/V in L2). The tables go to the
//    workspace (every CTA writes the same values). A persistent grid (one CTA per
//    SM) takes items from the list with an atomic ticket counter, so the load
//    balances itself whatever the length mix; the last CTA to finish resets the
//    counter for the next call.
//  - Short chunks of groups of 4 or 8 heads (at most 256/G tokens, as in speculative
//    verification) use the grouped layout: an item is one (sequence, kv-head), tile A
//    holds the group's first G/2 heads and tile B the rest, one row per (token, head)
//    of the chunk, token-major.
// Warp roles (12 warps; warp 11 only waits: at 384 threads the register allocator
// fits the softmax in 167 registers without spilling)
//  - warp 10 (planner): takes tickets, decodes the items and checks their block ids,
//    up to two items ahead of the TMA warp (a two-entry queue in shared memory).
//  - warp 8 (TMA): publishes each item with its Q_A and Q_B, then streams K_0, V_0,
//    K_1, V_1, ... through a ring of 5 tiles (8 for head_dim 64), each tile gathered
//    as 8 pages of 16 rows with 2-D tensor-map loads (128-byte swizzle). Block ids are
//    read 32 pages at a time, one chunk ahead, and the next item's first pages are
//    requested while the ring is full, so no load waits on a table read. Pages past
//    the sequence end are loaded from past the end of the cache view, which TMA
//    fills with zeros.
//  - warp 9 (MMA; the warp runs the issue loop, one elected lane issues): tcgen05.mma,
//    M = N = 128, f32 accumulators in TMEM:
//    S_X = Q_X K^T for X = A, B (both operands in shared memory) and O_X += P_X V with
//    P_X read from tensor memory (V MN-major in shared memory). Issue order per key
//    tile j: P_A V_j, S_A(j+1), P_B V_j, S_B(j+1), so the tensor core works on one
//    tile while the other's softmax runs; S_X(j+1) overwrites the columns P_X(j) was
//    in, so it waits for P_X V_j to complete (the other tile's MMAs fill the pipe).
//  - warps 0-3 / 4-7 (softmax of tile A / B; thread = query row = TMEM lane): one
//    load of the row's 128 scores from TMEM, the causal mask on the diagonal tile
//    only, the row max and sum over independent chains, P = 2^(s - m) as bf16 into
//    the first 64 columns of S_X, O rescaled in TMEM only when the running max grows
//    by more than 2^8 (exact either way: P and l use the same reference max); at the
//    end O / l -> bf16 out and lse.
// E4M3 cache (per-kv-head scales; stored value = code * scale_h)
//  - The MMAs run on f16 operands: every E4M3 code is exactly an f16, q is rounded
//    to f16 once (exact for |q| in f16's normal range), P is written as f16, and the
//    scales leave the MMAs: k_scale_h multiplies the softmax scale, v_scale_h the
//    output (1/l becomes v_scale_h/l).
//  - The TMA warp loads a tile's codes (8 pages of 16 rows, unswizzled) into its
//    ring slot, where the f16 tile will be: rows 0-63 and 64-127 each into a part of
//    the slot that only the f16 rows of the same half overwrite. Warps 10 and 11
//    (the planner's work moves to the TMA warp) then each widen one half of the
//    rows in place: load all of the half's codes, convert, store the f16 rows in
//    the 128-byte-swizzled K-major layout TMA would have written (rows past the
//    sequence end as zeros), and arrive on the slot's `converted` barrier, which
//    the MMA warp waits for instead of the TMA one. They also convert Q_A and Q_B
//    from bf16 to f16 in place before the item's first S MMAs.
// All waits are bounded (a wait that gives up records PGQA_ETIMEOUT).
#include <cuda_bf16.h>

#include "host.h"
#include "ptx.cuh"
#include "tc.cuh"

namespace pgqa {
namespace {

constexpr int kBlockM = 128;  // query rows per tile
constexpr int kBlockN = 128;  // keys per tile
constexpr int kThreads = 384;
constexpr int kWarpTma = 8, kWarpMma = 9, kWarpPlan = 10;
constexpr uint32_t kTmemCols = 512;  // S_A 0, S_B 128 (P_X over the first 64), O_A 256, O_B 384
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kRescaleThreshold = 8.f;  // log2 units
constexpr int kMaxSeqs = 4096;            // sequences per call
constexpr int kMaxLevels = 2048;          // query tiles of the longest sequence
static_assert(256 + (kMaxSeqs + 2 * kMaxLevels) * 4 == kPrefillWorkspaceBytes,
              "workspace layout");

template <int D>
struct PCfg {
  static constexpr int kSub = D / 64;        // 128-byte (64-element) column blocks
  static constexpr int kTile = 128 * D * 2;  // [128 rows][D] bf16 (f16 for an E4M3 cache)
  static constexpr int kStages = D == 128 ? 5 : 8;  // K/V ring: 160 KB / 128 KB
  static constexpr int kQ = 0;               // Q_A, Q_B
  static constexpr int kRing = 2 * kTile;    // kStages K/V tiles, in load order
  static constexpr int kBar = kRing + kStages * kTile;
  static constexpr int kSmem = 1024 + kBar + 512;
  // E4M3 codes of rows 64h .. 64h+63 (D bytes each) inside a ring slot: where only
  // the f16 rows of the same half land (D = 128: under f16 columns 64..127 of the
  // same rows; D = 64: the second quarter of half h's f16 rows)
  __host__ __device__ static constexpr int code_half(int h) { return D == 128 ? 16384 + 8192 * h : 8192 * h + 4096; }
};

// Scratch in the ring while the tables are built (before any tile is loaded).
constexpr int kScrHist = 0;                            // int [kMaxLevels]
constexpr int kScrSorted = kScrHist + kMaxLevels * 4;  // int [kMaxSeqs]
constexpr int kScrCnt = kScrSorted + kMaxSeqs * 4;     // int [kMaxLevels]
constexpr int kScrOff = kScrCnt + kMaxLevels * 4;      // int [kMaxLevels]
static_assert(kScrOff + kMaxLevels * 4 <= 5 * 128 * 64 * 2, "table scratch");

struct PrefillParams {
  __nv_bfloat16* out;
  float* lse;
  const int32_t* cu_seqlens;  // null: every sequence has max_seqlen new tokens, in order
  const int32_t* seq_lens_k;  // cached tokens per sequence (Lk), or null: Lk = Lq
  const int32_t* block_tables;
  int* dev_status;
  int* ticket;  // workspace: [0] next ticket, [1] finished CTAs (zero between calls)
  int* tables;  // workspace + 256 B: sorted [kMaxSeqs], lvl_cnt, lvl_off [kMaxLevels]
  int max_blocks_per_seq;
  int num_seqs, num_tokens, max_seqlen, max_seqlen_k;
  int num_q_heads, num_kv_heads, group;
  int num_blocks;
  int n_levels;  // query tiles of the longest allowed sequence
  int pairs;     // head pairs per (sequence, tile): num_kv_heads * ceil(group / 2)
  int oob_row;   // a row index past the end of the cache view (TMA fills zeros)
  float scale_log2;
};

// Sequence s: its first new token, new tokens (Lq) and cached tokens (Lk); false if
// it has no new token or is inconsistent.
__device__ __forceinline__ bool seq_ok(const PrefillParams& p, int s, int* start, int* lq,
                                       int* lk) {
  const int st = p.cu_seqlens ? __ldg(p.cu_seqlens + s) : s * p.max_seqlen;
  const int Lq = p.cu_seqlens ? __ldg(p.cu_seqlens + s + 1) - st : p.max_seqlen;
  const int Lk = p.seq_lens_k ? __ldg(p.seq_lens_k + s) : Lq;
  *start = st;
  *lq = Lq;
  *lk = Lk;
  return Lq > 0 && Lq <= p.max_seqlen && Lk >= Lq && Lk <= p.max_seqlen_k &&
         (Lk + 15) / 16 <= p.max_blocks_per_seq && st >= 0 && st + Lq <= p.num_tokens;
}

// Query tiles of sequence s (0 for an empty or invalid one).
__device__ __forceinline__ int tiles_of(const PrefillParams& p, int s) {
  int st, Lq, Lk;
  if (!seq_ok(p, s, &st, &Lq, &Lk)) return 0;
  return (Lq + kBlockM - 1) / kBlockM;
}

// One work item: query tile t of one sequence for heads hq (A) and hq + 1 (B, if
// active_b), as the TMA warp publishes it to the other roles (8 ints per slot).
// ticket < 0: end of the list.
struct Item {
  int ticket, seq, hq, t, start, Lq, Lk, active_b, bad;
  // key tiles: up to the one holding the tile's last query position (Lk - Lq + 128t
  // + 127), and no further than the last key
  __device__ int nkt() const {
    const int last_q = Lk - Lq + t * kBlockM + kBlockM - 1;
    return min(last_q, Lk - 1) / kBlockN + 1;
  }
};

// Query heads per tile: 1, or G/2 in the grouped layout (groups of 4 or 8 heads and
// chunks of at most 256/G tokens, as in speculative verification): tile A then holds
// the group's first G/2 heads and tile B the rest, for every token of the chunk, one
// row per (token, head), token-major. The host chooses it by setting pairs = Hkv.
__device__ __forceinline__ int heads_per_tile(const PrefillParams& p) {
  return p.pairs == p.num_kv_heads && p.group >= 4 ? p.group / 2 : 1;
}

// Maps ticket t of the dense item list to its item. `lvl` is the caller's level
// cursor (the tickets a CTA receives only grow, so it only moves down).
__device__ __forceinline__ Item item_of(const PrefillParams& p, int t, int& lvl) {
  const int* sorted = p.tables;
  const int* lvl_cnt = p.tables + kMaxSeqs;
  const int* lvl_off = lvl_cnt + kMaxLevels;
  while (lvl > 0 && t >= lvl_off[lvl] + lvl_cnt[lvl] * p.pairs) --lvl;
  Item w;
  w.ticket = t;
  w.t = lvl;
  const int j = t - lvl_off[lvl];
  w.seq = sorted[j / p.pairs];
  const bool grouped = heads_per_tile(p) > 1;
  const int per_group = grouped ? 1 : (p.group + 1) / 2, pi = j % p.pairs;
  const int kv = pi / per_group;
  w.hq = kv * p.group + (grouped ? 0 : 2 * (pi % per_group));
  w.active_b = grouped || w.hq + 1 < (kv + 1) * p.group;
  seq_ok(p, w.seq, &w.start, &w.Lq, &w.Lk);
  w.bad = 0;
  return w;
}

// Ticket t decoded, with the block ids its key tiles read checked (warp-collective;
// t warp-uniform). Past the list: the end-of-list marker.
__device__ __forceinline__ Item plan_item(const PrefillParams& p, int t, int total, int& lvl,
                                          int lane) {
  Item w{-1, 0, 0, 0, 0, 0, 0, 0, 0};
  if (t < total) {
    w = item_of(p, t, lvl);
    const int32_t* bt = p.block_tables + static_cast<size_t>(w.seq) * p.max_blocks_per_seq;
    const int npages = (min(w.Lk, w.nkt() * kBlockN) + 15) / 16;
    bool bad = false;
    for (int pg = lane; pg < npages; pg += 32) {  // block ids checked before Q is out
      const int32_t pbn = __ldg(bt + pg);
      bad |= pbn < 0 || pbn >= p.num_blocks;
    }
    w.bad = __any_sync(0xffffffffu, bad);
  }
  return w;
}

// Eight bf16 to eight f16, round to nearest even (exact in f16's normal range).
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  return make_uint4(pack_f16(bf16_lo(v.x), bf16_hi(v.x)), pack_f16(bf16_lo(v.y), bf16_hi(v.y)),
                    pack_f16(bf16_lo(v.z), bf16_hi(v.z)), pack_f16(bf16_lo(v.w), bf16_hi(v.w)));
}

// Sixteen E4M3 codes (byte i = element i) to sixteen f16 (exact), as two 8-element
// halves.
__device__ __forceinline__ void e4m3x16_to_f16(uint4 v, uint4& lo, uint4& hi) {
  lo = make_uint4(e4m3x2_to_f16x2(v.x & 0xffffu), e4m3x2_to_f16x2(v.x >> 16),
                  e4m3x2_to_f16x2(v.y & 0xffffu), e4m3x2_to_f16x2(v.y >> 16));
  hi = make_uint4(e4m3x2_to_f16x2(v.z & 0xffffu), e4m3x2_to_f16x2(v.z >> 16),
                  e4m3x2_to_f16x2(v.w & 0xffffu), e4m3x2_to_f16x2(v.w >> 16));
}

// Widens rows 64h .. 64h+63 of the E4M3 tile in ring slot `slot` (codes at
// code_half(h)) to f16 in place, in the 128-byte-swizzled K-major layout (16-byte
// chunk k of row r at chunk k ^ (r & 7) of the row's 128-byte line, 64-column blocks
// 16 KB apart). Rows at or past `valid` (keys past the sequence end) become zeros.
// Every code of the half is loaded before any store: the f16 rows overwrite them.
// Store order: a 16-byte store is served 8 lanes at a time, and at head_dim 128 the 8
// lanes of one row write chunks 2(c mod 4) and 2(c mod 4) + 1 of column block c / 4.
// Lanes c and c + 4 would hit the same chunk position (the same four banks) of lines
// 16 KB apart, so the lanes of the second column block write their high chunk first:
// each store then covers the 8 distinct positions (2(c mod 4) + c / 4) ^ (r & 7).
template <int D>
__device__ __forceinline__ void widen_tile_half(uint8_t* slot, int h, int lane, int valid) {
  constexpr int kChunks = D / 16;             // 16-byte chunks per code row
  constexpr int kRowsPerPass = 32 / kChunks;  // rows one warp-wide load covers
  constexpr int kPasses = 64 / kRowsPerPass;
  const int c = lane % kChunks, r0 = lane / kChunks;
  const uint8_t* codes = slot + PCfg<D>::code_half(h);
  uint4 v[kPasses];
#pragma unroll
  for (int i = 0; i < kPasses; ++i)
    v[i] = *reinterpret_cast<const uint4*>(codes + (r0 + i * kRowsPerPass) * D + c * 16);
  __syncwarp();
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    const int r = 64 * h + r0 + i * kRowsPerPass;
    uint4 lo = make_uint4(0, 0, 0, 0), hi = lo;
    if (r < valid) e4m3x16_to_f16(v[i], lo, hi);
    uint8_t* line = slot + (c >> 2) * 16384 + r * 128;
    const int hi_first = c >> 2;  // 0 or 1 (always 0 at head_dim 64)
    const int k_first = 2 * (c & 3) + hi_first, k_second = k_first ^ 1;
    *reinterpret_cast<uint4*>(line + ((k_first ^ (r & 7)) << 4)) = hi_first ? hi : lo;
    *reinterpret_cast<uint4*>(line + ((k_second ^ (r & 7)) << 4)) = hi_first ? lo : hi;
  }
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
__device__ __forceinline__ uint64_t add2(uint64_t a, uint64_t b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}
__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

__device__ __forceinline__ void publish(int* slot, const Item& w) {
  slot[0] = w.ticket;
  slot[1] = w.seq;
  slot[2] = w.hq;
  slot[3] = w.t;
  slot[4] = w.start;
  slot[5] = w.Lq;
  slot[6] = w.Lk;
  slot[7] = (w.active_b ? 1 : 0) | (w.bad ? 2 : 0);
}
__device__ __forceinline__ Item read_slot(const int* slot) {
  Item w;
  w.ticket = slot[0];
  w.seq = slot[1];
  w.hq = slot[2];
  w.t = slot[3];
  w.start = slot[4];
  w.Lq = slot[5];
  w.Lk = slot[6];
  w.active_b = slot[7] & 1;
  w.bad = (slot[7] >> 1) & 1;
  return w;
}

// Builds the longest-first item tables in shared scratch, copies them to the
// workspace and leaves the number of items in misc[0].
__device__ __forceinline__ void build_tables(const PrefillParams& p, uint8_t* scratch,
                                             int* misc) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int S = p.num_seqs, NL = p.n_levels;
  int* hist = reinterpret_cast<int*>(scratch + kScrHist);
  int* sorted = reinterpret_cast<int*>(scratch + kScrSorted);
  int* lvl_cnt = reinterpret_cast<int*>(scratch + kScrCnt);
  int* lvl_off = reinterpret_cast<int*>(scratch + kScrOff);
  for (int i = tid; i < NL; i += kThreads) hist[i] = 0;
  __syncthreads();
  for (int s = tid; s < S; s += kThreads) {
    const int np = tiles_of(p, s);
    if (np > 0) atomicAdd(&hist[np - 1], 1);
  }
  __syncthreads();
  if (warp == 0) {
    // lvl_cnt[m] = sequences with more than m tiles (a suffix sum over the histogram)
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
    // scatter cursor of tile count v: after the sequences with more than v tiles
    int* cursor = hist;
    for (int v = 1 + lane; v <= NL; v += 32) cursor[v - 1] = v < NL ? lvl_cnt[v] : 0;
    __syncwarp();
    // stable scatter: sequence index order within equal tile counts
    for (int base = 0; base < S; base += 32) {
      const int s = base + lane;
      const int v = s < S ? tiles_of(p, s) : 0;
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
        off += lvl_cnt[m] * p.pairs;
      }
      misc[0] = off;
    }
  }
  __syncthreads();
  const int n_sorted = NL > 0 ? lvl_cnt[0] : 0;
  for (int i = tid; i < n_sorted; i += kThreads) p.tables[i] = sorted[i];
  for (int i = tid; i < NL; i += kThreads) {
    p.tables[kMaxSeqs + i] = lvl_cnt[i];
    p.tables[kMaxSeqs + kMaxLevels + i] = lvl_off[i];
  }
}

template <int D, bool F8>
__global__ void __launch_bounds__(kThreads, 1) paged_prefill_kernel(
    const __grid_constant__ CUtensorMap qmap, const __grid_constant__ CUtensorMap kmap,
    const __grid_constant__ CUtensorMap vmap, const PrefillParams p,
    const float* __restrict__ k_scale, const float* __restrict__ v_scale) {
  // (the E4M3 scales, [num_kv_heads] each, are separate parameters: a larger
  // parameter struct pushes the bf16 softmax past its register budget)
  using C = PCfg<D>;
  constexpr int kStages = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kBar);
  uint64_t* q_full = bars + 0;
  uint64_t* q_empty = bars + 1;
  uint64_t* full = bars + 2;                 // [kStages] ring
  uint64_t* empty = full + kStages;          // [kStages]
  uint64_t* s_full = empty + kStages;        // [2] per tile: S_X computed
  uint64_t* p_full = s_full + 2;             // [2] P_X written (and O_X rescaled)
  uint64_t* o_full = p_full + 2;             // [2] P_X V accumulated
  uint64_t* plan_full = o_full + 2;          // [2] planner -> TMA warp item queue
  uint64_t* plan_empty = plan_full + 2;      // [2]
  uint64_t* q_conv = plan_empty + 2;         // E4M3: Q_A, Q_B converted to f16
  uint64_t* conv = q_conv + 1;               // E4M3: [kStages] ring slot widened to f16
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(conv + kStages);
  int* slots = reinterpret_cast<int*>(conv + kStages + 1);  // [2][8]: the item, by parity
  int* plans = slots + 16;                              // [2][8]: the planner's queue
  int* misc = plans + 16;                               // [0] total items

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, ncta = gridDim.x;
  grid_dependency_wait();  // the stream's previous kernel (e.g. the KV scatter) is done
  grid_launch_dependents();  // the next one may place its CTAs as these exit

  // length errors: reported once per sequence, by CTA 0
  if (c == 0) {
    for (int s = tid; s < p.num_seqs; s += kThreads) {
      int st, Lq, Lk;
      const bool ok = seq_ok(p, s, &st, &Lq, &Lk) || Lq == 0;
      if (!ok || (s == p.num_seqs - 1 && st + Lq != p.num_tokens))
        record_status(p.dev_status, PGQA_EINVAL);
    }
    if constexpr (F8) {  // E4M3 scales must be positive and finite
      for (int h = tid; h < p.num_kv_heads; h += kThreads) {
        const float ks = __ldg(k_scale + h), vs = __ldg(v_scale + h);
        if (!(ks > 0.f && ks < INFINITY && vs > 0.f && vs < INFINITY))
          record_status(p.dev_status, PGQA_EINVAL);
      }
    }
  }
  static_assert((2 + 3 * kStages + 11 + 1) * 8 + 32 * 4 + 16 <= 512, "barrier area");
  build_tables(p, smem + C::kRing, misc);
  if (tid == 0) {
    mbar_init(q_full, 1);
    // Q buffers are reused once the item's last S MMAs are done (one commit) and all
    // 8 softmax warps (and both converter warps) have taken the item (one arrival
    // each), so q_full can never run two phases ahead of their waits
    mbar_init(q_empty, 1 + 8 + (F8 ? 2 : 0));
    mbar_init(q_conv, 2);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&conv[s], 2);
    }
    for (int s = 0; s < 2; ++s) {
      mbar_init(&s_full[s], 1);
      mbar_init(&p_full[s], 4 * 32);
      mbar_init(&o_full[s], 1);
      mbar_init(&plan_full[s], 1);
      mbar_init(&plan_empty[s], 1);
    }
    fence_mbar_init();
  }
  if (warp == kWarpMma) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();  // also orders the table writes before the TMA warp reads them
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
    int it = 0, g = 0;
    bool ok = true;
    // cache row of page 32 * ch + lane of item w (past the end: the zero-fill row)
    auto chunk_rows = [&](const Item& w, int ch) {
      int y = p.oob_row;
      const int lp = ch * 32 + lane;
      if (w.ticket >= 0 && lp * 16 < w.Lk) {
        const int32_t pbn =
            __ldg(p.block_tables + static_cast<size_t>(w.seq) * p.max_blocks_per_seq + lp);
        if (pbn >= 0 && pbn < p.num_blocks) y = (pbn * p.num_kv_heads + w.hq / p.group) * 16;
      }
      return y;
    };
    // the next item from the planner's queue (decoded, block ids checked) and the
    // cache rows of its first 64 pages
    struct Plan {
      Item w;
      int ch0, ch1;
    };
    int n_plans = 0, lvl = p.n_levels - 1;
    auto plan_next = [&]() {
      Plan pl;
      pl.w = Item{-1, 0, 0, 0, 0, 0, 0, 0, 0};
      if constexpr (F8) {  // the planner warp converts: plan here
        int t = 0;
        if (lane == 0) t = atomicAdd(p.ticket, 1);
        pl.w = plan_item(p, __shfl_sync(0xffffffffu, t, 0), total, lvl, lane);
      } else {
        const int q = n_plans & 1;
        if (!__all_sync(0xffffffffu, mbar_wait(&plan_full[q], (n_plans >> 1) & 1))) {
          ok = false;  // the end marker stands in for the item
        } else {
          pl.w = read_slot(plans + q * 8);
          __syncwarp();
          if (lane == 0) mbar_arrive(&plan_empty[q]);
        }
      }
      ++n_plans;
      pl.ch0 = chunk_rows(pl.w, 0);
      pl.ch1 = chunk_rows(pl.w, 1);
      return pl;
    };
    // one ring load: K or V tile (g), rows y of this lane's page (lanes 0-7)
    auto load_tile = [&](const CUtensorMap* map, int y) {
      if (!ok) return;
      const int s = g % kStages;
      if (lane == 0) {
        if (g >= kStages && !mbar_wait(&empty[s], ((g / kStages) - 1) & 1))
          ok = false;
        else
          mbar_arrive_expect_tx(&full[s], F8 ? C::kTile / 2 : C::kTile);
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) return;
      if (lane < 8) {
        uint8_t* slot = smem + C::kRing + s * C::kTile;
        if constexpr (F8) {  // the page's 16 code rows, where the widening expects them
          tma_load_2d(slot + C::code_half(lane >> 2) + (lane & 3) * 16 * D, map, &full[s], 0, y);
        } else {
#pragma unroll
          for (int sub = 0; sub < C::kSub; ++sub)
            tma_load_2d(slot + lane * 2048 + sub * 16384, map, &full[s], sub * 64, y);
        }
      }
      ++g;
    };
    Plan cur = plan_next();
    for (;;) {
      if (!ok) break;
      const Item& w = cur.w;
      const bool last = w.ticket < 0;
      if (lane == 0) {
        if (it > 0 && !mbar_wait(q_empty, (it - 1) & 1)) {
          ok = false;
        } else {
          publish(slots + (it & 1) * 8, w);
          if (w.bad) record_status(p.dev_status, PGQA_EBADINDEX);
          if (last) {
            mbar_arrive(q_full);  // publishes the end of the list
          } else {
            mbar_arrive_expect_tx(q_full, (w.active_b ? 2 : 1) * C::kTile);
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub) {
              tma_load_3d(smem + C::kQ + sub * 16384, &qmap, q_full, sub * 64, w.hq,
                          w.start + w.t * kBlockM);
              if (w.active_b)
                tma_load_3d(smem + C::kQ + C::kTile + sub * 16384, &qmap, q_full, sub * 64,
                            w.hq + heads_per_tile(p), w.start + w.t * kBlockM);
            }
          }
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++it;
      if (last || !ok) break;
      const int nkt = w.nkt();
      // rows of key tile j for lanes 0-7, from the chunk registers (chunk j / 4)
      int ch_a = cur.ch0, ch_b = cur.ch1, ch_i = 0;
      auto tile_row = [&](int j) {
        if ((j >> 2) != ch_i) {  // j / 4 moves up by one at a time
          ch_i = j >> 2;
          ch_a = ch_b;
          ch_b = chunk_rows(w, ch_i + 1);  // one chunk ahead
        }
        return __shfl_sync(0xffffffffu, ch_a, ((j & 3) << 3) | (lane & 7));
      };
      Plan nxt;
      int n_loads = 0;
      bool planned = false;
      // once the ring is full, the warp plans the next item instead of waiting
      auto after_load = [&]() {
        if (++n_loads == kStages) {
          nxt = plan_next();
          planned = true;
        }
      };
      // K_0, V_0, K_1, V_1, ...
      for (int j = 0; j < nkt && ok; ++j) {
        const int y = tile_row(j);
        load_tile(&kmap, y);
        if (!ok) break;
        after_load();
        load_tile(&vmap, y);
        if (!ok) break;
        after_load();
        __syncwarp();
      }
      if (!ok) break;
      if (!planned) nxt = plan_next();
      cur = nxt;
    }
    if (lane == 0) {
      if (!ok) record_status(p.dev_status, PGQA_ETIMEOUT);
      // no TMA write may land after the CTA exits: wait for the last fill of each buffer
      bool done = mbar_wait(q_full, (it - 1) & 1);
      for (int i = max(0, g - kStages); i < g; ++i)
        done &= mbar_wait(&full[i % kStages], (i / kStages) & 1);
      if (!done) record_status(p.dev_status, PGQA_ETIMEOUT);
    }
  } else if (!F8 && warp == kWarpPlan) {
    // ================================================================ planner
    // Takes tickets, decodes them and checks the items' block ids, two items ahead
    // of the TMA warp, so no table read sits on the load path.
    int lvl = p.n_levels - 1;
    bool ok = true;
    for (int k = 0;; ++k) {
      const int q = k & 1;
      if (k >= 2 && !__all_sync(0xffffffffu, mbar_wait(&plan_empty[q], ((k >> 1) - 1) & 1))) {
        ok = false;
        break;
      }
      int t = 0;
      if (lane == 0) t = atomicAdd(p.ticket, 1);
      const Item w = plan_item(p, __shfl_sync(0xffffffffu, t, 0), total, lvl, lane);
      if (lane == 0) {
        publish(plans + q * 8, w);
        mbar_arrive(&plan_full[q]);
      }
      if (w.ticket < 0) break;
    }
    if (!ok && lane == 0) record_status(p.dev_status, PGQA_ETIMEOUT);
  } else if (F8 && warp >= kWarpPlan) {
    // ================================================================ E4M3 widening
    // Warp 10 + h widens rows 64h .. 64h+63 of every K/V tile, in ring order, and
    // half of Q_A's and Q_B's bytes.
    const int h = warp - kWarpPlan;
    int it = 0, g = 0;
    bool ok = true;
    for (;;) {
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(q_full, it & 1)))) break;
      const Item w = read_slot(slots + (it & 1) * 8);
      ++it;
      if (w.ticket < 0) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(q_empty);
      for (int X = 0; X < (w.active_b ? 2 : 1); ++X) {
        uint4* qx = reinterpret_cast<uint4*>(smem + C::kQ + X * C::kTile + h * (C::kTile / 2));
#pragma unroll 4
        for (int i = lane; i < C::kTile / 32; i += 32) qx[i] = bf16x8_to_f16x8(qx[i]);
      }
      fence_proxy_async_smem();  // the MMAs read what these generic stores wrote
      __syncwarp();
      if (lane == 0) mbar_arrive(q_conv);
      const int nkt = w.nkt();
      for (int j = 0; j < 2 * nkt; ++j, ++g) {  // K_0, V_0, K_1, V_1, ...
        const int st = g % kStages;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&full[st], (g / kStages) & 1)))) break;
        widen_tile_half<D>(smem + C::kRing + st * C::kTile, h, lane, w.Lk - (j >> 1) * kBlockN);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(&conv[st]);
      }
      if (!ok) break;
    }
    if (!ok && lane == 0) record_status(p.dev_status, PGQA_ETIMEOUT);
  } else if (warp == kWarpMma) {
    // ================================================================ MMA issuer
    // The whole warp runs the issue loop (waits, descriptors) and one elected lane
    // issues each tcgen05 instruction.
    {
      const uint32_t id_s = F8 ? idesc_f16_f32(128, kBlockN, false) : idesc_bf16_f32(128, kBlockN, false);
      const uint32_t id_o = F8 ? idesc_f16_f32(128, D, true) : idesc_bf16_f32(128, D, true);
      const uint32_t q_addr = smem_u32(smem + C::kQ), ring = smem_u32(smem + C::kRing);
      int it = 0, g = 0, np[2] = {0, 0}, pv_issued[2] = {0, 0};
      bool ok = true;
      // S_X = Q_X K^T, K in ring stage ks. Its columns held P_X of the previous tile:
      // wait for that P_X V to complete first.
      auto issue_s = [&](int X, int ks) {
        if (pv_issued[X] > 0) {
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&o_full[X], (pv_issued[X] - 1) & 1)))) return false;
          tc_fence_after();
        }
        const uint32_t qx = q_addr + X * C::kTile, kx = ring + ks * C::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          umma_f16_ss_warp(tmem + X * 128, smem_desc_sw128(qx + off, 16, 1024),
                      smem_desc_sw128(kx + off, 16, 1024), id_s, kk > 0 ? 1u : 0u);
        }
        umma_commit_warp(&s_full[X]);
        return true;
      };
      // O_X (+)= P_X V: P_X from TMEM (8 columns per 16 keys), V in ring stage vs
      auto issue_pv = [&](int X, int vs, bool accumulate) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&p_full[X], np[X] & 1)))) return false;
        ++np[X];
        tc_fence_after();
        const uint32_t vx = ring + vs * C::kTile;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          umma_f16_ts_warp(tmem + 256 + X * 128, tmem + X * 128 + kk * 8,
                      smem_desc_sw128(vx + kk * 2048, 16384, 1024), id_o,
                      (accumulate || kk > 0) ? 1u : 0u);
        umma_commit_warp(&o_full[X]);
        ++pv_issued[X];
        return true;
      };
      // waits for ring load gi to land (E4M3: and be widened); returns its stage in st
      auto take = [&](int gi, int& st) {
        st = gi % kStages;
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(F8 ? &conv[st] : &full[st], (gi / kStages) & 1)))) return false;
        tc_fence_after();
        return true;
      };
      // Items run back to back: the next item's S_X(0) takes the place of S_X(t+1)
      // in the last key tile, so the tensor pipe does not drain between items.
      Item w;
      int ks, vs;
      // the first item's S_A(0), S_B(0)
      auto start_item = [&](Item& nw) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(q_full, it & 1)))) return false;
        nw = read_slot(slots + (it & 1) * 8);
        if (F8 && nw.ticket >= 0 && !(ok = __all_sync(0xffffffffu, mbar_wait(q_conv, it & 1)))) return false;
        ++it;
        tc_fence_after();
        return nw.ticket >= 0;
      };
      if (start_item(w) && take(g++, ks) && issue_s(0, ks) && (!w.active_b || issue_s(1, ks))) {
        umma_commit_warp(&empty[ks]);
        if (w.nkt() == 1) umma_commit_warp(q_empty);
        for (;;) {
          const int nkt = w.nkt();  // both tiles visit key tiles 0..t
          Item nx;
          bool nx_valid = false;
          for (int j = 0; j < nkt; ++j) {
            const bool more = j + 1 < nkt;
            if (!take(g++, vs)) break;  // V_j
            if (!issue_pv(0, vs, j > 0)) break;
            if (more) {
              if (!take(g++, ks)) break;  // K_{j+1}
              if (!issue_s(0, ks)) break;
            } else {  // the next item (its Q is out once this item's S are done)
              nx_valid = start_item(nx);
              if (!ok) break;
              if (nx_valid && (!take(g++, ks) || !issue_s(0, ks))) break;
            }
            if (w.active_b && !issue_pv(1, vs, j > 0)) break;
            if (more) {
              if (w.active_b && !issue_s(1, ks)) break;
              umma_commit_warp(&empty[ks]);
              if (j + 1 == nkt - 1) umma_commit_warp(q_empty);
            } else if (nx_valid) {
              if (nx.active_b && !issue_s(1, ks)) break;
              umma_commit_warp(&empty[ks]);
              if (nx.nkt() == 1) umma_commit_warp(q_empty);
            }
            umma_commit_warp(&empty[vs]);
          }
          if (!ok || !nx_valid) break;
          w = nx;
        }
      }
      if (!ok && lane == 0) record_status(p.dev_status, PGQA_ETIMEOUT);
    }
  } else if (warp < kWarpTma) {
    // ================================================================ softmax rows
    const int X = warp >> 2;       // 0: tile A, 1: tile B
    const int wq = warp & 3;       // TMEM lane quadrant
    const int r = wq * 32 + lane;  // query row in the tile = TMEM lane
    const uint32_t lane_base = tmem + (static_cast<uint32_t>(wq * 32) << 16);
    const uint32_t s_col = X * 128, o_col = 256 + X * 128;
    float sc = p.scale_log2;  // softmax scale in log2 units, > 0 (checked on the host)
    uint64_t sc2 = f2(sc, sc);
    int it = 0, gl = 0, tcnt = 0;
    bool ok = true;
    for (;;) {
      // every softmax warp takes every item, including the warps of tile B when B
      // does not exist
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(q_full, it & 1)))) break;
      const Item w = read_slot(slots + (it & 1) * 8);
      ++it;
      if (w.ticket < 0) break;
      __syncwarp();
      if (lane == 0) mbar_arrive(q_empty);
      const int gl0 = gl;  // ring index of this item's K_0 (then V_0, K_1, V_1, ...)
      gl += 2 * w.nkt();
      if (X == 1 && !w.active_b) continue;
      const int tq = w.t;                   // this tile's index among the new tokens
      const int hpt = heads_per_tile(p);    // grouped layout: row r = (token r / hpt, head)
      const int qpos = tq * kBlockM + r / hpt;  // this row's position among the new tokens
      const int hq_row = w.hq + X * hpt + r % hpt;  // this row's query head
      const int off = w.Lk - w.Lq;          // cached tokens before the new ones
      const int lim = min(off + qpos, w.Lk - 1);  // last key this row attends
      const int first_lim = off + tq * kBlockM;   // the tile's first row's last key
      const int nkt = w.nkt();
      const int kvh = w.hq / p.group;
      if constexpr (F8) {  // E4M3: the softmax scale times k_scale_h
        sc = p.scale_log2 * __ldg(k_scale + kvh);
        sc2 = f2(sc, sc);
      }
      float m_ref = -INFINITY, l = 0.f;
      for (int j = 0; j < nkt; ++j) {
        if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[X], tcnt & 1)))) break;
        tc_fence_after();
        const int kbase = j * kBlockN;
        uint32_t sr[128];
        tmem_ld128(lane_base + s_col, sr);
        if (kbase + kBlockN - 1 > first_lim) {  // a tile with masked keys (the diagonal)
#pragma unroll
          for (int q = 0; q < 128; ++q)
            if (kbase + q > lim) sr[q] = __float_as_uint(-INFINITY);
        }
        // the row max of the raw scores over 8 independent chains (scale > 0)
        float mc[8];
#pragma unroll
        for (int u = 0; u < 8; ++u)
          mc[u] = fmaxf(__uint_as_float(sr[u]), __uint_as_float(sr[8 + u]));
#pragma unroll
        for (int q = 16; q < 128; q += 16) {
#pragma unroll
          for (int u = 0; u < 8; ++u)
            mc[u] = max3(mc[u], __uint_as_float(sr[q + u]), __uint_as_float(sr[q + 8 + u]));
        }
        const float mx =
            max3(max3(mc[0], mc[1], mc[2]), max3(mc[3], mc[4], mc[5]), fmaxf(mc[6], mc[7])) * sc;
        // (S_X(j) was issued after P_X V_{j-1} completed: O_X is stable here)
        const bool grow = mx > m_ref + kRescaleThreshold;
        const float alpha = grow ? ex2(m_ref - mx) : 1.f;  // 0 while m_ref = -inf
        if (grow) {
          l *= alpha;
          m_ref = mx;
        }
        // P = 2^(s * scale - m_ref) as bf16 (E4M3: f16), two keys per TMEM column over
        // the first 64 columns of S_X (masked keys: 2^-inf = 0); the row sum over 8
        // chains
        const uint64_t neg_m2 = f2(-m_ref, -m_ref);
        uint64_t acc[4] = {0, 0, 0, 0};
        uint32_t pk[64];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
          float a0, a1;
          unf2(fma2(f2(__uint_as_float(sr[2 * c]), __uint_as_float(sr[2 * c + 1])), sc2, neg_m2),
               a0, a1);
          const float e0 = ex2(a0), e1 = ex2(a1);
          acc[c & 3] = add2(acc[c & 3], f2(e0, e1));
          pk[c] = F8 ? pack_f16(e0, e1) : pack_bf16(e0, e1);
        }
        tmem_st64(lane_base + s_col, pk);
        {
          float s0, s1, s2, s3, s4, s5, s6, s7;
          unf2(acc[0], s0, s1);
          unf2(acc[1], s2, s3);
          unf2(acc[2], s4, s5);
          unf2(acc[3], s6, s7);
          l += ((s0 + s1) + (s2 + s3)) + ((s4 + s5) + (s6 + s7));
        }
        // rescale O_X when some row's max grew (warp-collective TMEM access)
        if (j > 0 && __any_sync(0xffffffffu, grow)) {
#pragma unroll 1
          for (int cc = 0; cc < D / 64; ++cc) {
            uint32_t o[64];
            tmem_ld64(lane_base + o_col + cc * 64, o);
#pragma unroll
            for (int q = 0; q < 64; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * alpha);
            tmem_st64(lane_base + o_col + cc * 64, o);
          }
        }
        tmem_wait_st();
        // V rows past the sequence end may hold anything (NaN included): zero them so
        // that P = 0 there contributes exactly nothing. Only the last key tile of the
        // item reaches past the end; tile A's softmax zeroes it (P_B V is issued after
        // P_A V, which waits for this). E4M3: the widening wrote those rows as zeros.
        if (!F8 && X == 0 && kbase + kBlockN > w.Lk) {
          const int gi = gl0 + 2 * j + 1, vs = gi % kStages;
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&full[vs], (gi / kStages) & 1)))) break;
          if (kbase + r >= w.Lk) {
            uint8_t* vrow = smem + C::kRing + vs * C::kTile + r * 128;
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub) {
              uint4* row = reinterpret_cast<uint4*>(vrow + sub * 16384);
#pragma unroll
              for (int q = 0; q < 8; ++q) row[q] = make_uint4(0, 0, 0, 0);
            }
          }
          fence_proxy_async_smem();  // the MMAs read what these generic stores wrote
        }
        tc_fence_before();
        mbar_arrive(&p_full[X]);
        ++tcnt;
      }
      if (!ok) break;
      // epilogue: O / l -> bf16, lse
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&o_full[X], (tcnt - 1) & 1)))) break;
      tc_fence_after();
      const bool store = qpos < w.Lq;
      const size_t orow =
          static_cast<size_t>(w.start + (store ? qpos : 0)) * p.num_q_heads + hq_row;
      if (store && p.lse) p.lse[orow] = w.bad ? -INFINITY : (m_ref + log2f(l)) * kLn2;
      uint8_t* dst = reinterpret_cast<uint8_t*>(p.out + orow * D);
      const float inv = (F8 ? __ldg(v_scale + kvh) : 1.f) / l;
      // the row's D values in one TMEM load (D = 128: 128 columns; D = 64: 64), then
      // 32-byte stores when out is 32-byte aligned (a row is D * 2 bytes), else 16-byte
      uint32_t o[D];
      if constexpr (D == 128) {
        tmem_ld128(lane_base + o_col, o);  // every lane: warp-collective
      } else {
        tmem_ld64(lane_base + o_col, o);
      }
      const uint32_t keep = w.bad ? 0u : 0xffffffffu;  // a bad item's rows are written as zeros
      if ((reinterpret_cast<uintptr_t>(p.out) & 31) == 0) {
#pragma unroll
        for (int q = 0; q < D / 16; ++q) {  // 16 values = 32 bytes per store
          const float* f = reinterpret_cast<const float*>(o) + q * 16;
          uint32_t v[8];
#pragma unroll
          for (int u = 0; u < 8; ++u) v[u] = pack_bf16(f[2 * u] * inv, f[2 * u + 1] * inv) & keep;
          if (store) st_global_v8(dst + q * 32, v);
        }
      } else {
#pragma unroll
        for (int q = 0; q < D / 8; ++q) {  // 8 values = 16 bytes per store
          const float* f = reinterpret_cast<const float*>(o) + q * 8;
          const uint4 v = make_uint4(
              pack_bf16(f[0] * inv, f[1] * inv) & keep, pack_bf16(f[2] * inv, f[3] * inv) & keep,
              pack_bf16(f[4] * inv, f[5] * inv) & keep, pack_bf16(f[6] * inv, f[7] * inv) & keep);
          if (store) reinterpret_cast<uint4*>(dst)[q] = v;
        }
      }
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

template <int D, bool F8>
pgqa_status_t launch_prefill_variant(const PrefillArgs& a) {
  using C = PCfg<D>;
  const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * 16;
  CUtensorMap qmap, kmap, vmap;
  // bf16 cache: 64-column boxes, 128-byte swizzle; E4M3: one unswizzled box per page
  const CUtensorMapDataType kv_type =
      F8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t row_bytes = F8 ? D : D * 2;
  const uint32_t box_inner = F8 ? D : 64;
  const CUtensorMapSwizzle kv_swz = F8 ? CU_TENSOR_MAP_SWIZZLE_NONE : CU_TENSOR_MAP_SWIZZLE_128B;
  // grouped layout (see heads_per_tile) for short chunks of groups of 4 or 8 heads: a Q
  // tile is G/2 heads x 256/G tokens (128 rows, token-major), else 1 head x 128 tokens
  const int group = a.num_q_heads / a.num_kv_heads;
  const bool grouped = (group == 4 || group == 8) && a.max_seqlen <= 256 / group;
  if (!tensor_map_3d(&qmap, a.q, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, D, a.num_q_heads,
                     a.num_tokens, static_cast<uint64_t>(D) * 2,
                     static_cast<uint64_t>(a.num_q_heads) * D * 2, 64, grouped ? group / 2 : 1,
                     grouped ? 256 / group : kBlockM, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tensor_map_2d(&kmap, a.k_cache, kv_type, D, rows, row_bytes, box_inner, 16, kv_swz) ||
      !tensor_map_2d(&vmap, a.v_cache, kv_type, D, rows, row_bytes, box_inner, 16, kv_swz))
    return PGQA_ECUDA;
  if (!smem_attr_ready(reinterpret_cast<const void*>(paged_prefill_kernel<D, F8>), C::kSmem))
    return PGQA_ECUDA;
  const int sms = num_sms_current_device();
  if (sms <= 0) return PGQA_ECUDA;
  PrefillParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.cu_seqlens = a.cu_seqlens;
  p.seq_lens_k = a.seq_lens_k;
  p.max_seqlen_k = a.seq_lens_k ? a.max_seqlen_k : a.max_seqlen;
  p.block_tables = a.block_tables;
  p.dev_status = a.dev_status;
  p.ticket = static_cast<int*>(a.workspace);
  p.tables = reinterpret_cast<int*>(static_cast<uint8_t*>(a.workspace) + 256);
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_tokens = a.num_tokens;
  p.max_seqlen = a.max_seqlen;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.n_levels = (a.max_seqlen + kBlockM - 1) / kBlockM;
  p.pairs = grouped ? a.num_kv_heads : a.num_kv_heads * ((p.group + 1) / 2);
  p.oob_row = static_cast<int>(rows);
  p.scale_log2 = a.scale * kLog2e;
  const long long items = static_cast<long long>(p.n_levels) * a.num_seqs * p.pairs;
  const int grid = static_cast<int>(items < sms ? items : sms);
  if (launch_after_previous(paged_prefill_kernel<D, F8>, dim3(grid), dim3(kThreads), C::kSmem,
                            a.stream, qmap, kmap, vmap, p, a.k_scale, a.v_scale) != cudaSuccess)
    return PGQA_ECUDA;
  return cudaPeekAtLastError() == cudaSuccess ? PGQA_OK : PGQA_ECUDA;
}

}  // namespace

int prefill_max_seqs() { return kMaxSeqs; }
int prefill_max_seqlen() { return kMaxLevels * kBlockM; }

pgqa_status_t launch_paged_prefill(const PrefillArgs& a) {
  const bool f8 = a.cache_dtype == PGQA_DTYPE_E4M3;
  if (a.head_dim == 128) return f8 ? launch_prefill_variant<128, true>(a)
                                   : launch_prefill_variant<128, false>(a);
  if (a.head_dim == 64) return f8 ? launch_prefill_variant<64, true>(a)
                                  : launch_prefill_variant<64, false>(a);
  return PGQA_EUNSUPPORTED;
}

}  // namespace pgqa
