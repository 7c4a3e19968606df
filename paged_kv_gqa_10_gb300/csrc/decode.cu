// Paged decode attention for sm_103a.
//
// Computes, for every sequence b and query head hq, softmax(scale * q K^T) V over
// b's cached tokens read through its block table ("LLaMA structure and inference
// performance" (wmrh.cn) sec. 3.1 steps 3-6, with repeat_kv of sec. 2.1 as the
// index map kv_head = hq / G; pages addressed as in the rkmt.cn article, sec. 3.1),
// plus lse = ln sum exp(score).
//
// Work decomposition (bandwidth-bound: every KV byte is read exactly once)
//  - A unit is one (sequence, kv-head): its pages are read once for all G = Hq/Hkv
//    query heads of the group.
//  - Stream-K: the units' pages, laid end to end in (sequence, kv-head, page) order,
//    are cut into equal ranges, one per CTA of a grid sized to fill the GPU (SMs x
//    resident CTAs). Each CTA streams its range without a break, so ragged context
//    lengths cannot unbalance the grid. Units inside a range are finished in place;
//    a unit cut by range boundaries is finished by whichever of its CTAs arrives
//    last (an atomic ticket: no CTA waits for another), which merges the partial
//    results with their LSEs. Only the first and the last unit of a range can be
//    cut, so each CTA owns two partial slots. A CTA takes its range as runs: the unit
//    holding its last page, then the unit holding its first page, then the whole
//    units between, so the shared units are merged mid-kernel and the range ends,
//    when it can, on a unit no other CTA touches.
//  - The range plan (context-length scan, unit search, first block-table rows) reads
//    only context lengths and block tables and runs before the wait for the stream's
//    previous kernel (programmatic launch); q, K/V and the workspace come after it.
//  - Fused append (optional): the warp that reads the page holding key L-1 writes the
//    step's new K/V row into the cache and over that row of its shared-memory copy.
//  - Warp roles: one producer warp streams pages with TMA (2-D tensor map over the
//    cache viewed as [num_blocks*Hkv*16 rows][head_dim], 128-byte swizzle) into
//    mbarrier-guarded stages; 4 consumer warps take pages round-robin. Each consumer
//    warp owns its own sub-ring of stages, so consecutive uses of a stage belong to
//    one warp and a parity wait can never be two phases behind. The producer reads
//    the block table 64 pages ahead (coalesced, into a shared ring of row
//    coordinates) and refills each consumer warp's stages as soon as that warp frees
//    one (non-blocking polls), so a slow warp never holds back the others' loads. A
//    merge warp takes each finished unit's per-warp states and writes its output or
//    partial, so the consumers go straight on to the next unit.
//    Consumers read each unit's query rows straight from global memory, one unit
//    ahead.
//  - Math per 16-token page on the warp-level tensor path (mma.m16n8k16):
//      S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]   (tokens fill M = 16)
//      online softmax on the S^T fragment (column = query head), with a lazy
//      reference: the max reduction and the rescale of l and O run only on pages
//      where a score exceeds the column's reference by more than 2^8
//      P^T fragment -> B operand with movmatrix (an 8x8 transpose in registers)
//      O^T[D x 8] += V^T[D x 16] . P^T[16 x 8]            (V^T via ldmatrix.trans)
//    G <= 8 heads sit in N = 8; padded heads have q = 0 and are never stored.
//  - FP8 E4M3 cache: codes are widened to f16 in registers (exact) and fed to the
//    f16 MMA; k_scale folds into the score scale, v_scale into the final output.
//    The head-dimension order inside an MMA is a free permutation (it is the
//    contraction index for QK^T and a row relabelling for PV), chosen so that each
//    thread's bytes are contiguous in shared memory.
//  - Multi-token decode (speculative verification): a unit then has q_len x G query
//    rows (row i = token i / G, head i % G), token t seeing keys 0 .. L - q_len + t
//    (each fragment column has its own causal limit). Up to 8 rows run as above. Up to
//    32 run in the row-split form: consumer warp w holds rows 8w .. 8w+7 and reads every
//    page, from one ring filled in page order whose stages every warp with rows frees;
//    each warp hands its rows' state to the merge warp, which finishes the units as in
//    the plain form. Over a bf16 cache its warps take two pages a step (one softmax
//    step over their 32 keys): a page's softmax is a dependency chain the next page
//    cannot start before, and two pages per chain halve the chains.
//  - Per page, each lane's swizzled fragment offsets are precomputed, pages that every
//    column sees whole skip the mask arithmetic, and the V masking of a context's last
//    page is one branch per page.
//  - Every wait is bounded; a warp whose wait gives up records PGQA_ETIMEOUT, stops
//    computing, but keeps taking part in every CTA barrier, so nothing can hang.
#include <cuda_bf16.h>
#include <float.h>

#include <atomic>

#include "host.h"
#include "ptx.cuh"

namespace pgqa {
namespace {

constexpr int kNW = 4;  // consumer warps per CTA
constexpr int kWarpProd = kNW, kWarpMerge = kNW + 1;
constexpr int kThreads = (kNW + 2) * 32;
constexpr int kMinChunk = 8;  // pages per CTA range, at least
// online softmax: a column's reference max moves only when a score exceeds it by more
// than this (log2 units), so P <= 256 and most pages skip the max reduction and rescale
constexpr float kLazyLog2 = 8.f;
constexpr int kYRing = 256;   // TMA row coordinates fetched ahead of issue
static_assert(kYRing >= 64 + 32, "the fetch lookahead must fit the ring");
constexpr int kScanSlots = kThreads / 32 + 1;  // one per warp, then the found unit start
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct DecodeParams {
  __nv_bfloat16* out;
  float* lse;
  const __nv_bfloat16* q;
  const int32_t* block_tables;
  const int32_t* context_lens;
  const float* k_scale;
  const float* v_scale;
  int* counters;    // [B * Hkv] tickets, zero between calls
  float* part_lse;  // [grid][2][8] base-2 LSE of a partial (+inf = poisoned)
  float* part_o;    // [grid][2][8][D] normalised partial output
  int* dev_status;
  int max_blocks_per_seq;
  int num_seqs, num_q_heads, num_kv_heads, group;
  int q_len;  // new tokens per sequence: 1 (decode), or the tokens a multi-token decode
              // verifies (q is [num_seqs][q_len][num_q_heads][D], token t sees keys
              // 0 .. L - q_len + t)
  int num_blocks;
  int max_context_len;
  int block_size;    // 8, 16 or 32 tokens per block; the kernel works on 16-token pages
  int window;        // > 0: each context's last `window` keys only
  float scale_log2;  // scale * log2(e)
  // limit of the bounded waits while the CTA streams (kWaitLimitNs unless a test set a
  // shorter one); the producer's final wait for its own copies always uses kWaitLimitNs
  unsigned long long wait_ns;
};

// Fused append: the step's new token, key L-1 of every sequence, is written into the
// cache by the warp that reads the page holding it, which also puts the row into its
// copy of that page in shared memory (the TMA load may have read the row before or
// after the global store: no other CTA reads that page). Null pointers: no append.
struct DecodeAppend {
  const uint4* key;    // [num_seqs][Hkv][D] bf16
  const uint4* value;
  uint8_t* k_cache;    // the caches, written through
  uint8_t* v_cache;
};

template <int D, bool kFp8, int NT = 1, bool kRS = false>
struct Cfg {
  // query rows of a unit, in NT 8-row n-tiles per warp: the group's G <= 8 heads, or
  // q_len tokens x G heads for multi-token decode (up to 8 rows with NT = 1; the
  // row-split form kRS: one 8-row tile per consumer warp, up to 32 rows, every warp
  // reading every page of one shared ring). The launches use NT = 1 only: giving a
  // warp all the rows of a larger unit (NT = 3, one CTA per SM) ran slower than the
  // row-split form; the template keeps NT general.
  static constexpr int kRows = kRS ? 8 * kNW : 8 * NT;
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;      // one token row of one head
  // 64-byte rows (E4M3 at head_dim 64) are staged two tokens to a 128-byte swizzled
  // row: token t of a page is in shared row t / 2, bytes 64 (t % 2) .. 64 (t % 2) + 63
  static constexpr bool kPack = kRowBytes == 64;
  static constexpr int kSub = kPack ? 1 : kRowBytes / 128;  // 128-byte TMA boxes per row
  static constexpr int kPageBytes = 16 * kRowBytes;
  static constexpr int kStageBytes = 2 * kPageBytes;  // K page + V page
  // about 16 KB of pages in flight per consumer warp (E4M3: 20 KB, with one merge
  // buffer instead of two paying for the fifth stage); NT > 1 would run one CTA per SM
  // and give each warp 32-40 KB
  static constexpr int kStagesPerWarp =
      kRS ? 0
          : NT > 1 ? (kStageBytes >= 8192 ? 5 : 8)
                   : (kStageBytes >= 8192 ? 2 : kFp8 ? 20480 / kStageBytes : 16384 / kStageBytes);
  // unit states in flight to the merge warp
  static constexpr int kMergeBufs = (kRS || kFp8 || NT > 1) ? 1 : 2;
  // the row-split form: one ring of 88 KB, filled in page order
  static constexpr int kStages = kRS ? 90112 / kStageBytes : kNW * kStagesPerWarp;
  static constexpr int kNkc = D / 16;              // 16-wide chunks of head_dim
  static constexpr int kRing = kStages * kStageBytes;
  // a merge buffer holds every consumer warp's O of one unit, [kNW][kRows] rows of D
  // floats, or in the row-split form each row once (the warp holding it wrote it),
  // [kRows] rows of D + 4 floats (the padding spreads a warp's stores over the banks)
  static constexpr int kStateWarps = kRS ? 1 : kNW;
  static constexpr int kLd = kRS ? D + 4 : D;
  static constexpr int kMergeFloats = kStateWarps * kRows * kLd;
  static constexpr int kMlFloats = kStateWarps * kRows * 2;  // (m, l) per state row
  static constexpr int kOffMerge = kRing;                    // [bufs] by unit parity
  static constexpr int kOffMl = kOffMerge + kMergeBufs * kMergeFloats * 4;
  static constexpr int kOffBar = kOffMl + kMergeBufs * kMlFloats * 4;  // full[S], empty[S],
                                                                      // unit_done[2], merge_free[2]
  static constexpr int kOffMeta = kOffBar + (2 * kStages + 4) * 8;    // [S] int
  static constexpr int kOffY = (kOffMeta + kStages * 4 + 15) / 16 * 16;  // [kYRing] int
  static constexpr int kOffY2 = kOffY + kYRing * 4;                   // [kYRing] int (block 8)
  static constexpr int kOffMisc = kOffY2 + kYRing * 4;                // 32 ints, kScanSlots int64
  static constexpr int kOffRuns = kOffMisc + 32 * 4 + kScanSlots * 8;   // Run[3], Walk w0
  static constexpr int kSmem = 1024 + kOffRuns + 4 * 48;
  static_assert(kPack || kRowBytes % 128 == 0, "rows must be whole 128-byte swizzle rows");
  static_assert(!kRS || 227 * 1024 / (kSmem + 1024) >= 2, "row-split: two CTAs per SM");
  static_assert(kStageBytes % 1024 == 0 && kOffMerge % 16 == 0 && kOffMl % 16 == 0 &&
                    kOffBar % 8 == 0 && kOffY % 16 == 0 && (kOffMisc + 32 * 4) % 8 == 0 &&
                    kOffRuns % 8 == 0 && (kLd * 4) % 16 == 0,
                "shared-memory regions must be aligned for their types");
};

// CTAs of one decode kernel resident per SM (the grid is this times the SM count).
template <int D, bool kFp8, int NT = 1, bool kRS = false>
constexpr int ctas_per_sm() {
  static_assert(Cfg<D, kFp8, NT, kRS>::kSmem + 1024 <= 227 * 1024, "shared memory");
  return (227 * 1024) / (Cfg<D, kFp8, NT, kRS>::kSmem + 1024) >= 2 ? 2 : 1;
}

// First key attended in a context of L keys: L - window with a sliding window (the
// last `window` keys: query i sees keys i-W+1..i, "PageAttention + FlashAttention,
// the golden combination", sec. 4.1), else 0.
__device__ __forceinline__ int first_key(const DecodeParams& p, int L) {
  return p.window > 0 && L > p.window ? L - p.window : 0;
}

// Pages the step reads of a sequence of context length L (those holding keys
// first_key .. L-1); 0 for an invalid length.
__device__ __forceinline__ int pages_of_len(const DecodeParams& p, int L, bool* valid = nullptr) {
  const int n = (L + 15) >> 4;
  const bool ok = L >= 0 && L <= p.max_context_len && (L == 0 || L >= p.q_len) &&
                  (L + p.block_size - 1) / p.block_size <= p.max_blocks_per_seq;
  if (valid) *valid = ok;
  return ok && L > 0 ? n - (first_key(p, L) >> 4) : 0;
}

// Pages of sequence b the step reads.
__device__ __forceinline__ int pages_of(const DecodeParams& p, int b, bool* valid = nullptr) {
  return pages_of_len(p, __ldg(p.context_lens + b), valid);
}

// Logical page of sequence b's first page read.
__device__ __forceinline__ int first_page(const DecodeParams& p, int b) {
  return first_key(p, __ldg(p.context_lens + b)) >> 4;
}

// Sum over the CTA (every thread of the CTA must call it).
__device__ __forceinline__ long long block_sum(long long v, long long* scratch) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  __syncthreads();
  if (lane == 0) scratch[warp] = v;
  __syncthreads();
  long long t = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) t += scratch[w];
  return t;
}

// Inclusive prefix sum over the CTA's threads; *total receives the sum.
__device__ __forceinline__ long long block_scan(long long v, long long* scratch,
                                                long long* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long n = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += n;
  }
  __syncthreads();
  if (lane == 31) scratch[warp] = v;
  __syncthreads();
  long long before = 0, t = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < warp) before += scratch[w];
    t += scratch[w];
  }
  *total = t;
  return v + before;
}

// A CTA's walk over units: unit (b, h) holds pages [S, S + P) of the global order.
struct Walk {
  int b, h, P;
  int fp;  // 16-token page of the unit's first page read
  int L;   // the sequence's context length
  long long S;
  __device__ __forceinline__ void next(const DecodeParams& p) {
    S += P;
    if (++h == p.num_kv_heads) {
      h = 0;
      do {
        ++b;
        P = b < p.num_seqs ? pages_of(p, b) : 0;
      } while (P == 0 && b < p.num_seqs);
      fp = b < p.num_seqs ? first_page(p, b) : 0;
      L = b < p.num_seqs ? __ldg(p.context_lens + b) : 0;
    }
  }
};

// The order a CTA works through its range [r0, r1): runs of consecutive pages of the
// global order, `count` pages from page `first` of unit w on (crossing into the
// following units). The unit holding r1 - 1 (its part in the range) comes first, then
// the unit holding r0, then the whole units between: the two units the CTA may share
// with its neighbours are done early (their cross-CTA merge happens mid-kernel) and the
// range ends on a unit of its own, whose epilogue needs no other CTA.
struct Run {
  Walk w;
  int first, count;
};
static_assert(sizeof(Run) <= 48, "run slot");

// Walks the units of the runs in order: unit w, its pages [seg0, seg0 + npg()).
struct Cursor {
  Walk w;
  int seg0, left, run, nruns;
  __device__ __forceinline__ int npg() const { return min(w.P - seg0, left); }
  __device__ __forceinline__ void start(const Run* runs, int n) {
    nruns = n;
    run = 0;
    w = runs[0].w;
    seg0 = runs[0].first;
    left = runs[0].count;
  }
  // false past the last unit
  __device__ __forceinline__ bool next(const DecodeParams& p, const Run* runs) {
    left -= npg();
    if (left > 0) {
      w.next(p);
      seg0 = 0;
      return true;
    }
    if (++run >= nruns) return false;
    w = runs[run].w;
    seg0 = runs[run].first;
    left = runs[run].count;
    return true;
  }
};

// The runs of range [r0, r1), w0 = the unit holding r0; returns how many (1 to 3).
__device__ __forceinline__ int plan_runs(const DecodeParams& p, const Walk& w0, long long r0,
                                         long long r1, Run* runs) {
  Walk wt = w0;
  while (wt.S + wt.P < r1) wt.next(p);  // the unit holding r1 - 1
  if (wt.S <= r0) {                     // the range lies inside one unit
    runs[0] = Run{w0, static_cast<int>(r0 - w0.S), static_cast<int>(r1 - r0)};
    return 1;
  }
  const long long h1 = w0.S + w0.P;  // end of the unit holding r0 (<= wt.S)
  runs[0] = Run{wt, 0, static_cast<int>(r1 - wt.S)};
  runs[1] = Run{w0, static_cast<int>(r0 - w0.S), static_cast<int>(h1 - r0)};
  if (h1 == wt.S) return 2;
  Walk wm = w0;
  wm.next(p);
  runs[2] = Run{wm, 0, static_cast<int>(wt.S - h1)};
  return 3;
}

// The consumer warps' barrier: all kNW of them, or those with rows (row-split).
__device__ __forceinline__ void bar_consumers(int nthreads) {
  asm volatile("bar.sync 1, %0;" ::"r"(nthreads) : "memory");
}

// What a unit epilogue reads and writes (passed by value: the epilogue functions are
// not inlined, so the consumer warps' end-of-range call runs the code the merge warp
// has already brought into the instruction cache mid-kernel).
struct Epi {
  __nv_bfloat16* out;
  float* lse;
  float* part_lse;
  float* part_o;
  const float* v_scale;
  int num_q_heads, group, q_len;
  // output row of query row i = t * group + g of unit (b, h): token t, head h * group + g
  __device__ __forceinline__ size_t out_row(int b, int h, int i) const {
    const int t = i / group, g = i - t * group;
    return (static_cast<size_t>(b) * q_len + t) * num_q_heads + h * group + g;
  }
};

// This CTA's state of query row g, columns 8 cc .. 8 cc + 7, from the consumer warps'
// states in the merge buffer (M = max m_w, l = sum l_w 2^(m_w - M), O likewise; in the
// row-split form a row has one state); poisoned if a warp's state was.
template <int D, bool kFp8, int NT, bool kRS>
__device__ __forceinline__ void cta_state(const float* wob, const float* wmlb, int g, int cc,
                                          float& M, float& lsum, float (&o)[8],
                                          bool& poisoned) {
  using C = Cfg<D, kFp8, NT, kRS>;
  constexpr int kRows = C::kRows;
  M = -INFINITY;
  poisoned = false;
#pragma unroll
  for (int ww = 0; ww < C::kStateWarps; ++ww) {
    M = fmaxf(M, wmlb[(ww * kRows + g) * 2]);
    poisoned |= isnan(wmlb[(ww * kRows + g) * 2 + 1]);
  }
  lsum = 0.f;
#pragma unroll
  for (int q = 0; q < 8; ++q) o[q] = 0.f;
#pragma unroll
  for (int ww = 0; ww < C::kStateWarps; ++ww) {
    const float mw = wmlb[(ww * kRows + g) * 2];
    const float wt = mw == -INFINITY ? 0.f : ex2(mw - M);
    lsum += wmlb[(ww * kRows + g) * 2 + 1] * wt;
    const float4* src = reinterpret_cast<const float4*>(wob + (ww * kRows + g) * C::kLd + cc * 8);
    const float4 x = src[0], y = src[1];
    o[0] += x.x * wt; o[1] += x.y * wt; o[2] += x.z * wt; o[3] += x.w * wt;
    o[4] += y.x * wt; o[5] += y.y * wt; o[6] += y.z * wt; o[7] += y.w * wt;
  }
}

// Unit epilogue, run by nt threads (t = this thread's index among them).
// combine_unit: this CTA's state of unit (b, h) (cta_state) -> the output, or, for a
// unit cut by range boundaries (nseg > 1), this CTA's partial (slot 0 or 1).
template <int D, bool kFp8, int NT, bool kRS = false>
__device__ __noinline__ void combine_unit(const Epi e, int b, int h, int nseg, int slot,
                                          const float* wob, const float* wmlb, int t, int nt) {
  using C = Cfg<D, kFp8, NT, kRS>;
  constexpr int kRows = C::kRows;
  const int R = e.group * e.q_len;  // the unit's query rows (<= kRows)
  constexpr int kChunks = D / 8;  // 8 consecutive d per work item
  const float vsc = kFp8 ? __ldg(e.v_scale + h) : 1.f;
  for (int it = t; it < R * kChunks; it += nt) {
    const int g = it / kChunks, cc = it % kChunks;  // g: the query row
    float M, lsum, o[8];
    bool poisoned;
    cta_state<D, kFp8, NT, kRS>(wob, wmlb, g, cc, M, lsum, o, poisoned);
    // (a row that saw no key in this CTA's part of a unit, e.g. a draft token whose last
    // key lies before the part, has lsum = 0: its partial is 0 with lse -inf)
    const float inv = lsum > 0.f ? 1.f / lsum : 0.f;
    const size_t row = e.out_row(b, h, g);
    if (nseg == 1) {
      uint4 pk = make_uint4(0, 0, 0, 0);
      if (!poisoned) {
        const float f = inv * vsc;
        pk = make_uint4(pack_bf16(o[0] * f, o[1] * f), pack_bf16(o[2] * f, o[3] * f),
                        pack_bf16(o[4] * f, o[5] * f), pack_bf16(o[6] * f, o[7] * f));
      }
      reinterpret_cast<uint4*>(e.out + row * D)[cc] = pk;
      if (cc == 0 && e.lse) e.lse[row] = poisoned ? -INFINITY : (M + log2f(lsum)) * kLn2;
    } else {
      const size_t ps = (static_cast<size_t>(blockIdx.x) * 2 + slot) * kRows + g;
      float4* dst = reinterpret_cast<float4*>(e.part_o + ps * D + cc * 8);
      dst[0] = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
      dst[1] = make_float4(o[4] * inv, o[5] * inv, o[6] * inv, o[7] * inv);
      if (cc == 0) e.part_lse[ps] = poisoned ? INFINITY : M + log2f(lsum);
    }
  }
}

// merge_rows: the last of the unit's CTAs to arrive merges their partials. The unit
// starts at page S; CTA c (range [c * chunk, ...)) keeps it in slot 0 when the unit
// starts at or before its range (its first unit), else in slot 1 (its last). Partials
// are taken four at a time: a group's loads are all issued before any is used, then
// merged into a running (M, l, O); kItems work items (row, 8 values) go at once, their
// loads in flight together (the arithmetic of an item does not depend on kItems, so
// every caller gets the same bits). With wob/wmlb (the merge buffer of this CTA's
// state) this CTA's partial is not read back but formed from its state, with the
// arithmetic combine_unit uses to write it, so the result is the same bit for bit.
template <int D, bool kFp8, int NT, bool kRS, int kItems>
__device__ __forceinline__ void merge_rows(const Epi& e, int b, int h, long long S, int P,
                                           long long chunk, int t, int nt, int row0, int row1,
                                           const float* wob, const float* wmlb) {
  constexpr int kRows = Cfg<D, kFp8, NT, kRS>::kRows;
  const int R = min(e.group * e.q_len, row1) - row0;  // rows row0 .. row1-1 of the unit
  constexpr int kChunks = D / 8;
  constexpr int kGroup = 4;
  const float vsc = kFp8 ? __ldg(e.v_scale + h) : 1.f;
  const long long c_first = S / chunk, c_last = (S + P - 1) / chunk;
  for (int it0 = t; it0 < R * kChunks; it0 += kItems * nt) {
    int g[kItems], cc[kItems];
    bool live[kItems];
    float M[kItems], lsum[kItems], o[kItems][8];
    bool any_bad[kItems];
#pragma unroll
    for (int v = 0; v < kItems; ++v) {
      const int it = it0 + v * nt;
      live[v] = it < R * kChunks;
      g[v] = row0 + (live[v] ? it : it0) / kChunks;
      cc[v] = (live[v] ? it : it0) % kChunks;
      M[v] = -INFINITY;
      lsum[v] = 0.f;
#pragma unroll
      for (int q = 0; q < 8; ++q) o[v][q] = 0.f;
      any_bad[v] = false;
    }
    for (long long base = c_first; base <= c_last; base += kGroup) {
      float ls[kItems][kGroup];
      float4 x[kItems][kGroup], y[kItems][kGroup];
#pragma unroll
      for (int v = 0; v < kItems; ++v) {
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
          const long long cta = base + k;
          ls[v][k] = -INFINITY;
          x[v][k] = y[v][k] = make_float4(0.f, 0.f, 0.f, 0.f);
          if (!live[v]) continue;
          if (wob != nullptr && cta == blockIdx.x) {
            float Mo, lo, oo[8];
            bool po;
            cta_state<D, kFp8, NT, kRS>(wob, wmlb, g[v], cc[v], Mo, lo, oo, po);
            const float inv = lo > 0.f ? 1.f / lo : 0.f;
            ls[v][k] = po ? INFINITY : Mo + log2f(lo);
            x[v][k] = make_float4(oo[0] * inv, oo[1] * inv, oo[2] * inv, oo[3] * inv);
            y[v][k] = make_float4(oo[4] * inv, oo[5] * inv, oo[6] * inv, oo[7] * inv);
          } else if (cta <= c_last) {
            const size_t ps =
                static_cast<size_t>(cta * 2 + (S <= cta * chunk ? 0 : 1)) * kRows + g[v];
            const float4* src = reinterpret_cast<const float4*>(e.part_o + ps * D + cc[v] * 8);
            ls[v][k] = __ldcg(e.part_lse + ps);
            x[v][k] = __ldcg(src);
            y[v][k] = __ldcg(src + 1);
          }
        }
      }
#pragma unroll
      for (int v = 0; v < kItems; ++v) {
        float Mn = M[v];
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
          any_bad[v] |= ls[v][k] == INFINITY;
          Mn = fmaxf(Mn, ls[v][k]);
        }
        if (Mn == INFINITY) continue;  // a poisoned partial: the result is discarded
        const float a = M[v] == -INFINITY ? 0.f : ex2(M[v] - Mn);
        lsum[v] *= a;
#pragma unroll
        for (int q = 0; q < 8; ++q) o[v][q] *= a;
#pragma unroll
        for (int k = 0; k < kGroup; ++k) {
          const float wt = ls[v][k] == -INFINITY ? 0.f : ex2(ls[v][k] - Mn);
          lsum[v] += wt;
          o[v][0] += x[v][k].x * wt; o[v][1] += x[v][k].y * wt;
          o[v][2] += x[v][k].z * wt; o[v][3] += x[v][k].w * wt;
          o[v][4] += y[v][k].x * wt; o[v][5] += y[v][k].y * wt;
          o[v][6] += y[v][k].z * wt; o[v][7] += y[v][k].w * wt;
        }
        M[v] = Mn;
      }
    }
#pragma unroll
    for (int v = 0; v < kItems; ++v) {
      if (!live[v]) continue;
      const size_t row = e.out_row(b, h, g[v]);
      uint4 pk = make_uint4(0, 0, 0, 0);
      if (!any_bad[v]) {
        const float f = vsc / lsum[v];
        pk = make_uint4(pack_bf16(o[v][0] * f, o[v][1] * f), pack_bf16(o[v][2] * f, o[v][3] * f),
                        pack_bf16(o[v][4] * f, o[v][5] * f), pack_bf16(o[v][6] * f, o[v][7] * f));
      }
      reinterpret_cast<uint4*>(e.out + row * D)[cc[v]] = pk;
      if (cc[v] == 0 && e.lse)
        e.lse[row] = any_bad[v] ? -INFINITY : (M[v] + log2f(lsum[v])) * kLn2;
    }
  }
}

// merge_rows one item at a time, as one non-inlined copy (for the consumer warps'
// last unit, whose registers are in use around the call)
template <int D, bool kFp8, int NT, bool kRS = false>
__device__ __noinline__ void merge_partials(const Epi e, int b, int h, long long S, int P,
                                            long long chunk, int t, int nt, int row0 = 0,
                                            int row1 = 1 << 30, const float* wob = nullptr,
                                            const float* wmlb = nullptr) {
  merge_rows<D, kFp8, NT, kRS, 1>(e, b, h, S, P, chunk, t, nt, row0, row1, wob, wmlb);
}

// Arrival on a unit's ticket, wrapping to 0 on the last of `count` arrivals (so the
// counter is ready for the next call). Release: this thread's writes, and those it has
// seen through a barrier, are visible before the count moves; acquire: the arrival
// that sees count - 1 sees every other arrival's writes. Returns true for that one.
__device__ __forceinline__ bool ticket_last(int* counter, int count) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.inc.u32 %0, [%1], %2;"
               : "=r"(old)
               : "l"(counter), "r"(static_cast<unsigned>(count - 1))
               : "memory");
  return old == static_cast<unsigned>(count - 1);
}

// Arrivals on a unit's ticket so far, read with acquire: when it shows every other CTA
// of the unit, their partials are visible to this thread (and, through a later CTA
// barrier, to the others).
__device__ __forceinline__ unsigned ticket_peek(const int* counter) {
  unsigned v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(counter) : "memory");
  return v;
}

// Segments of unit w over the CTA ranges, and which partial slot this CTA uses.
__device__ __forceinline__ int unit_segments(const Walk& w, long long chunk) {
  return static_cast<int>((w.S + w.P - 1) / chunk - w.S / chunk + 1);
}

// The merge warp: the epilogue of every unit of this CTA's range but the last (the
// consumer warps, which have nothing left to stream then, do that one together), so
// the consumers hand a unit over and go straight on to the next.
template <int D, bool kFp8, int NT, bool kRS>
__device__ __forceinline__ void merge_units(const DecodeParams& p, const Epi epi,
                                            const Run* runs, int nruns, long long r0,
                                            long long chunk, const float* wo,
                                            const float* wml, uint64_t* unit_done,
                                            uint64_t* merge_free) {
  const int lane = threadIdx.x & 31;
  Cursor cur;
  cur.start(runs, nruns);
  for (int cu = 0;; ++cu) {
    const Walk w = cur.w;
    if (!cur.next(p, runs)) return;  // w is the range's last unit
    using C = Cfg<D, kFp8, NT, kRS>;
    constexpr int kBufs = C::kMergeBufs;
    const int mb = cu % kBufs;
    if (!__all_sync(0xffffffffu, mbar_wait(&unit_done[mb], (cu / kBufs) & 1, p.wait_ns))) {
      if (lane == 0) record_status(p.dev_status, PGQA_ETIMEOUT);
      return;
    }
    const int nseg = unit_segments(w, chunk);
    combine_unit<D, kFp8, NT, kRS>(epi, w.b, w.h, nseg, w.S <= r0 ? 0 : 1,
                                   wo + mb * C::kMergeFloats, wml + mb * C::kMlFloats, lane, 32);
    __syncwarp();  // every lane has read the buffer and issued its writes
    if (lane == 0) mbar_arrive(&merge_free[mb]);
    if (nseg > 1) {
      bool last = false;
      if (lane == 0) last = ticket_last(p.counters + w.b * p.num_kv_heads + w.h, nseg);
      last = __shfl_sync(0xffffffffu, last, 0);
      __syncwarp();  // the lanes' reads of the partials come after lane 0's acquire
      // (inline, two items at a time: the merge warp has its registers to itself)
      if (last)
        merge_rows<D, kFp8, NT, kRS, 2>(epi, w.b, w.h, w.S, w.P, chunk, lane, 32, 0, 1 << 30,
                                        nullptr, nullptr);
    }
  }
}

template <int D, bool kFp8, int NT, bool kRS>
__global__ void __launch_bounds__(kThreads, (ctas_per_sm<D, kFp8, NT, kRS>()))
    paged_decode_kernel(const __grid_constant__ CUtensorMap kmap,
                        const __grid_constant__ CUtensorMap vmap, const DecodeParams p,
                        const DecodeAppend ap) {
  using C = Cfg<D, kFp8, NT, kRS>;
  // row-split: consumer warp w holds row tile w (rows 8w .. 8w+7) of every unit and
  // reads every page; kRT of them have rows (the others leave at once)
  const int kRT = kRS ? (p.group * p.q_len + 7) / 8 : 1;
  constexpr int kRows = C::kRows;
  constexpr int S = C::kStages;
  constexpr int SPW = C::kStagesPerWarp;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  float* wo = reinterpret_cast<float*>(smem + C::kOffMerge);  // [bufs][kNW][kRows][D]
  float* wml = reinterpret_cast<float*>(smem + C::kOffMl);    // [bufs][kNW][kRows][2] (m, l)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* empty = full + S;
  uint64_t* unit_done = empty + S;       // [2] the consumer warps' states of a unit are in
  uint64_t* merge_free = unit_done + 2;  // [2] the merge warp has read them
  int* meta = reinterpret_cast<int*>(smem + C::kOffMeta);  // per stage: bad block id seen
  int* yring = reinterpret_cast<int*>(smem + C::kOffY);    // row coordinate of page i % kYRing
  int* yring2 = reinterpret_cast<int*>(smem + C::kOffY2);  // its second 8-row block (block 8)
  // misc[1]: the last-unit ticket result; [2]: number of runs
  int* misc = reinterpret_cast<int*>(smem + C::kOffMisc);
  long long* scratch = reinterpret_cast<long long*>(misc + 32);  // kScanSlots slots
  Run* runs = reinterpret_cast<Run*>(smem + C::kOffRuns);         // the range's order, w0

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int c = blockIdx.x, ncta = gridDim.x;
  const int G = p.group, Hkv = p.num_kv_heads, B = p.num_seqs;
  const Epi epi{p.out, p.lse, p.part_lse, p.part_o, p.v_scale, p.num_q_heads, p.group, p.q_len};
  if (warp == kWarpProd && lane == 0) {
    tma_prefetch_desc(&kmap);
    tma_prefetch_desc(&vmap);
  }
  grid_launch_dependents();  // the next kernel may place its CTAs as these exit
  // Up to grid_dependency_wait() below, this CTA reads only context lengths and block
  // tables, which no kernel of this library writes: the plan below may run while the
  // stream's previous kernel finishes (programmatic launch).

  // ---- the barriers, one per thread
  for (int i = tid; i < 2 * S + 4; i += kThreads) {
    if (i < S) mbar_init(&full[i], 1);
    else if (i < 2 * S) mbar_init(&empty[i - S], kRS ? kRT : 1);  // row-split: every warp
                                                                     // with rows frees it
    else if (i < 2 * S + 2) mbar_init(&unit_done[i - 2 * S], kRS ? kRT : kNW);
    else mbar_init(&merge_free[i - 2 * S - 2], 1);
    fence_mbar_init();
  }

  // ---- context lengths: sequence tid's (the first kThreads sequences in one load each,
  //      kept in a register) and sequence c's, whose block-table entries this CTA asks
  //      L2 for (the producers will read them soon), all loaded together
  const int L_t = tid < B ? __ldg(p.context_lens + tid) : 0;
  const int L_c = c < B ? __ldg(p.context_lens + c) : 0;
  for (int b = c; b < B; b += ncta) {
    const int L = b == c ? L_c : __ldg(p.context_lens + b);
    const int e0 = first_key(p, L) / p.block_size, e1 = (L + p.block_size - 1) / p.block_size;
    const int32_t* row = p.block_tables + static_cast<size_t>(b) * p.max_blocks_per_seq;
    for (int e = e0 + tid * 32; e < e1 && e < p.max_blocks_per_seq; e += kThreads * 32)
      prefetch_l2(row + e);
  }

  // ---- the global page order holds N pages; this CTA owns [r0, r1). One scan over the
  //      sequences' pages gives N and each sequence's place in the order; the thread
  //      whose sequence holds r0 publishes that unit (w0). Batches of more than kThreads
  //      sequences take the scan chunk by chunk.
  Walk* w0s = reinterpret_cast<Walk*>(runs + 3);
  long long N, incl0, tot0;
  const long long P_t = tid < B ? pages_of_len(p, L_t) : 0;
  incl0 = block_scan(P_t, scratch, &tot0);
  if (B <= kThreads) {
    N = static_cast<long long>(Hkv) * tot0;
  } else {
    long long local = 0;
    for (int b = tid + kThreads; b < B; b += kThreads) local += pages_of(p, b);
    N = static_cast<long long>(Hkv) * (tot0 + block_sum(local, scratch));
  }
  long long chunk = N > 0 ? (N + ncta - 1) / ncta : 0;
  if (chunk > 0 && chunk < kMinChunk) chunk = kMinChunk;
  const long long r0 = static_cast<long long>(c) * chunk;
  const long long r1 = r0 + chunk < N ? r0 + chunk : N;
  // (scan chunk k covers sequences k kThreads ..; the first is scanned already)
  long long running = 0;  // pages of the sequences before the chunk
  for (int base = 0; r0 < r1 && base < B; base += kThreads) {
    const int b = base + tid;
    long long P = P_t, incl = incl0, tot = tot0;
    int L = L_t;
    if (base > 0) {
      L = b < B ? __ldg(p.context_lens + b) : 0;
      P = b < B ? pages_of_len(p, L) : 0;
      incl = block_scan(P, scratch, &tot);
    }
    const long long s0 = static_cast<long long>(Hkv) * (running + incl - P);
    if (P > 0 && s0 <= r0 && r0 < s0 + Hkv * P) {
      Walk w;
      w.b = b;
      w.P = static_cast<int>(P);
      w.fp = first_key(p, L) >> 4;
      w.L = L;
      w.h = static_cast<int>((r0 - s0) / P);
      w.S = s0 + static_cast<long long>(w.h) * P;
      *w0s = w;
    }
    running += tot;
    if (running * Hkv > r0) break;  // (uniform: the unit holding r0 is in this chunk)
    __syncthreads();                // (scratch is reused by the next chunk's scan)
  }
  __syncthreads();
  const Walk w0 = r0 < r1 ? *w0s : Walk{};

  if (tid == 0) misc[2] = r0 < r1 ? plan_runs(p, w0, r0, r1, runs) : 0;
  __syncthreads();

  // ---- the producer's fetch cursor: row coordinates of this CTA's pages, read from
  //      the block tables into yring; the first 32 before the wait
  const int n = static_cast<int>(r1 - r0);  // pages of this CTA, CTA-local index 0..n-1
  const int nruns = misc[2];
  // fetch cursor: run, unit and page within it, pages left in the run
  int frun = 0;
  Walk fw = nruns > 0 ? runs[0].w : w0;
  int fpg = nruns > 0 ? runs[0].first : 0, fleft = nruns > 0 ? runs[0].count : 0;
  int fetched = 0;  // pages whose row coordinate is in yring (CTA-local order)
  auto fetch_rows = [&]() {
    const int cnt = min(32, min(fw.P - fpg, fleft));
    if (lane < cnt) {
      // cache rows of 16-token page lp: one block of 16, half of a block of 32, or
      // two blocks of 8 (the second only if the context reaches it)
      const int32_t* btb = p.block_tables + static_cast<size_t>(fw.b) * p.max_blocks_per_seq;
      const int lp = fw.fp + fpg + lane, bs = p.block_size;
      const int blk = bs == 32 ? lp >> 1 : bs == 8 ? 2 * lp : lp;
      const int32_t pbn = __ldg(btb + blk);
      const bool ok0 = pbn >= 0 && pbn < p.num_blocks;
      int y0 = ok0 ? (pbn * Hkv + fw.h) * bs + (bs == 32 ? (lp & 1) * 16 : 0) : -1, y1 = 0;
      if (bs == 8) {
        const int32_t pbn1 = (blk + 1) * 8 < fw.L ? __ldg(btb + blk + 1) : pbn;
        y1 = (pbn1 >= 0 && pbn1 < p.num_blocks) ? (pbn1 * Hkv + fw.h) * 8 : -1;
      }
      yring[(fetched + lane) % kYRing] = y0;
      yring2[(fetched + lane) % kYRing] = y1;
    }
    fetched += cnt;
    fpg += cnt;
    fleft -= cnt;
    if (fleft == 0) {
      if (++frun < nruns) {
        fw = runs[frun].w;
        fpg = runs[frun].first;
        fleft = runs[frun].count;
      }
    } else if (fpg == fw.P) {
      fw.next(p);
      fpg = 0;
    }
    __syncwarp();
  };
  if (warp == kWarpProd && n > 0) fetch_rows();

  grid_dependency_wait();  // the stream's previous kernel (e.g. the KV append) is done

  // ---- sequences with nothing to read (empty or invalid), spread over the CTAs:
  //      out = 0, lse = -inf
  for (int b = c; b < B; b += ncta) {
    bool valid;
    if (pages_of(p, b, &valid) != 0) continue;
    if (!valid && tid == 0) record_status(p.dev_status, PGQA_EINVAL);
    for (int i = tid; i < p.q_len * p.num_q_heads * (D / 8); i += kThreads) {
      const size_t row = static_cast<size_t>(b) * p.q_len * p.num_q_heads + i / (D / 8);
      reinterpret_cast<uint4*>(p.out + row * D)[i % (D / 8)] = make_uint4(0, 0, 0, 0);
      if (i % (D / 8) == 0 && p.lse) p.lse[row] = -INFINITY;
    }
  }
  if (r0 >= r1) return;

  // ================================================================ producer
  if (warp == kWarpProd) {
    // lane w < kNW serves consumer warp w: its pages are w, w + kNW, ... (row-split:
    // lane 0 serves the one ring every consumer warp reads, all pages in order)
    constexpr int kPW = kRS ? 1 : kNW;       // page streams
    constexpr int kSPW = kRS ? S : SPW;      // stages per stream
    const int nw_pages = lane < kPW && n > lane ? (n - lane + kPW - 1) / kPW : 0;
    int next_li = 0;  // next local index of that stream to issue
    uint64_t idle_since = 0;
    for (;;) {
      const int pend = __reduce_min_sync(
          0xffffffffu, lane < kPW && next_li < nw_pages ? lane + kPW * next_li : INT_MAX);
      if (pend == INT_MAX) break;  // every page issued
      bool progress = false;
      // refill stream `lane`'s next stage if it is free
      if (lane < kPW && next_li < nw_pages) {
        const int i = lane + kPW * next_li;
        const int s = lane * kSPW + next_li % kSPW, use = next_li / kSPW;
        if (i < fetched && (use == 0 || mbar_try_wait(&empty[s], (use - 1) & 1))) {
          int y = yring[i % kYRing], y1 = yring2[i % kYRing];
          int bad = 0;
          if (y < 0 || y1 < 0) {
            bad = 1;
            y = y1 = 0;  // load a valid page; the unit's result is discarded
            record_status(p.dev_status, PGQA_EBADINDEX);
          }
          meta[s] = bad;
          uint8_t* st = ring + s * C::kStageBytes;
          mbar_arrive_expect_tx(&full[s], C::kStageBytes);
          if constexpr (C::kPack) {  // the tensor maps count 128-byte rows
            y >>= 1;
            y1 >>= 1;
          }
          if (p.block_size != 8) {  // one 16-row box per 128-byte column block
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub)
              tma_load_2d(st + sub * 2048, &kmap, &full[s], sub * (128 / C::kElem), y);
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub)
              tma_load_2d(st + C::kPageBytes + sub * 2048, &vmap, &full[s],
                          sub * (128 / C::kElem), y);
          } else {  // two 8-row boxes (rows 8-15 land half a page in: same swizzle phase)
            constexpr int kHalf = C::kPack ? 512 : 1024;
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub) {
              tma_load_2d(st + sub * 2048, &kmap, &full[s], sub * (128 / C::kElem), y);
              tma_load_2d(st + sub * 2048 + kHalf, &kmap, &full[s], sub * (128 / C::kElem), y1);
              tma_load_2d(st + C::kPageBytes + sub * 2048, &vmap, &full[s],
                          sub * (128 / C::kElem), y);
              tma_load_2d(st + C::kPageBytes + sub * 2048 + kHalf, &vmap, &full[s],
                          sub * (128 / C::kElem), y1);
            }
          }
          ++next_li;
          progress = true;
        }
      }
      // then fetch up to 32 more row coordinates of the current unit while fewer than
      // 64 are ahead of the issue cursor (a table read stalls this warp; the loads
      // above are out by then), never overwriting an entry still to be issued
      if (fetched < n && fetched < pend + 64) {
        fetch_rows();
        progress = true;
      }
      if (__any_sync(0xffffffffu, progress)) {
        idle_since = 0;
      } else if (idle_since == 0) {
        idle_since = globaltimer_ns();
      } else if (globaltimer_ns() - idle_since > p.wait_ns) {
        if (lane == 0) record_status(p.dev_status, PGQA_ETIMEOUT);
        break;
      }
    }
    // No TMA write may land after this CTA exits: wait for the last fill of each
    // stage (complete already on the normal path).
    if (lane < kPW) {
      for (int k = 0; k < kSPW && k < next_li; ++k) {
        const int last_li = k + ((next_li - 1 - k) / kSPW) * kSPW;
        if (!mbar_wait(&full[lane * kSPW + k], (last_li / kSPW) & 1))
          record_status(p.dev_status, PGQA_ETIMEOUT);
      }
    }
    return;
  }

  // ================================================================ merge warp
  if (warp == kWarpMerge) {
    merge_units<D, kFp8, NT, kRS>(p, epi, runs, nruns, r0, chunk, wo, wml, unit_done,
                                  merge_free);
    return;
  }

  // ================================================================ consumers
  const int gid = lane >> 2, tig = lane & 3;
  const uint32_t rowK = (lane & 7) + (((lane >> 3) & 1) << 3);
  const uint32_t cK = lane >> 4;
  const uint32_t rowV = (lane & 7) + ((lane >> 4) << 3);
  const uint32_t cV = (lane >> 3) & 1;
  // this lane's swizzled fragment offsets within a 128-byte column block, computed once
  // (per page each load is then one add): K for the four 16-element chunks q = kc & 3
  // (E4M3: the pair kc = 2q); V for the four chunks (bf16) or the four key rows this
  // lane reads (E4M3)
  uint32_t offK[4], offV[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    offK[q] = C::kPack ? swz128(rowK >> 1, (rowK & 1) * 4 + 2 * q + cK) : swz128(rowK, 2 * q + cK);
    if constexpr (!kFp8) {
      offV[q] = swz128(rowV, 2 * q + cV);
    } else if constexpr (C::kPack) {  // 8 bytes: rows 2 tig .. (two tokens per shared row)
      offV[q] = swz128(tig + (q >> 1) * 4, (q & 1) * 4 + (gid >> 1)) + (gid & 1) * 8;
    } else {
      offV[q] = swz128(2 * tig + (q & 1) + (q >> 1) * 8, gid);
    }
  }
  const int R = G * p.q_len;  // query rows of a unit: row i = token i / G, head i % G
  const int rbase = kRS ? 8 * warp : 0;  // row-split: this warp's row tile
  if (kRS && warp >= kRT) return;        // (no rows: not counted by the stage barriers)
  bool alive = true;  // false once one of this warp's waits gave up
  int i_base = 0;     // CTA-local index of the unit's first page
  int cu = 0;         // units of this CTA done so far
  // raw query words of a unit, column n = query row 8 nt + gid of the unit:
  //   bf16: the two B-fragment registers per 16-wide chunk as stored;
  //   E4M3: k index 2tig+{0,1} <-> d = 16kc + 4tig + {0,1}; 2tig+8+{0,1} <-> +{2,3}
  uint32_t qraw[C::kNkc][NT][2];
  auto load_q = [&](const Walk& u) {
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int i = rbase + 8 * nt + gid;
      const bool live = i < R;
      const int t = live ? i / G : 0, g = live ? i - t * G : 0;
      const __nv_bfloat16* qrow =
          p.q + ((static_cast<size_t>(u.b) * p.q_len + t) * p.num_q_heads + u.h * G + g) * D;
#pragma unroll
      for (int kc = 0; kc < C::kNkc; ++kc) {
        if constexpr (!kFp8) {
          const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow + 16 * kc + 2 * tig);
          qraw[kc][nt][0] = live ? __ldg(q32) : 0u;
          qraw[kc][nt][1] = live ? __ldg(q32 + 4) : 0u;
        } else {
          const uint2 q4 = live ? __ldg(reinterpret_cast<const uint2*>(qrow + 16 * kc + 4 * tig))
                                : make_uint2(0, 0);
          qraw[kc][nt][0] = q4.x;
          qraw[kc][nt][1] = q4.y;
        }
      }
    }
  };
  // keys a column of the fragment (query row 8 nt + 2 tig + c) sees fewer than the last
  // key of the context: q_len - 1 - its token (0 for single-token decode)
  auto key_shift = [&](int nt, int c) {
    const int i = rbase + 8 * nt + 2 * tig + c;
    return i < R ? p.q_len - 1 - i / G : 0;
  };
  Cursor cur;
  cur.start(runs, nruns);
  if (NT == 1) load_q(cur.w);
  for (bool more = true; more;) {
    const Walk w = cur.w;
    const int seg0 = cur.seg0, npg = cur.npg();
    Cursor nxt = cur;  // the next unit, if any
    more = nxt.next(p, runs);
    const int L = __ldg(p.context_lens + w.b);
    const int kfirst = first_key(p, L);
    // the range's last unit, when cut: the other CTAs' arrivals on its ticket, read now
    // so that the load is out of the way by the unit's end
    unsigned peek = 0;
    if (!more && tid == 0 && unit_segments(w, chunk) > 1)
      peek = ticket_peek(p.counters + w.b * Hkv + w.h);

    // Q^T fragments (B operand) of this unit; single-row-tile units start loading the
    // next unit's here (the multi-token form loads its larger fragments unit by unit)
    if (NT > 1) load_q(w);
    uint32_t qf[C::kNkc][NT][2];
#pragma unroll
    for (int kc = 0; kc < C::kNkc; ++kc) {
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        if constexpr (!kFp8) {
          qf[kc][nt][0] = qraw[kc][nt][0];
          qf[kc][nt][1] = qraw[kc][nt][1];
        } else {
          qf[kc][nt][0] = pack_f16(bf16_lo(qraw[kc][nt][0]), bf16_hi(qraw[kc][nt][0]));
          qf[kc][nt][1] = pack_f16(bf16_lo(qraw[kc][nt][1]), bf16_hi(qraw[kc][nt][1]));
        }
      }
    }
    if (NT == 1 && more) load_q(nxt.w);
    int dq[NT][2];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      dq[nt][0] = key_shift(nt, 0);
      dq[nt][1] = key_shift(nt, 1);
    }

    // fused append: the page holding key L-1, if this warp reads it (segment-relative),
    // this lane's 16-byte chunk of the new K (lanes 0..kAppLanes-1) or V row, still
    // bf16 (E4M3: two loads, quantised when the page comes), and the row's block id
    constexpr int kAppLanes = C::kRowBytes / 16;
    int app_j = -1, app_pbn = -1;
    uint4 app_x0 = make_uint4(0, 0, 0, 0), app_x1 = app_x0;
    if (ap.key != nullptr) {
      const int jl = (L - 1) / 16 - w.fp - seg0;
      if (jl >= 0 && jl < npg && (i_base + jl) % kNW == warp) {
        app_j = jl;
        if (lane < 2 * kAppLanes) {
          const int c = lane % kAppLanes;
          const uint4* src = (lane < kAppLanes ? ap.key : ap.value) +
                             (static_cast<size_t>(w.b) * Hkv + w.h) * (D / 8);
          if constexpr (!kFp8) {
            app_x0 = __ldg(src + c);
          } else {
            app_x0 = __ldg(src + 2 * c);
            app_x1 = __ldg(src + 2 * c + 1);
          }
        }
        app_pbn = __ldg(p.block_tables + static_cast<size_t>(w.b) * p.max_blocks_per_seq +
                        (L - 1) / p.block_size);
      }
    }

    const float sl2 = p.scale_log2 * (kFp8 ? __ldg(p.k_scale + w.h) : 1.f);
    float m_run[NT][2], l_run[NT][2];
    float acc[C::kNkc][NT][4];
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      m_run[nt][0] = m_run[nt][1] = -INFINITY;
      l_run[nt][0] = l_run[nt][1] = 0.f;
#pragma unroll
      for (int i = 0; i < C::kNkc; ++i)
        acc[i][nt][0] = acc[i][nt][1] = acc[i][nt][2] = acc[i][nt][3] = 0.f;
    }
    int bad = 0;

    // this warp's pages of the unit: CTA-local index i = i_base + j with i % kNW == warp
    // (row-split: every page, from the one ring in page order)
    for (int j = kRS ? 0 : (warp - i_base % kNW + kNW) % kNW; j < npg && alive;
         j += kRS ? 1 : kNW) {
      if constexpr (kRS && !kFp8) {
        // Row-split over a bf16 cache, two pages a step while two are left: both pages'
        // S^T, one online-softmax step over their 32 keys, both P.V. A page's softmax is
        // a dependency chain the next page cannot start before; taking two pages per
        // chain halves the chains. (The row-split form never appends, and only a unit's
        // last page can be partial, so page a here is whole.)
        static_assert(!kRS || NT == 1, "one row tile per warp in the row-split form");
        if (j + 1 < npg) {
          const int ia = i_base + j, ib = ia + 1;
          const int sa = ia % S, sb = ib % S;
          if (!mbar_wait(&full[sa], (ia / S) & 1, p.wait_ns) ||
              !mbar_wait(&full[sb], (ib / S) & 1, p.wait_ns)) {
            alive = false;
            record_status(p.dev_status, PGQA_ETIMEOUT);
            break;
          }
          bad |= meta[sa] | meta[sb];
          const uint32_t stKa = smem_u32(ring + sa * C::kStageBytes);
          const uint32_t stKb = smem_u32(ring + sb * C::kStageBytes);
          float sc[4] = {0.f, 0.f, 0.f, 0.f}, sd[4] = {0.f, 0.f, 0.f, 0.f};
          float tc[4] = {0.f, 0.f, 0.f, 0.f}, td[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int kc = 0; kc < C::kNkc; ++kc) {
            uint32_t a0, a1, a2, a3, b0, b1, b2, b3;
            ldsm_x4(stKa + (kc >> 2) * 2048 + offK[kc & 3], a0, a1, a2, a3);
            ldsm_x4(stKb + (kc >> 2) * 2048 + offK[kc & 3], b0, b1, b2, b3);
            mma_bf16((kc & 1) ? sd : sc, a0, a1, a2, a3, qf[kc][0][0], qf[kc][0][1]);
            mma_bf16((kc & 1) ? td : tc, b0, b1, b2, b3, qf[kc][0][0], qf[kc][0][1]);
          }
          const int pka = (w.fp + seg0 + j) * 16, pkb = pka + 16;
          const int nvb = min(16, L - pkb);  // page b's rows holding keys < L
          const int loa = max(0, kfirst - pka), lob = max(0, kfirst - pkb);
          float s0 = (sc[0] + sd[0]) * sl2, s1 = (sc[1] + sd[1]) * sl2,
                s2 = (sc[2] + sd[2]) * sl2, s3 = (sc[3] + sd[3]) * sl2;
          float u0 = (tc[0] + td[0]) * sl2, u1 = (tc[1] + td[1]) * sl2,
                u2 = (tc[2] + td[2]) * sl2, u3 = (tc[3] + td[3]) * sl2;
          if (!(loa == 0 && pkb + 16 <= L - (p.q_len - 1))) {
            const int a0 = min(16, L - dq[0][0] - pka), a1 = min(16, L - dq[0][1] - pka);
            const int b0 = min(16, L - dq[0][0] - pkb), b1 = min(16, L - dq[0][1] - pkb);
            if (gid >= a0 || gid < loa) s0 = -INFINITY;
            if (gid >= a1 || gid < loa) s1 = -INFINITY;
            if (gid + 8 >= a0 || gid + 8 < loa) s2 = -INFINITY;
            if (gid + 8 >= a1 || gid + 8 < loa) s3 = -INFINITY;
            if (gid >= b0 || gid < lob) u0 = -INFINITY;
            if (gid >= b1 || gid < lob) u1 = -INFINITY;
            if (gid + 8 >= b0 || gid + 8 < lob) u2 = -INFINITY;
            if (gid + 8 >= b1 || gid + 8 < lob) u3 = -INFINITY;
          }
          const float x0 = fmaxf(fmaxf(s0, s2), fmaxf(u0, u2));
          const float x1 = fmaxf(fmaxf(s1, s3), fmaxf(u1, u3));
          if (__any_sync(0xffffffffu, x0 > m_run[0][0] + kLazyLog2 || x1 > m_run[0][1] + kLazyLog2)) {
            float mx0 = x0, mx1 = x1;
#pragma unroll
            for (int o = 4; o < 32; o <<= 1) {
              mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
              mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
            }
            const float mn0 = fmaxf(m_run[0][0], mx0), mn1 = fmaxf(m_run[0][1], mx1);
            const float rf0 = mn0 == -INFINITY ? 0.f : mn0, rf1 = mn1 == -INFINITY ? 0.f : mn1;
            const float al0 = ex2(m_run[0][0] - rf0), al1 = ex2(m_run[0][1] - rf1);
            m_run[0][0] = mn0;
            m_run[0][1] = mn1;
            l_run[0][0] *= al0;
            l_run[0][1] *= al1;
#pragma unroll
            for (int dc = 0; dc < C::kNkc; ++dc) {
              acc[dc][0][0] *= al0;
              acc[dc][0][1] *= al1;
              acc[dc][0][2] *= al0;
              acc[dc][0][3] *= al1;
            }
          }
          const float rf0 = m_run[0][0] == -INFINITY ? 0.f : m_run[0][0];
          const float rf1 = m_run[0][1] == -INFINITY ? 0.f : m_run[0][1];
          const float p0 = ex2(s0 - rf0), p1 = ex2(s1 - rf1), p2 = ex2(s2 - rf0), p3 = ex2(s3 - rf1);
          const float q0 = ex2(u0 - rf0), q1 = ex2(u1 - rf1), q2 = ex2(u2 - rf0), q3 = ex2(u3 - rf1);
          l_run[0][0] += (p0 + p2) + (q0 + q2);
          l_run[0][1] += (p1 + p3) + (q1 + q3);
          const uint32_t pa0 = movmatrix_t(pack_bf16(p0, p1)), pa1 = movmatrix_t(pack_bf16(p2, p3));
          const uint32_t pb0 = movmatrix_t(pack_bf16(q0, q1)), pb1 = movmatrix_t(pack_bf16(q2, q3));
          const uint32_t stVa = stKa + C::kPageBytes, stVb = stKb + C::kPageBytes;
          // (page b's rows past the context may hold NaN: zeroed)
          const uint32_t m01 = nvb >= 16 ? 0xffffffffu
                                         : (2 * tig < nvb ? 0x0000ffffu : 0u) |
                                               (2 * tig + 1 < nvb ? 0xffff0000u : 0u);
          const uint32_t m89 = nvb >= 16 ? 0xffffffffu
                                         : (2 * tig + 8 < nvb ? 0x0000ffffu : 0u) |
                                               (2 * tig + 9 < nvb ? 0xffff0000u : 0u);
#pragma unroll
          for (int dc = 0; dc < C::kNkc; ++dc) {
            uint32_t v0, v1, v2, v3, w0, w1, w2, w3;
            ldsm_x4_t(stVa + (dc >> 2) * 2048 + offV[dc & 3], v0, v1, v2, v3);
            ldsm_x4_t(stVb + (dc >> 2) * 2048 + offV[dc & 3], w0, w1, w2, w3);
            mma_bf16(acc[dc][0], v0, v1, v2, v3, pa0, pa1);
            mma_bf16(acc[dc][0], w0 & m01, w1 & m01, w2 & m89, w3 & m89, pb0, pb1);
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(&empty[sa]);
            mbar_arrive(&empty[sb]);
          }
          ++j;  // (and the loop's own step)
          continue;
        }
      }
      const int i = i_base + j;
      const int li = i / kNW;
      const int s = kRS ? i % S : warp * SPW + li % SPW;
      if (!mbar_wait(&full[s], kRS ? (i / S) & 1 : (li / SPW) & 1, p.wait_ns)) {
        alive = false;
        record_status(p.dev_status, PGQA_ETIMEOUT);
        break;
      }
      bad |= meta[s];
      if (j == app_j) {
        // the new token's row: into the cache and over row (L-1) % 16 of this page
        if (lane < 2 * kAppLanes) {
          const bool isv = lane >= kAppLanes;
          const int c = lane % kAppLanes, rr = (L - 1) & 15;
          uint4 v = app_x0;
          if constexpr (kFp8) {
            const float sc = __ldg((isv ? p.v_scale : p.k_scale) + w.h);
            const uint2 a = e4m3_quant8(app_x0, sc), b = e4m3_quant8(app_x1, sc);
            v = make_uint4(a.x, a.y, b.x, b.y);
          }
          uint8_t* srow = ring + s * C::kStageBytes + (isv ? C::kPageBytes : 0) + (c >> 3) * 2048;
          *reinterpret_cast<uint4*>(
              srow + (C::kPack ? swz128(rr >> 1, (rr & 1) * 4 + c) : swz128(rr, c & 7))) = v;
          if (app_pbn >= 0 && app_pbn < p.num_blocks) {
            const size_t row = (static_cast<size_t>(app_pbn) * Hkv + w.h) * p.block_size +
                               (L - 1) % p.block_size;
            *reinterpret_cast<uint4*>((isv ? ap.v_cache : ap.k_cache) + row * C::kRowBytes +
                                      c * 16) = v;
          }
          fence_proxy_async_smem();  // a later TMA fill of this stage comes after it
        }
        __syncwarp();
      }
      const uint32_t stK = smem_u32(ring + s * C::kStageBytes);
      const uint32_t stV = stK + C::kPageBytes;
      const int pk0 = (w.fp + seg0 + j) * 16;       // key of the page's first row
      const int nv = min(16, L - pk0);               // rows below nv hold keys < L
      const int lo = max(0, kfirst - pk0);           // rows below lo are outside the window
      // every column attends every key of the page (all pages but a unit's last ones
      // and a window's first): no masks
      const bool whole = lo == 0 && pk0 + 16 <= L - (p.q_len - 1);

      // ---- S^T = K Q^T per row tile, over two accumulators (even / odd 16-wide chunks
      //      of head_dim) so the MMA chain is half as long; each K fragment is loaded
      //      (and, E4M3, widened) once for all row tiles
      float sc[NT][4], sd[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt)
#pragma unroll
        for (int q = 0; q < 4; ++q) sc[nt][q] = sd[nt][q] = 0.f;
      if constexpr (!kFp8) {
#pragma unroll
        for (int kc = 0; kc < C::kNkc; ++kc) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(stK + (kc >> 2) * 2048 + offK[kc & 3], a0, a1, a2, a3);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt)
            mma_bf16((kc & 1) ? sd[nt] : sc[nt], a0, a1, a2, a3, qf[kc][nt][0], qf[kc][nt][1]);
        }
      } else {
#pragma unroll
        for (int kc = 0; kc < C::kNkc; kc += 2) {
          uint32_t r0v, r1v, r2v, r3v;
          ldsm_x4(stK + offK[kc >> 1], r0v, r1v, r2v, r3v);
          const uint32_t a0 = e4m3x2_to_f16x2(r0v & 0xffff), a1 = e4m3x2_to_f16x2(r1v & 0xffff),
                         a2 = e4m3x2_to_f16x2(r0v >> 16), a3 = e4m3x2_to_f16x2(r1v >> 16);
          const uint32_t b0 = e4m3x2_to_f16x2(r2v & 0xffff), b1 = e4m3x2_to_f16x2(r3v & 0xffff),
                         b2 = e4m3x2_to_f16x2(r2v >> 16), b3 = e4m3x2_to_f16x2(r3v >> 16);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) {
            mma_f16(sc[nt], a0, a1, a2, a3, qf[kc][nt][0], qf[kc][nt][1]);
            mma_f16(sd[nt], b0, b1, b2, b3, qf[kc + 1][nt][0], qf[kc + 1][nt][1]);
          }
        }
      }
      // ---- per row tile: masks, the online softmax, P^T as the B operand
      //      fragment: sc[0] (tok gid, row 2tig), sc[1] (gid, 2tig+1),
      //                sc[2] (gid+8, 2tig),    sc[3] (gid+8, 2tig+1)
      uint32_t pb0[NT], pb1[NT];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int q = 0; q < 4; ++q) sc[nt][q] += sd[nt][q];
        float s0 = sc[nt][0] * sl2, s1 = sc[nt][1] * sl2, s2 = sc[nt][2] * sl2,
              s3 = sc[nt][3] * sl2;
        if (!whole) {
          // rows below nv0 / nv1 hold keys the column attends (multi-token: token t of
          // q_len sees keys up to L - q_len + t)
          const int nv0 = min(16, L - dq[nt][0] - pk0), nv1 = min(16, L - dq[nt][1] - pk0);
          if (gid >= nv0 || gid < lo) s0 = -INFINITY;
          if (gid >= nv1 || gid < lo) s1 = -INFINITY;
          if (gid + 8 >= nv0 || gid + 8 < lo) s2 = -INFINITY;
          if (gid + 8 >= nv1 || gid + 8 < lo) s3 = -INFINITY;
        }
        // m_run is the column's reference: every score seen so far is at most
        // m_run + kLazyLog2. Only a score above that (the first page with a key, or a
        // jump in the maximum) moves it, to the maximum so far, and rescales l and O;
        // otherwise P = 2^(s - m_run) <= 2^kLazyLog2 as is. Exact either way: l and O
        // share the reference, and lse = m_run + log2 l.
        const bool grow = fmaxf(s0, s2) > m_run[nt][0] + kLazyLog2 ||
                          fmaxf(s1, s3) > m_run[nt][1] + kLazyLog2;
        if (__any_sync(0xffffffffu, grow)) {
          float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
          for (int o = 4; o < 32; o <<= 1) {
            mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
            mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
          }
          const float mn0 = fmaxf(m_run[nt][0], mx0), mn1 = fmaxf(m_run[nt][1], mx1);
          // a column that has seen no key yet (a page past a draft token's last key)
          // keeps m = -inf; 0 as the reference then gives 2^-inf = 0 instead of NaN
          const float rf0 = mn0 == -INFINITY ? 0.f : mn0, rf1 = mn1 == -INFINITY ? 0.f : mn1;
          const float al0 = ex2(m_run[nt][0] - rf0), al1 = ex2(m_run[nt][1] - rf1);
          m_run[nt][0] = mn0;
          m_run[nt][1] = mn1;
          l_run[nt][0] *= al0;
          l_run[nt][1] *= al1;
#pragma unroll
          for (int dc = 0; dc < C::kNkc; ++dc) {
            acc[dc][nt][0] *= al0;
            acc[dc][nt][1] *= al1;
            acc[dc][nt][2] *= al0;
            acc[dc][nt][3] *= al1;
          }
        }
        const float rf0 = m_run[nt][0] == -INFINITY ? 0.f : m_run[nt][0];
        const float rf1 = m_run[nt][1] == -INFINITY ? 0.f : m_run[nt][1];
        const float p0v = ex2(s0 - rf0), p1v = ex2(s1 - rf1), p2v = ex2(s2 - rf0),
                    p3v = ex2(s3 - rf1);
        l_run[nt][0] += p0v + p2v;
        l_run[nt][1] += p1v + p3v;
        pb0[nt] = movmatrix_t(kFp8 ? pack_f16(p0v, p1v) : pack_bf16(p0v, p1v));
        pb1[nt] = movmatrix_t(kFp8 ? pack_f16(p2v, p3v) : pack_bf16(p2v, p3v));
      }

      // ---- O^T += V^T P^T; rows past the context are zeroed (they may hold NaN)
      // (rows below lo hold real keys and get P = 0; only rows past the context,
      // which may hold NaN, need zeroing)
      if constexpr (!kFp8) {
        if (nv < 16) {  // the context's last page
          const uint32_t m01 =
              (2 * tig < nv ? 0x0000ffffu : 0u) | (2 * tig + 1 < nv ? 0xffff0000u : 0u);
          const uint32_t m89 =
              (2 * tig + 8 < nv ? 0x0000ffffu : 0u) | (2 * tig + 9 < nv ? 0xffff0000u : 0u);
#pragma unroll
          for (int dc = 0; dc < C::kNkc; ++dc) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(stV + (dc >> 2) * 2048 + offV[dc & 3], v0, v1, v2, v3);
            v0 &= m01;
            v1 &= m01;
            v2 &= m89;
            v3 &= m89;
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_bf16(acc[dc][nt], v0, v1, v2, v3, pb0[nt], pb1[nt]);
          }
        } else {
#pragma unroll
          for (int dc = 0; dc < C::kNkc; ++dc) {
            uint32_t v0, v1, v2, v3;
            ldsm_x4_t(stV + (dc >> 2) * 2048 + offV[dc & 3], v0, v1, v2, v3);
#pragma unroll
            for (int nt = 0; nt < NT; ++nt)
              mma_bf16(acc[dc][nt], v0, v1, v2, v3, pb0[nt], pb1[nt]);
          }
        }
      } else {
        // thread rows d in [(D/8) gid, (D/8) (gid + 1)): row r of chunk dc <-> d =
        // (D/8) (r & 7) + 2 dc + (r >> 3); (D/8) bytes of each of the thread's 4 keys
        uint4 R0, R1, R2, R3;
        if constexpr (C::kPack) {  // 8 bytes: rows 2 tig .. (two tokens per shared row)
          const uint2 a = lds64(stV + offV[0]);
          const uint2 b = lds64(stV + offV[1]);
          const uint2 c = lds64(stV + offV[2]);
          const uint2 d = lds64(stV + offV[3]);
          R0 = make_uint4(a.x, a.y, 0, 0);
          R1 = make_uint4(b.x, b.y, 0, 0);
          R2 = make_uint4(c.x, c.y, 0, 0);
          R3 = make_uint4(d.x, d.y, 0, 0);
        } else {
          R0 = lds128(stV + offV[0]);
          R1 = lds128(stV + offV[1]);
          R2 = lds128(stV + offV[2]);
          R3 = lds128(stV + offV[3]);
        }
        if (nv < 16) {
          if (2 * tig >= nv) R0 = make_uint4(0, 0, 0, 0);
          if (2 * tig + 1 >= nv) R1 = make_uint4(0, 0, 0, 0);
          if (2 * tig + 8 >= nv) R2 = make_uint4(0, 0, 0, 0);
          if (2 * tig + 9 >= nv) R3 = make_uint4(0, 0, 0, 0);
        }
        const uint32_t w0[4] = {R0.x, R0.y, R0.z, R0.w}, w1[4] = {R1.x, R1.y, R1.z, R1.w};
        const uint32_t w8[4] = {R2.x, R2.y, R2.z, R2.w}, w9[4] = {R3.x, R3.y, R3.z, R3.w};
#pragma unroll
        for (int dc = 0; dc < C::kNkc; ++dc) {
          const uint32_t sel = (dc & 1) ? 0x7362u : 0x5140u;
          const uint32_t lo = prmt(w0[dc >> 1], w1[dc >> 1], sel);
          const uint32_t hi = prmt(w8[dc >> 1], w9[dc >> 1], sel);
          const uint32_t v0 = e4m3x2_to_f16x2(lo & 0xffff), v1 = e4m3x2_to_f16x2(lo >> 16),
                         v2 = e4m3x2_to_f16x2(hi & 0xffff), v3 = e4m3x2_to_f16x2(hi >> 16);
#pragma unroll
          for (int nt = 0; nt < NT; ++nt) mma_f16(acc[dc][nt], v0, v1, v2, v3, pb0[nt], pb1[nt]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    i_base += npg;

    // ---- this warp's state for the unit -> the merge buffer of the unit's parity;
    //      the merge warp takes it from there and this warp goes on to the next unit
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        l_run[nt][0] += __shfl_xor_sync(0xffffffffu, l_run[nt][0], o);
        l_run[nt][1] += __shfl_xor_sync(0xffffffffu, l_run[nt][1], o);
      }
    }
    const bool poisoned_w = __any_sync(0xffffffffu, bad != 0) || !__all_sync(0xffffffffu, alive);
    constexpr int kBufs = C::kMergeBufs;
    const int mb = cu % kBufs;
    if (cu >= kBufs &&
        !__all_sync(0xffffffffu, mbar_wait(&merge_free[mb], ((cu / kBufs) - 1) & 1, p.wait_ns))) {
      alive = false;
      if (lane == 0) record_status(p.dev_status, PGQA_ETIMEOUT);
    }
    float* wob = wo + mb * C::kMergeFloats;
    float* wmlb = wml + mb * C::kMlFloats;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      // state rows of this thread's columns: per warp, or (row-split) the rows themselves
      const int srow = (kRS ? rbase : warp * kRows + 8 * nt) + 2 * tig;
#pragma unroll
      for (int dc = 0; dc < C::kNkc; ++dc) {
        int d0, d1;
        if constexpr (!kFp8) {
          d0 = 16 * dc + gid;
          d1 = d0 + 8;
        } else {
          d0 = (D / 8) * gid + 2 * dc;
          d1 = d0 + 1;
        }
        float* o0 = wob + srow * C::kLd;
        float* o1 = o0 + C::kLd;
        o0[d0] = acc[dc][nt][0];
        o1[d0] = acc[dc][nt][1];
        o0[d1] = acc[dc][nt][2];
        o1[d1] = acc[dc][nt][3];
      }
      if (gid == 0) {
        float* ml = wmlb + srow * 2;
        ml[0] = m_run[nt][0];
        ml[1] = poisoned_w ? NAN : l_run[nt][0];  // NaN l marks a poisoned warp state
        ml[2] = m_run[nt][1];
        ml[3] = poisoned_w ? NAN : l_run[nt][1];
      }
    }
    __syncwarp();
    cur = nxt;
    if (more) {  // the merge warp takes the unit
      if (lane == 0) mbar_arrive(&unit_done[mb]);
      ++cu;
      continue;
    }
    // the range's last unit: nothing left to stream, so the consumer warps (those with
    // rows, in the row-split form) finish it
    const int nseg = unit_segments(w, chunk);
    const int nthr = (kRS ? kRT : kNW) * 32;
    int* const ticket = p.counters + w.b * Hkv + w.h;
    // When every other CTA of a cut unit has already arrived (as the run order makes
    // likely: they took their parts first), this CTA is the last one: it merges their
    // partials with its own state straight into the output and resets the ticket, with
    // no partial of its own, no ticket update and no reading back (the same arithmetic
    // as the ticket path below, so the same result bit for bit)
    if (tid == 0)
      misc[1] = nseg > 1 && (peek == static_cast<unsigned>(nseg - 1) ||
                             ticket_peek(ticket) == static_cast<unsigned>(nseg - 1));
    bar_consumers(nthr);
    if (misc[1]) {
      merge_partials<D, kFp8, NT, kRS>(epi, w.b, w.h, w.S, w.P, chunk, tid, nthr, 0, 1 << 30,
                                       wob, wmlb);
      if (tid == 0) *reinterpret_cast<volatile int*>(ticket) = 0;
    } else {
      combine_unit<D, kFp8, NT, kRS>(epi, w.b, w.h, nseg, w.S <= r0 ? 0 : 1, wob, wmlb, tid,
                                     nthr);
      if (nseg > 1) {
        bar_consumers(nthr);  // this CTA's partial writes are issued
        if (tid == 0) misc[1] = ticket_last(ticket, nseg);
        bar_consumers(nthr);  // (and the reads below come after the acquire)
        if (misc[1])
          merge_partials<D, kFp8, NT, kRS>(epi, w.b, w.h, w.S, w.P, chunk, tid, nthr);
      }
    }
    ++cu;
  }
}

template <int D, bool kFp8, int NT, bool kRS = false>
pgqa_status_t launch_variant(const DecodeArgs& a, const DecodePlan& plan) {
  using C = Cfg<D, kFp8, NT, kRS>;
  const CUtensorMapDataType dt =
      kFp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * a.block_size;
  const uint32_t box_rows = a.block_size == 8 ? 8 : 16;
  // 64-byte rows: the cache viewed as 128-byte rows of two tokens each
  const int pk = C::kPack ? 2 : 1;
  CUtensorMap kmap, vmap;
  if (!tensor_map_2d(&kmap, a.k_cache, dt, D * pk, rows / pk, C::kRowBytes * pk, 128 / C::kElem,
                     box_rows / pk, CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tensor_map_2d(&vmap, a.v_cache, dt, D * pk, rows / pk, C::kRowBytes * pk, 128 / C::kElem,
                     box_rows / pk, CU_TENSOR_MAP_SWIZZLE_128B))
    return PGQA_ECUDA;
  if (!smem_attr_ready(reinterpret_cast<const void*>(paged_decode_kernel<D, kFp8, NT, kRS>),
                       C::kSmem))
    return PGQA_ECUDA;
  DecodeParams p;
  p.out = static_cast<__nv_bfloat16*>(a.out);
  p.lse = a.lse;
  p.q = static_cast<const __nv_bfloat16*>(a.q);
  p.block_tables = a.block_tables;
  p.context_lens = a.context_lens;
  p.k_scale = a.k_scale;
  p.v_scale = a.v_scale;
  uint8_t* ws = static_cast<uint8_t*>(a.workspace);
  p.counters = reinterpret_cast<int*>(ws + plan.counters_off);
  p.part_lse = reinterpret_cast<float*>(ws + plan.lse_off);
  p.part_o = reinterpret_cast<float*>(ws + plan.o_off);
  p.dev_status = a.dev_status;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_seqs = a.num_seqs;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.q_len = a.q_len;
  p.num_blocks = a.num_blocks;
  p.max_context_len = a.max_context_len;
  p.window = a.window;
  p.block_size = a.block_size;
  p.scale_log2 = a.scale * kLog2e;
  p.wait_ns = decode_wait_limit_ns();
  DecodeAppend ap;
  ap.key = static_cast<const uint4*>(a.new_key);
  ap.value = static_cast<const uint4*>(a.new_value);
  ap.k_cache = static_cast<uint8_t*>(const_cast<void*>(a.k_cache));
  ap.v_cache = static_cast<uint8_t*>(const_cast<void*>(a.v_cache));
  if (launch_after_previous(paged_decode_kernel<D, kFp8, NT, kRS>, dim3(plan.grid),
                            dim3(kThreads),
                            C::kSmem, a.stream, kmap, vmap, p, ap) != cudaSuccess)
    return PGQA_ECUDA;
  return cudaPeekAtLastError() == cudaSuccess ? PGQA_OK : PGQA_ECUDA;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

namespace {
std::atomic<unsigned long long> g_decode_wait_ns{0};  // 0: kWaitLimitNs
}  // namespace

unsigned long long decode_wait_limit_ns() {
  const unsigned long long v = g_decode_wait_ns.load(std::memory_order_relaxed);
  return v ? v : kWaitLimitNs;
}

void set_decode_wait_limit_ns(unsigned long long ns) {
  g_decode_wait_ns.store(ns, std::memory_order_relaxed);
}

int decode_row_tiles(int q_len, int group) {
  const int rows = q_len * group;
  return rows <= 8 ? 1 : rows <= 8 * kNW ? kNW : 0;
}

int decode_ctas_per_sm(int head_dim, int cache_dtype, int row_tiles) {
  const bool e4m3 = cache_dtype == PGQA_DTYPE_E4M3, d64 = head_dim == 64;
  if (row_tiles == kNW) {  // row-split
    if (e4m3) return d64 ? ctas_per_sm<64, true, 1, true>() : ctas_per_sm<128, true, 1, true>();
    return d64 ? ctas_per_sm<64, false, 1, true>() : ctas_per_sm<128, false, 1, true>();
  }
  if (e4m3) return d64 ? ctas_per_sm<64, true>() : ctas_per_sm<128, true>();
  return d64 ? ctas_per_sm<64, false>() : ctas_per_sm<128, false>();
}

DecodePlan decode_plan(int num_seqs, int num_kv_heads, int head_dim, int cache_dtype,
                       int num_sms, int row_tiles) {
  DecodePlan plan{};
  plan.row_tiles = row_tiles;
  plan.grid = (num_sms > 0 ? num_sms : 1) * decode_ctas_per_sm(head_dim, cache_dtype, row_tiles);
  const size_t units = static_cast<size_t>(num_seqs > 0 ? num_seqs : 0) *
                       static_cast<size_t>(num_kv_heads > 0 ? num_kv_heads : 0);
  const size_t slots = static_cast<size_t>(plan.grid) * 2 * 8 * row_tiles;
  const size_t tickets = units;  // one per unit
  plan.counters_off = 0;
  plan.lse_off = align256(tickets * sizeof(int));
  plan.o_off = plan.lse_off + align256(slots * sizeof(float));
  plan.bytes = plan.o_off + align256(slots * static_cast<size_t>(head_dim) * sizeof(float));
  return plan;
}

bool decode_prepare() {
  return smem_attr_ready(reinterpret_cast<const void*>(paged_decode_kernel<128, false, 1, false>),
                         Cfg<128, false>::kSmem) &&
         smem_attr_ready(reinterpret_cast<const void*>(paged_decode_kernel<64, false, 1, false>),
                         Cfg<64, false>::kSmem) &&
         smem_attr_ready(reinterpret_cast<const void*>(paged_decode_kernel<128, true, 1, false>),
                         Cfg<128, true>::kSmem) &&
         smem_attr_ready(reinterpret_cast<const void*>(paged_decode_kernel<64, true, 1, false>),
                         Cfg<64, true>::kSmem);
}

pgqa_status_t launch_paged_decode(const DecodeArgs& a, const DecodePlan& plan) {
  if (plan.row_tiles == 1) {
    if (a.cache_dtype == PGQA_DTYPE_BF16) {
      if (a.head_dim == 128) return launch_variant<128, false, 1>(a, plan);
      if (a.head_dim == 64) return launch_variant<64, false, 1>(a, plan);
    } else if (a.cache_dtype == PGQA_DTYPE_E4M3) {
      if (a.head_dim == 128) return launch_variant<128, true, 1>(a, plan);
      if (a.head_dim == 64) return launch_variant<64, true, 1>(a, plan);
    }
  } else if (plan.row_tiles == kNW) {
    if (a.cache_dtype == PGQA_DTYPE_BF16) {
      if (a.head_dim == 128) return launch_variant<128, false, 1, true>(a, plan);
      if (a.head_dim == 64) return launch_variant<64, false, 1, true>(a, plan);
    } else if (a.cache_dtype == PGQA_DTYPE_E4M3) {
      if (a.head_dim == 128) return launch_variant<128, true, 1, true>(a, plan);
      if (a.head_dim == 64) return launch_variant<64, true, 1, true>(a, plan);
    }
  }
  return PGQA_EUNSUPPORTED;
}

}  // namespace pgqa
