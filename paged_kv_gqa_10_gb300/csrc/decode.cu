// Paged decode attention for sm_103a.
//
// Computes, for every sequence b and query head hq, softmax(scale * q K^T) V over
// the b's cached tokens read through its block table ("LLaMA structure and
// inference performance" (wmrh.cn) sec. 3.1 steps 3-6, with repeat_kv of sec.
// 2.1 as the index map kv_head = hq / G; pages addressed as in the rkmt.cn
// article, sec. 3.1), plus lse = ln sum exp(score).
//
// Work decomposition (bandwidth-bound: every KV byte must be read exactly once)
//  - One CTA per (split, kv-head, sequence). It serves all G = Hq/Hkv query
//    heads of its kv-head, so a K/V page is fetched once for the whole group.
//  - Long contexts are cut into splits of `pages_per_split` 16-token pages so
//    that the grid fills the 152 SMs; split results are merged with their LSEs
//    by whichever CTA of the (sequence, kv-head) finishes last (an atomic ticket,
//    no CTA ever waits for another).
//  - Warp roles: one producer warp streams pages with TMA (2-D tensor map over
//    the cache viewed as [num_blocks*Hkv*16 rows][head_dim], 128-byte swizzle)
//    into mbarrier-guarded stages; NW consumer warps take pages round-robin,
//    each keeping its own online-softmax state, merged at the end. Every consumer
//    warp owns its own sub-ring of stages, so consecutive uses of a stage belong
//    to one warp and a parity wait can never be two phases behind.
//  - Math per 16-token page on the warp-level tensor path (mma.m16n8k16):
//      S^T[16 tok x 8 heads] = K[16 x D] . Q^T[D x 8]   (tokens fill M = 16)
//      online softmax on the S^T fragment (column = query head)
//      P^T fragment -> B operand with movmatrix (an 8x8 transpose in registers)
//      O^T[D x 8] += V^T[D x 16] . P^T[16 x 8]            (V^T via ldmatrix.trans)
//    G <= 8 heads sit in N = 8; padded heads have q = 0 and are never stored.
//  - FP8 E4M3 cache: codes are widened to f16 in registers (exact) and fed to the
//    f16 MMA; k_scale folds into the score scale, v_scale into the final output.
//    The head-dimension order inside an MMA is a free permutation (it is the
//    contraction index for QK^T and a row relabelling for PV), chosen so that each
//    thread's bytes are contiguous in shared memory.
#include <cuda_bf16.h>
#include <float.h>

#include "host.h"
#include "ptx.cuh"

namespace pgqa {
namespace {

constexpr int kNW = 4;              // consumer warps per CTA
constexpr int kThreads = (kNW + 1) * 32;
constexpr int kMinPagesPerSplit = 8;  // never split below 128 tokens
constexpr int kCtasPerSmTarget = 8;   // aim for this many (split) CTAs per SM
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
  int* counters;
  float* ws_lse;
  float* ws_o;
  int* dev_status;
  int max_blocks_per_seq;
  int num_q_heads, num_kv_heads, group;
  int num_blocks;
  int max_context_len;
  int pages_per_split, num_splits;
  float scale_log2;  // scale * log2(e)
};

template <int D, bool kFp8>
struct Cfg {
  static constexpr int kElem = kFp8 ? 1 : 2;
  static constexpr int kRowBytes = D * kElem;      // one token row of one head
  static constexpr int kSub = kRowBytes / 128;     // 128-byte TMA boxes per row
  static constexpr int kPageBytes = 16 * kRowBytes;
  static constexpr int kStageBytes = 2 * kPageBytes;  // K page + V page
  static constexpr int kStagesPerWarp = kFp8 ? 3 : 2;  // each consumer warp owns a sub-ring
  static constexpr int kStages = kNW * kStagesPerWarp;
  static constexpr int kRingBytes = kStages * kStageBytes;
  static constexpr int kNkc = D / 16;              // 16-wide chunks of head_dim
  static constexpr int kMergeBytes = kNW * 8 * D * 4;
  static constexpr int kSmem = 1024 + kRingBytes + 2 * kStages * 8 + 16 + kNW * 8 * 2 * 4;
  static_assert(kRowBytes % 128 == 0, "rows must be whole 128-byte swizzle rows");
  static_assert(kMergeBytes <= kRingBytes, "merge buffers reuse the ring");
};

template <int D>
__device__ __forceinline__ void zero_outputs(const DecodeParams& p, int b, int h) {
  const int G = p.group;
  for (int i = threadIdx.x; i < G * D / 8; i += blockDim.x) {
    const int g = i / (D / 8), c = i % (D / 8);
    const size_t row = static_cast<size_t>(b) * p.num_q_heads + h * G + g;
    reinterpret_cast<uint4*>(p.out + row * D)[c] = make_uint4(0, 0, 0, 0);
    if (c == 0 && p.lse) p.lse[row] = -INFINITY;
  }
}

template <int D, bool kFp8>
__global__ void __launch_bounds__(kThreads) paged_decode_kernel(
    const __grid_constant__ CUtensorMap kmap, const __grid_constant__ CUtensorMap vmap,
    const DecodeParams p) {
  using C = Cfg<D, kFp8>;
  constexpr int S = C::kStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + C::kRingBytes);
  uint64_t* empty = full + S;
  int* flags = reinterpret_cast<int*>(empty + S);  // [0] bad block id, [1] timeout, [2] last
  float* wml = reinterpret_cast<float*>(flags + 4);  // [kNW][8][2] per-warp (m, l), base 2
  float* wo = reinterpret_cast<float*>(ring);        // [kNW][8][D] per-warp O, after the loop

  const int split = blockIdx.x, h = blockIdx.y, b = blockIdx.z;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = p.group;
  const int L = __ldg(p.context_lens + b);
  const int npages_all = (L + 15) >> 4;
  const bool len_bad = L < 0 || L > p.max_context_len || npages_all > p.max_blocks_per_seq;
  if (len_bad || L == 0) {
    if (split == 0) {
      if (len_bad && tid == 0) record_status(p.dev_status, PGQA_EINVAL);
      zero_outputs<D>(p, b, h);
    }
    return;
  }
  const int pps = p.pages_per_split;
  const int p0 = split * pps;
  if (p0 >= npages_all) return;
  const int np = min(pps, npages_all - p0);
  const int nsplit = (npages_all + pps - 1) / pps;

  if (tid == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    flags[0] = flags[1] = flags[2] = 0;
    fence_mbar_init();
  }
  __syncthreads();

  // ------------------------------------------------------------ producer
  if (warp == kNW) {
    if (lane == 0) {
      tma_prefetch_desc(&kmap);
      tma_prefetch_desc(&vmap);
    }
    const int32_t* bt = p.block_tables + static_cast<size_t>(b) * p.max_blocks_per_seq + p0;
    int issued = 0;
    bool ok = true;
    for (int base = 0; base < np && ok; base += 32) {
      const int32_t mine = base + lane < np ? __ldg(bt + base + lane) : 0;
      const int n = min(32, np - base);
      for (int k = 0; k < n; ++k) {
        int32_t pbn = __shfl_sync(0xffffffffu, mine, k);
        const int i = base + k;
        if (lane == 0) {
          const int li = i / kNW;  // index among this consumer warp's pages
          const int s = (i % kNW) * C::kStagesPerWarp + li % C::kStagesPerWarp;
          const int use = li / C::kStagesPerWarp;
          if (use > 0 && !mbar_wait(&empty[s], (use - 1) & 1)) {
            record_status(p.dev_status, PGQA_ETIMEOUT);
            flags[1] = 1;
            ok = false;
          } else {
            if (pbn < 0 || pbn >= p.num_blocks) {
              flags[0] = 1;
              pbn = 0;  // load a valid page; the result is discarded
            }
            uint8_t* st = ring + s * C::kStageBytes;
            mbar_arrive_expect_tx(&full[s], C::kStageBytes);
            const int y = (pbn * p.num_kv_heads + h) * 16;
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub)
              tma_load_2d(st + sub * 2048, &kmap, &full[s], sub * (128 / C::kElem), y);
#pragma unroll
            for (int sub = 0; sub < C::kSub; ++sub)
              tma_load_2d(st + C::kPageBytes + sub * 2048, &vmap, &full[s],
                          sub * (128 / C::kElem), y);
            ++issued;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
      }
    }
    // No TMA write may land after this CTA moves on: wait for the last phase of
    // every stage used (already complete on the normal path).
    if (lane == 0) {
      for (int w = 0; w < kNW; ++w) {
        const int n_w = issued > w ? (issued - w + kNW - 1) / kNW : 0;  // pages issued to w
        for (int k = 0; k < C::kStagesPerWarp && k < n_w; ++k) {
          const int last_li = k + ((n_w - 1 - k) / C::kStagesPerWarp) * C::kStagesPerWarp;
          if (!mbar_wait(&full[w * C::kStagesPerWarp + k], (last_li / C::kStagesPerWarp) & 1))
            record_status(p.dev_status, PGQA_ETIMEOUT);
        }
      }
    }
  }

  // ------------------------------------------------------------ consumers
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  float acc[C::kNkc][4];
#pragma unroll
  for (int i = 0; i < C::kNkc; ++i) acc[i][0] = acc[i][1] = acc[i][2] = acc[i][3] = 0.f;
  const int gid = lane >> 2, tig = lane & 3;

  if (warp < kNW) {
    // Q^T as the B operand: column n = query head gid of the group.
    uint32_t qf[C::kNkc][2];
    {
      const bool live = gid < G;
      const __nv_bfloat16* qrow =
          p.q + (static_cast<size_t>(b) * p.num_q_heads + h * G + (live ? gid : 0)) * D;
#pragma unroll
      for (int kc = 0; kc < C::kNkc; ++kc) {
        if constexpr (!kFp8) {
          const uint32_t* q32 = reinterpret_cast<const uint32_t*>(qrow + 16 * kc + 2 * tig);
          qf[kc][0] = live ? __ldg(q32) : 0u;
          qf[kc][1] = live ? __ldg(q32 + 4) : 0u;
        } else {
          // k index 2tig+{0,1} <-> d = 16kc + 4tig + {0,1}; 2tig+8+{0,1} <-> +{2,3}
          const uint2 q4 = live ? __ldg(reinterpret_cast<const uint2*>(qrow + 16 * kc + 4 * tig))
                                : make_uint2(0, 0);
          qf[kc][0] = pack_f16(bf16_lo(q4.x), bf16_hi(q4.x));
          qf[kc][1] = pack_f16(bf16_lo(q4.y), bf16_hi(q4.y));
        }
      }
    }
    const float sl2 = p.scale_log2 * (kFp8 ? __ldg(p.k_scale + h) : 1.f);
    // lane-invariant parts of the ldmatrix addresses
    const uint32_t rowK = (lane & 7) + (((lane >> 3) & 1) << 3);
    const uint32_t cK = lane >> 4;
    const uint32_t rowV = (lane & 7) + ((lane >> 4) << 3);
    const uint32_t cV = (lane >> 3) & 1;

    for (int i = warp; i < np; i += kNW) {
      const int li = i / kNW;
      const int s = warp * C::kStagesPerWarp + li % C::kStagesPerWarp;
      if (!mbar_wait(&full[s], (li / C::kStagesPerWarp) & 1)) {
        record_status(p.dev_status, PGQA_ETIMEOUT);
        flags[1] = 1;
        break;
      }
      const uint32_t stK = smem_u32(ring + s * C::kStageBytes);
      const uint32_t stV = stK + C::kPageBytes;
      const int nv = min(16, L - (p0 + i) * 16);  // valid tokens in this page

      // ---- S^T = K Q^T
      float sc[4] = {0.f, 0.f, 0.f, 0.f};
      if constexpr (!kFp8) {
#pragma unroll
        for (int kc = 0; kc < C::kNkc; ++kc) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(stK + (kc >> 2) * 2048 + swz128(rowK, (kc & 3) * 2 + cK), a0, a1, a2, a3);
          mma_bf16(sc, a0, a1, a2, a3, qf[kc][0], qf[kc][1]);
        }
      } else {
#pragma unroll
        for (int kc = 0; kc < C::kNkc; kc += 2) {
          uint32_t r0, r1, r2, r3;
          ldsm_x4(stK + swz128(rowK, kc + cK), r0, r1, r2, r3);
          mma_f16(sc, e4m3x2_to_f16x2(r0 & 0xffff), e4m3x2_to_f16x2(r1 & 0xffff),
                  e4m3x2_to_f16x2(r0 >> 16), e4m3x2_to_f16x2(r1 >> 16), qf[kc][0], qf[kc][1]);
          mma_f16(sc, e4m3x2_to_f16x2(r2 & 0xffff), e4m3x2_to_f16x2(r3 & 0xffff),
                  e4m3x2_to_f16x2(r2 >> 16), e4m3x2_to_f16x2(r3 >> 16), qf[kc + 1][0],
                  qf[kc + 1][1]);
        }
      }
      // fragment: sc[0] (tok gid, head 2tig), sc[1] (gid, 2tig+1),
      //           sc[2] (gid+8, 2tig),      sc[3] (gid+8, 2tig+1)
      float s0 = sc[0] * sl2, s1 = sc[1] * sl2, s2 = sc[2] * sl2, s3 = sc[3] * sl2;
      if (gid >= nv) s0 = s1 = -INFINITY;
      if (gid + 8 >= nv) s2 = s3 = -INFINITY;
      float mx0 = fmaxf(s0, s2), mx1 = fmaxf(s1, s3);
#pragma unroll
      for (int o = 4; o < 32; o <<= 1) {
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, o));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, o));
      }
      const float mn0 = fmaxf(m_run[0], mx0), mn1 = fmaxf(m_run[1], mx1);
      const float al0 = ex2(m_run[0] - mn0), al1 = ex2(m_run[1] - mn1);
      m_run[0] = mn0;
      m_run[1] = mn1;
      const float p0v = ex2(s0 - mn0), p1v = ex2(s1 - mn1), p2v = ex2(s2 - mn0),
                  p3v = ex2(s3 - mn1);
      l_run[0] = l_run[0] * al0 + (p0v + p2v);
      l_run[1] = l_run[1] * al1 + (p1v + p3v);
#pragma unroll
      for (int dc = 0; dc < C::kNkc; ++dc) {
        acc[dc][0] *= al0;
        acc[dc][1] *= al1;
        acc[dc][2] *= al0;
        acc[dc][3] *= al1;
      }
      // ---- P^T as the B operand (k = token, n = head)
      const uint32_t pb0 = movmatrix_t(kFp8 ? pack_f16(p0v, p1v) : pack_bf16(p0v, p1v));
      const uint32_t pb1 = movmatrix_t(kFp8 ? pack_f16(p2v, p3v) : pack_bf16(p2v, p3v));

      // ---- O^T += V^T P^T; rows past the context are zeroed (they may hold NaN)
      const uint32_t m01 = (2 * tig < nv ? 0x0000ffffu : 0u) | (2 * tig + 1 < nv ? 0xffff0000u : 0u);
      const uint32_t m89 =
          (2 * tig + 8 < nv ? 0x0000ffffu : 0u) | (2 * tig + 9 < nv ? 0xffff0000u : 0u);
      if constexpr (!kFp8) {
#pragma unroll
        for (int dc = 0; dc < C::kNkc; ++dc) {
          uint32_t v0, v1, v2, v3;
          ldsm_x4_t(stV + (dc >> 2) * 2048 + swz128(rowV, (dc & 3) * 2 + cV), v0, v1, v2, v3);
          if (nv < 16) {
            v0 &= m01;
            v1 &= m01;
            v2 &= m89;
            v3 &= m89;
          }
          mma_bf16(acc[dc], v0, v1, v2, v3, pb0, pb1);
        }
      } else {
        // thread rows d in [16 gid, 16 gid + 16): row r of chunk dc <-> d = 16 (r & 7) + 2 dc + (r >> 3)
        uint4 R0 = lds128(stV + swz128(2 * tig, gid));
        uint4 R1 = lds128(stV + swz128(2 * tig + 1, gid));
        uint4 R2 = lds128(stV + swz128(2 * tig + 8, gid));
        uint4 R3 = lds128(stV + swz128(2 * tig + 9, gid));
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
          mma_f16(acc[dc], e4m3x2_to_f16x2(lo & 0xffff), e4m3x2_to_f16x2(lo >> 16),
                  e4m3x2_to_f16x2(hi & 0xffff), e4m3x2_to_f16x2(hi >> 16), pb0, pb1);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    // full row sums for this thread's two head columns
#pragma unroll
    for (int o = 4; o < 32; o <<= 1) {
      l_run[0] += __shfl_xor_sync(0xffffffffu, l_run[0], o);
      l_run[1] += __shfl_xor_sync(0xffffffffu, l_run[1], o);
    }
  }
  __syncthreads();  // every page consumed and every TMA landed: the ring is free

  // ---- per-warp state to shared memory
  if (warp < kNW) {
#pragma unroll
    for (int dc = 0; dc < C::kNkc; ++dc) {
      int d0, d1;
      if constexpr (!kFp8) {
        d0 = 16 * dc + gid;
        d1 = d0 + 8;
      } else {
        d0 = 16 * gid + 2 * dc;
        d1 = d0 + 1;
      }
      float* o0 = wo + (warp * 8 + 2 * tig) * D;
      float* o1 = o0 + D;
      o0[d0] = acc[dc][0];
      o1[d0] = acc[dc][1];
      o0[d1] = acc[dc][2];
      o1[d1] = acc[dc][3];
    }
    if (gid == 0) {
      wml[(warp * 8 + 2 * tig) * 2 + 0] = m_run[0];
      wml[(warp * 8 + 2 * tig) * 2 + 1] = l_run[0];
      wml[(warp * 8 + 2 * tig + 1) * 2 + 0] = m_run[1];
      wml[(warp * 8 + 2 * tig + 1) * 2 + 1] = l_run[1];
    }
  }
  __syncthreads();

  const bool bad = flags[0] != 0 || flags[1] != 0;
  if (flags[0] != 0 && tid == 0) record_status(p.dev_status, PGQA_EBADINDEX);
  const int u = b * p.num_kv_heads + h;
  const float vsc = kFp8 ? __ldg(p.v_scale + h) : 1.f;
  constexpr int kChunks = D / 8;  // 8 consecutive d per thread item

  // ---- combine the warps: M = max m_w, l = sum l_w 2^(m_w - M), O likewise
  for (int it = tid; it < G * kChunks; it += blockDim.x) {
    const int g = it / kChunks, c = it % kChunks;
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < kNW; ++w) M = fmaxf(M, wml[(w * 8 + g) * 2]);
    float lsum = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kNW; ++w) {
      const float mw = wml[(w * 8 + g) * 2];
      const float wt = mw == -INFINITY ? 0.f : ex2(mw - M);
      lsum += wml[(w * 8 + g) * 2 + 1] * wt;
      const float4* src = reinterpret_cast<const float4*>(wo + (w * 8 + g) * D + c * 8);
      const float4 x = src[0], y = src[1];
      o[0] += x.x * wt; o[1] += x.y * wt; o[2] += x.z * wt; o[3] += x.w * wt;
      o[4] += y.x * wt; o[5] += y.y * wt; o[6] += y.z * wt; o[7] += y.w * wt;
    }
    const float inv = 1.f / lsum;
    const float lse2 = M + log2f(lsum);
    const size_t row = static_cast<size_t>(b) * p.num_q_heads + h * G + g;
    if (nsplit == 1) {
      uint4 pk;
      if (bad) {
        pk = make_uint4(0, 0, 0, 0);
      } else {
        const float f = inv * vsc;
        pk = make_uint4(pack_bf16(o[0] * f, o[1] * f), pack_bf16(o[2] * f, o[3] * f),
                        pack_bf16(o[4] * f, o[5] * f), pack_bf16(o[6] * f, o[7] * f));
      }
      reinterpret_cast<uint4*>(p.out + row * D)[c] = pk;
      if (c == 0 && p.lse) p.lse[row] = bad ? -INFINITY : lse2 * kLn2;
    } else {
      const size_t slot = (static_cast<size_t>(u) * p.num_splits + split) * 8 + g;
      float4* dst = reinterpret_cast<float4*>(p.ws_o + slot * D + c * 8);
      dst[0] = make_float4(o[0] * inv, o[1] * inv, o[2] * inv, o[3] * inv);
      dst[1] = make_float4(o[4] * inv, o[5] * inv, o[6] * inv, o[7] * inv);
      if (c == 0) p.ws_lse[slot] = bad ? INFINITY : lse2;
    }
  }
  if (nsplit == 1) return;

  // ---- split-K: the last CTA of this (sequence, kv-head) to arrive merges
  __threadfence();
  __syncthreads();
  if (tid == 0) {
    // atomicInc wraps to 0 on the last arrival, leaving the counter ready for the next call
    const unsigned prev = atomicInc(reinterpret_cast<unsigned*>(p.counters + u),
                                    static_cast<unsigned>(nsplit - 1));
    flags[2] = prev == static_cast<unsigned>(nsplit - 1);
  }
  __syncthreads();
  if (!flags[2]) return;
  __threadfence();
  for (int it = tid; it < G * kChunks; it += blockDim.x) {
    const int g = it / kChunks, c = it % kChunks;
    const size_t base = static_cast<size_t>(u) * p.num_splits * 8 + g;
    float M = -INFINITY;
    bool any_bad = false;
    for (int s = 0; s < nsplit; ++s) {
      const float ls = __ldcg(p.ws_lse + base + s * 8);
      any_bad |= ls == INFINITY;
      M = fmaxf(M, ls);
    }
    float lsum = 0.f, o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    if (!any_bad) {
      for (int s = 0; s < nsplit; ++s) {
        const float wt = ex2(__ldcg(p.ws_lse + base + s * 8) - M);
        lsum += wt;
        const float4* src =
            reinterpret_cast<const float4*>(p.ws_o + (base + s * 8) * D + c * 8);
        const float4 x = __ldcg(src), y = __ldcg(src + 1);
        o[0] += x.x * wt; o[1] += x.y * wt; o[2] += x.z * wt; o[3] += x.w * wt;
        o[4] += y.x * wt; o[5] += y.y * wt; o[6] += y.z * wt; o[7] += y.w * wt;
      }
    }
    const size_t row = static_cast<size_t>(b) * p.num_q_heads + h * G + g;
    uint4 pk = make_uint4(0, 0, 0, 0);
    if (!any_bad) {
      const float f = vsc / lsum;
      pk = make_uint4(pack_bf16(o[0] * f, o[1] * f), pack_bf16(o[2] * f, o[3] * f),
                      pack_bf16(o[4] * f, o[5] * f), pack_bf16(o[6] * f, o[7] * f));
    }
    reinterpret_cast<uint4*>(p.out + row * D)[c] = pk;
    if (c == 0 && p.lse) p.lse[row] = any_bad ? -INFINITY : (M + log2f(lsum)) * kLn2;
  }
}

template <int D, bool kFp8>
pgqa_status_t launch_variant(const DecodeArgs& a, const DecodePlan& plan) {
  using C = Cfg<D, kFp8>;
  const CUtensorMapDataType dt =
      kFp8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  const uint64_t rows = static_cast<uint64_t>(a.num_blocks) * a.num_kv_heads * 16;
  CUtensorMap kmap, vmap;
  if (!tensor_map_2d(&kmap, a.k_cache, dt, D, rows, C::kRowBytes, 128 / C::kElem, 16,
                     CU_TENSOR_MAP_SWIZZLE_128B) ||
      !tensor_map_2d(&vmap, a.v_cache, dt, D, rows, C::kRowBytes, 128 / C::kElem, 16,
                     CU_TENSOR_MAP_SWIZZLE_128B))
    return PGQA_ECUDA;
  if (!smem_attr_ready(reinterpret_cast<const void*>(paged_decode_kernel<D, kFp8>), C::kSmem))
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
  p.counters = plan.num_splits > 1 ? reinterpret_cast<int*>(ws + plan.counters_off) : nullptr;
  p.ws_lse = plan.num_splits > 1 ? reinterpret_cast<float*>(ws + plan.lse_off) : nullptr;
  p.ws_o = plan.num_splits > 1 ? reinterpret_cast<float*>(ws + plan.o_off) : nullptr;
  p.dev_status = a.dev_status;
  p.max_blocks_per_seq = a.max_blocks_per_seq;
  p.num_q_heads = a.num_q_heads;
  p.num_kv_heads = a.num_kv_heads;
  p.group = a.num_q_heads / a.num_kv_heads;
  p.num_blocks = a.num_blocks;
  p.max_context_len = a.max_context_len;
  p.pages_per_split = plan.pages_per_split;
  p.num_splits = plan.num_splits;
  p.scale_log2 = a.scale * kLog2e;
  dim3 grid(plan.num_splits, a.num_kv_heads, a.num_seqs);
  paged_decode_kernel<D, kFp8><<<grid, kThreads, C::kSmem, a.stream>>>(kmap, vmap, p);
  return cudaPeekAtLastError() == cudaSuccess ? PGQA_OK : PGQA_ECUDA;
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

}  // namespace

DecodePlan decode_plan(int num_seqs, int num_kv_heads, int head_dim, int max_context_len,
                       int block_size, int num_sms) {
  DecodePlan plan{1, 1, 0, 0, 0, 0};
  const int max_pages = (max_context_len + block_size - 1) / block_size;
  const long units = static_cast<long>(num_seqs) * num_kv_heads;
  if (max_pages <= 0 || units <= 0) {
    plan.pages_per_split = max_pages > 0 ? max_pages : 1;
    return plan;
  }
  const long target = static_cast<long>(num_sms > 0 ? num_sms : 1) * kCtasPerSmTarget;
  long splits = (target + units - 1) / units;
  const long max_splits = (max_pages + kMinPagesPerSplit - 1) / kMinPagesPerSplit;
  if (splits > max_splits) splits = max_splits;
  if (splits < 1) splits = 1;
  const int pps = static_cast<int>((max_pages + splits - 1) / splits);
  plan.pages_per_split = pps;
  plan.num_splits = (max_pages + pps - 1) / pps;
  if (plan.num_splits > 1) {
    const size_t n = static_cast<size_t>(units) * plan.num_splits * 8;
    plan.counters_off = 0;
    plan.lse_off = align256(static_cast<size_t>(units) * sizeof(int));
    plan.o_off = plan.lse_off + align256(n * sizeof(float));
    plan.bytes = plan.o_off + align256(n * head_dim * sizeof(float));
  }
  return plan;
}

pgqa_status_t launch_paged_decode(const DecodeArgs& a, const DecodePlan& plan) {
  if (a.cache_dtype == PGQA_DTYPE_BF16) {
    if (a.head_dim == 128) return launch_variant<128, false>(a, plan);
    if (a.head_dim == 64) return launch_variant<64, false>(a, plan);
  } else if (a.cache_dtype == PGQA_DTYPE_E4M3) {
    if (a.head_dim == 128) return launch_variant<128, true>(a, plan);
  }
  return PGQA_EUNSUPPORTED;
}

}  // namespace pgqa
