/*
 * Oracle for paged grouped-query attention -- TEST INFRASTRUCTURE ONLY.
 *
 * This file is the slow, plain, obviously-correct CPU definition that the CUDA
 * library is checked against. Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg may load it. The product path never calls it and
 * shares no code, header, table or constant with it.
 *
 * Everything is computed in IEEE double precision from the exact input values
 * (bf16 -> double and E4M3 -> double are exact). Loops run in the order the
 * definitions state: gather the pages into contiguous K/V, then dense softmax
 * attention. There is no tiling, no online softmax and no fusion.
 *
 * Sources (web pages on LLM-serving optimisation; titles shortened):
 *  [P1] "Llama 4 inference speed-up: FlashAttention-3 + PagedAttention + vLLM"
 *       (rkmt.cn) -- sec. 2.4 (varlen, causal, out + log-sum-exp),
 *       sec. 3.1 (logical pages -> physical blocks, 16 tokens per block,
 *       page-table fields, pbn = -1 means unallocated).
 *  [P2] "PageAttention + FlashAttention, the golden combination" (lpnh.cn) --
 *       sec. 2.1 (block table maps logical blocks to physical blocks,
 *       block_size 16, copy-on-write sharing of a prompt's blocks).
 *  [P4] "LLM inference surgery log" (xdnf.cn) -- sec. 3.1 (block table int32,
 *       pre-allocated KV blocks updated in place at decode).
 *  [P5] "LLaMA structure and inference performance" (wmrh.cn) -- sec. 2.1
 *       (GQA: query heads of one group share one K/V head), sec. 3.1 (the
 *       attention steps: repeat_kv, Q.K^T / sqrt(head_dim), + mask, softmax in
 *       float32, weighted sum of V), sec. 3.2 (paged KV cache, shared prompt).
 *  OCP 8-bit floating point specification (E4M3: 1 sign, 4 exponent bits with
 *       bias 7, 3 mantissa bits, no infinities, S.1111.111 is NaN, max 448).
 *
 * Readings where the pages are silent or contradictory (listed again in the
 * design notes):
 *  - Cache layout: separate K and V caches, each [num_blocks][num_kv_heads]
 *    [block_size][head_dim], row-major; one (block, kv-head) is contiguous.
 *  - repeat_kv is the index map kv_head = q_head / (num_q_heads/num_kv_heads).
 *  - lse is the natural log of sum_j exp(s_j), with s_j including the scale
 *    (and the fp8 K scale); an empty context gives out = 0, lse = -inf.
 *  - Causal prefill without a cached prefix: query position p of a sequence
 *    sees keys 0..p of the same sequence.
 *  - Sliding-window decode ([P2] sec. 4.1 builds a mask that lets query i see
 *    keys max(0, i-W+1)..i): the decode step of a context of L keys attends to
 *    keys max(0, L-W)..L-1, the last W of them.
 *  - Prefill over a cached prefix ([P1] sec. 2.4 passes separate cumulative
 *    lengths for queries and keys): a chunk of Lq new tokens of a sequence whose
 *    cache holds Lk >= Lq tokens (the chunk's own tokens last) sits at the end of
 *    the sequence, so query i of the chunk (0-based) sees keys 0..Lk-Lq+i
 *    (bottom-right causal alignment); Lk = Lq is the prefill above.
 *  - FP8 cache: stored code = E4M3_rne_satfinite(float(x) / float(scale_h)),
 *    the division done in binary32 (the precision the GPU kernel decides the
 *    code in); dequantised value = E4M3 value * scale_h.
 *  - A negative slot in slot_mapping means "skip this token".
 *
 * Every function returns 0 on success or a negative code on a bad index:
 *   -1 invalid argument, -5 block id or slot out of range.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORACLE_OK 0
#define ORACLE_EINVAL (-1)
#define ORACLE_EBADINDEX (-5)

enum { ORACLE_BF16 = 0, ORACLE_E4M3 = 1 };

/* ---------------------------------------------------------------- scalars */

/* bf16 is the top half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_f64(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* E4M3 code -> value, straight from the format definition. */
double oracle_e4m3_to_f64(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 15;
    int m = code & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);          /* subnormal: 0.m * 2^(1-7) */
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7); /* normal: 1.m * 2^(e-7) */
    return sign ? -v : v;
}

/* binary32 -> E4M3 by round-to-nearest, ties to the even code, saturating
 * finite values to +-448. Written as a search over the 127 finite magnitudes so
 * that it is the definition itself: the nearest representable value wins; at an
 * exact midpoint the code whose last bit is 0 wins. NaN maps to the NaN code. */
uint8_t oracle_e4m3_from_f32(float x) {
    uint8_t sign = signbit(x) ? 0x80 : 0x00;
    double a, best_err = INFINITY;
    int best = 0;
    if (isnan(x)) return 0x7F;
    a = fabs((double)x);
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    for (int c = 0; c <= 0x7E; ++c) {
        double err = fabs(oracle_e4m3_to_f64((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0 && (best & 1) == 1)) {
            best_err = err;
            best = c;
        }
    }
    return (uint8_t)(sign | best);
}

/* Value of one cache element as a double. */
static double cache_elem(const void* cache, int dtype, size_t idx, double scale_h) {
    if (dtype == ORACLE_BF16) return oracle_bf16_to_f64(((const uint16_t*)cache)[idx]);
    return oracle_e4m3_to_f64(((const uint8_t*)cache)[idx]) * scale_h;
}

/* Flat index of (block, kv-head, row, d) in a [NB][Hkv][bs][D] cache. */
static size_t cache_index(int64_t block, int h, int row, int d, int Hkv, int bs, int D) {
    return (((size_t)block * Hkv + h) * bs + row) * D + d;
}

/* ------------------------------------------------------- kv cache write */

/* Scatter of new K/V rows into their slots ([P4] sec. 3.1 in-place update;
 * [P1] sec. 3.1 slot = physical block * block_size + row).
 * key, value: [T][Hkv][D] bf16. slot_mapping: [T] int64, negative = skip.
 * k_cache/v_cache: [NB][Hkv][bs][D], bf16 (uint16) or E4M3 (uint8).
 * k_scale/v_scale: [Hkv] float (E4M3 only). */
int oracle_kv_cache_write(const uint16_t* key, const uint16_t* value, const int64_t* slot_mapping,
                          int T, int Hkv, int D, void* k_cache, void* v_cache, int num_blocks,
                          int block_size, int dtype, const float* k_scale, const float* v_scale) {
    if (T < 0 || Hkv <= 0 || D <= 0 || block_size <= 0) return ORACLE_EINVAL;
    if (dtype == ORACLE_E4M3 && (!k_scale || !v_scale)) return ORACLE_EINVAL;
    for (int t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        int64_t block;
        int row;
        if (slot < 0) continue;
        block = slot / block_size;
        row = (int)(slot % block_size);
        if (block >= num_blocks) return ORACLE_EBADINDEX;
        for (int h = 0; h < Hkv; ++h) {
            for (int d = 0; d < D; ++d) {
                size_t src = ((size_t)t * Hkv + h) * D + d;
                size_t dst = cache_index(block, h, row, d, Hkv, block_size, D);
                if (dtype == ORACLE_BF16) {
                    ((uint16_t*)k_cache)[dst] = key[src];
                    ((uint16_t*)v_cache)[dst] = value[src];
                } else {
                    float xk = (float)oracle_bf16_to_f64(key[src]);
                    float xv = (float)oracle_bf16_to_f64(value[src]);
                    ((uint8_t*)k_cache)[dst] = oracle_e4m3_from_f32(xk / k_scale[h]);
                    ((uint8_t*)v_cache)[dst] = oracle_e4m3_from_f32(xv / v_scale[h]);
                }
            }
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------------ page gather */

/* Logical token j of sequence s lives in physical block block_table[s][j / bs],
 * row j % bs ([P1] sec. 3.1, [P2] sec. 2.1). Copies the first L tokens of kv-head
 * h into contiguous K, V [L][D] (doubles, dequantised). Returns EBADINDEX if a
 * block id needed for j < L is negative (unallocated) or >= num_blocks. */
int oracle_gather_kv(const void* k_cache, const void* v_cache, int dtype, const float* k_scale,
                     const float* v_scale, const int32_t* block_table_row, int max_blocks_per_seq,
                     int L, int h, int Hkv, int D, int num_blocks, int block_size, double* K,
                     double* V) {
    double ks = 1.0, vs = 1.0;
    if (dtype == ORACLE_E4M3) {
        ks = k_scale[h];
        vs = v_scale[h];
    }
    for (int j = 0; j < L; ++j) {
        int lpn = j / block_size;
        int row = j % block_size;
        int32_t pbn;
        if (lpn >= max_blocks_per_seq) return ORACLE_EBADINDEX;
        pbn = block_table_row[lpn];
        if (pbn < 0 || pbn >= num_blocks) return ORACLE_EBADINDEX;
        for (int d = 0; d < D; ++d) {
            size_t idx = cache_index(pbn, h, row, d, Hkv, block_size, D);
            K[(size_t)j * D + d] = cache_elem(k_cache, dtype, idx, ks);
            V[(size_t)j * D + d] = cache_elem(v_cache, dtype, idx, vs);
        }
    }
    return ORACLE_OK;
}

/* ------------------------------------------------------ dense attention */

/* One query row against contiguous K, V [L][D] ([P5] sec. 3.1 steps 3-6):
 *   s_j = scale * sum_d q_d K_jd
 *   lse = ln sum_j exp(s_j)           (computed as m + ln sum_j exp(s_j - m))
 *   p_j = exp(s_j - lse)
 *   out_d = sum_j p_j V_jd
 * L == 0 gives out = 0, lse = -inf. scores is caller scratch of length >= L. */
static void attend_row(const double* q, const double* K, const double* V, int L, int D,
                       double scale, double* scores, double* out, double* lse) {
    double m = -INFINITY, sum = 0.0, l;
    for (int d = 0; d < D; ++d) out[d] = 0.0;
    if (L == 0) {
        *lse = -INFINITY;
        return;
    }
    for (int j = 0; j < L; ++j) {
        double s = 0.0;
        for (int d = 0; d < D; ++d) s += q[d] * K[(size_t)j * D + d];
        scores[j] = scale * s;
        if (scores[j] > m) m = scores[j];
    }
    for (int j = 0; j < L; ++j) sum += exp(scores[j] - m);
    l = m + log(sum);
    for (int j = 0; j < L; ++j) {
        double p = exp(scores[j] - l);
        for (int d = 0; d < D; ++d) out[d] += p * V[(size_t)j * D + d];
    }
    *lse = l;
}

/* ------------------------------------------------------------ decode */

/* Paged decode: one query token per sequence.
 * q: [B][Hq][D] bf16. block_tables: [B][max_blocks_per_seq] int32.
 * context_lens: [B] int32. out: [B][Hq][D] double. lse: [B][Hq] double.
 * GQA index map ([P5] sec. 2.1, repeat_kv in sec. 3.1): kv-head = hq / (Hq/Hkv). */
int oracle_paged_decode(const uint16_t* q, const void* k_cache, const void* v_cache, int dtype,
                        const float* k_scale, const float* v_scale, const int32_t* block_tables,
                        int max_blocks_per_seq, const int32_t* context_lens, int B, int Hq,
                        int Hkv, int D, int num_blocks, int block_size, double scale, double* out,
                        double* lse, int nthreads) {
    int G, status = ORACLE_OK;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || block_size <= 0)
        return ORACLE_EINVAL;
    if (dtype == ORACLE_E4M3 && (!k_scale || !v_scale)) return ORACLE_EINVAL;
    G = Hq / Hkv;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t bh = 0; bh < (int64_t)B * Hkv; ++bh) {
        int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
        int L = context_lens[b];
        double *K, *V, *qd, *scores;
        int rc;
        if (L < 0) {
#pragma omp critical
            status = ORACLE_EINVAL;
            continue;
        }
        K = (double*)malloc(sizeof(double) * ((size_t)L * D + 1));
        V = (double*)malloc(sizeof(double) * ((size_t)L * D + 1));
        qd = (double*)malloc(sizeof(double) * D);
        scores = (double*)malloc(sizeof(double) * ((size_t)L + 1));
        rc = oracle_gather_kv(k_cache, v_cache, dtype, k_scale, v_scale,
                              block_tables + (size_t)b * max_blocks_per_seq, max_blocks_per_seq, L,
                              h, Hkv, D, num_blocks, block_size, K, V);
        if (rc != ORACLE_OK) {
#pragma omp critical
            status = rc;
        } else {
            for (int g = 0; g < G; ++g) {
                int hq = h * G + g;
                const uint16_t* qrow = q + ((size_t)b * Hq + hq) * D;
                for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);
                attend_row(qd, K, V, L, D, scale, scores, out + ((size_t)b * Hq + hq) * D,
                           lse + (size_t)b * Hq + hq);
            }
        }
        free(K);
        free(V);
        free(qd);
        free(scores);
    }
    return status;
}

/* ------------------------------------------------------------ prefill */

/* Causal variable-length prefill over a paged cache ([P1] sec. 2.4: varlen
 * batch given by cumulative lengths, causal=True, returns out and lse).
 * q: [T][Hq][D] bf16 with T = cu_seqlens[num_seqs]. Sequence i owns tokens
 * cu_seqlens[i] .. cu_seqlens[i+1]-1; the token at position p of sequence i
 * attends to keys 0..p of sequence i, read through block_tables[i].
 * rows: optional list of n_rows (token, q_head) pairs to compute (int32 pairs);
 * NULL computes every (token, head). out: [T][Hq][D] double, lse: [T][Hq] double
 * (only the requested rows are written). dtype/k_scale/v_scale as for
 * oracle_paged_decode (an E4M3 cache is dequantised per kv-head). */
int oracle_paged_prefill(const uint16_t* q, const void* k_cache, const void* v_cache, int dtype,
                         const float* k_scale, const float* v_scale, const int32_t* block_tables,
                         int max_blocks_per_seq, const int32_t* cu_seqlens, int num_seqs, int Hq,
                         int Hkv, int D, int num_blocks, int block_size, double scale,
                         const int32_t* rows, int64_t n_rows, double* out, double* lse,
                         int nthreads) {
    int G, status = ORACLE_OK;
    int64_t T, n_items;
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || block_size <= 0)
        return ORACLE_EINVAL;
    if (dtype == ORACLE_E4M3 && (!k_scale || !v_scale)) return ORACLE_EINVAL;
    for (int i = 0; i < num_seqs; ++i)
        if (cu_seqlens[i + 1] < cu_seqlens[i] || cu_seqlens[0] != 0) return ORACLE_EINVAL;
    G = Hq / Hkv;
    T = cu_seqlens[num_seqs];
    n_items = rows ? n_rows : T * Hq;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t it = 0; it < n_items; ++it) {
        int64_t t = rows ? rows[2 * it] : it / Hq;
        int hq = rows ? rows[2 * it + 1] : (int)(it % Hq);
        int i = 0, p, L, h, rc;
        double *K, *V, *qd, *scores;
        if (t < 0 || t >= T || hq < 0 || hq >= Hq) {
#pragma omp critical
            status = ORACLE_EINVAL;
            continue;
        }
        while (cu_seqlens[i + 1] <= t) ++i; /* the sequence that owns token t */
        p = (int)(t - cu_seqlens[i]);        /* its position in that sequence */
        L = p + 1;                           /* causal: keys 0..p */
        h = hq / G;
        K = (double*)malloc(sizeof(double) * (size_t)L * D);
        V = (double*)malloc(sizeof(double) * (size_t)L * D);
        qd = (double*)malloc(sizeof(double) * D);
        scores = (double*)malloc(sizeof(double) * (size_t)L);
        rc = oracle_gather_kv(k_cache, v_cache, dtype, k_scale, v_scale,
                              block_tables + (size_t)i * max_blocks_per_seq, max_blocks_per_seq, L,
                              h, Hkv, D, num_blocks, block_size, K, V);
        if (rc != ORACLE_OK) {
#pragma omp critical
            status = rc;
        } else {
            const uint16_t* qrow = q + ((size_t)t * Hq + hq) * D;
            for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);
            attend_row(qd, K, V, L, D, scale, scores, out + ((size_t)t * Hq + hq) * D,
                       lse + (size_t)t * Hq + hq);
        }
        free(K);
        free(V);
        free(qd);
        free(scores);
    }
    return status;
}

/* Sliding-window decode: as oracle_paged_decode, attending only to keys
 * max(0, L-W)..L-1 of each context ([P2] sec. 4.1, query i sees keys i-W+1..i). */
int oracle_paged_decode_window(const uint16_t* q, const void* k_cache, const void* v_cache,
                               int dtype, const float* k_scale, const float* v_scale,
                               const int32_t* block_tables, int max_blocks_per_seq,
                               const int32_t* context_lens, int B, int Hq, int Hkv, int D,
                               int num_blocks, int block_size, double scale, int window,
                               double* out, double* lse, int nthreads) {
    int G, status = ORACLE_OK;
    if (B < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || block_size <= 0 ||
        window <= 0)
        return ORACLE_EINVAL;
    if (dtype == ORACLE_E4M3 && (!k_scale || !v_scale)) return ORACLE_EINVAL;
    G = Hq / Hkv;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t bh = 0; bh < (int64_t)B * Hkv; ++bh) {
        int b = (int)(bh / Hkv), h = (int)(bh % Hkv);
        int L = context_lens[b];
        int first = L > window ? L - window : 0; /* the window's first key */
        double *K, *V, *qd, *scores;
        int rc;
        if (L < 0) {
#pragma omp critical
            status = ORACLE_EINVAL;
            continue;
        }
        K = (double*)malloc(sizeof(double) * ((size_t)L * D + 1));
        V = (double*)malloc(sizeof(double) * ((size_t)L * D + 1));
        qd = (double*)malloc(sizeof(double) * D);
        scores = (double*)malloc(sizeof(double) * ((size_t)L + 1));
        rc = oracle_gather_kv(k_cache, v_cache, dtype, k_scale, v_scale,
                              block_tables + (size_t)b * max_blocks_per_seq, max_blocks_per_seq, L,
                              h, Hkv, D, num_blocks, block_size, K, V);
        if (rc != ORACLE_OK) {
#pragma omp critical
            status = rc;
        } else {
            for (int g = 0; g < G; ++g) {
                int hq = h * G + g;
                const uint16_t* qrow = q + ((size_t)b * Hq + hq) * D;
                for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);
                attend_row(qd, K + (size_t)first * D, V + (size_t)first * D, L - first, D, scale,
                           scores, out + ((size_t)b * Hq + hq) * D, lse + (size_t)b * Hq + hq);
            }
        }
        free(K);
        free(V);
        free(qd);
        free(scores);
    }
    return status;
}

/* Chunked prefill over a cached prefix: as oracle_paged_prefill, with seq_lens_k[i]
 * (>= the chunk's length Lq) the number of tokens sequence i has in the cache,
 * the chunk's tokens last; query i of the chunk sees keys 0..Lk-Lq+i ([P1] sec. 2.4,
 * the varlen call with separate query and key lengths; bottom-right alignment). */
int oracle_paged_prefill_kv(const uint16_t* q, const void* k_cache, const void* v_cache,
                            int dtype, const float* k_scale, const float* v_scale,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, int num_seqs,
                            int Hq, int Hkv, int D, int num_blocks, int block_size, double scale,
                            const int32_t* rows, int64_t n_rows, double* out, double* lse,
                            int nthreads) {
    int G, status = ORACLE_OK;
    int64_t T, n_items;
    if (num_seqs < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || D <= 0 || block_size <= 0)
        return ORACLE_EINVAL;
    if (dtype == ORACLE_E4M3 && (!k_scale || !v_scale)) return ORACLE_EINVAL;
    if (num_seqs > 0 && cu_seqlens_q[0] != 0) return ORACLE_EINVAL;
    for (int i = 0; i < num_seqs; ++i)
        if (cu_seqlens_q[i + 1] < cu_seqlens_q[i] ||
            seq_lens_k[i] < cu_seqlens_q[i + 1] - cu_seqlens_q[i])
            return ORACLE_EINVAL;
    G = Hq / Hkv;
    T = num_seqs > 0 ? cu_seqlens_q[num_seqs] : 0;
    n_items = rows ? n_rows : T * Hq;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 4) num_threads(nthreads > 0 ? nthreads : 1)
    for (int64_t it = 0; it < n_items; ++it) {
        int64_t t = rows ? rows[2 * it] : it / Hq;
        int hq = rows ? rows[2 * it + 1] : (int)(it % Hq);
        int i = 0, p, L, h, rc, Lq, Lk;
        double *K, *V, *qd, *scores;
        if (t < 0 || t >= T || hq < 0 || hq >= Hq) {
#pragma omp critical
            status = ORACLE_EINVAL;
            continue;
        }
        while (cu_seqlens_q[i + 1] <= t) ++i; /* the sequence that owns token t */
        p = (int)(t - cu_seqlens_q[i]);        /* its position in the chunk */
        Lq = cu_seqlens_q[i + 1] - cu_seqlens_q[i];
        Lk = seq_lens_k[i];
        L = Lk - Lq + p + 1; /* keys 0..Lk-Lq+p */
        h = hq / G;
        K = (double*)malloc(sizeof(double) * (size_t)L * D);
        V = (double*)malloc(sizeof(double) * (size_t)L * D);
        qd = (double*)malloc(sizeof(double) * D);
        scores = (double*)malloc(sizeof(double) * (size_t)L);
        rc = oracle_gather_kv(k_cache, v_cache, dtype, k_scale, v_scale,
                              block_tables + (size_t)i * max_blocks_per_seq, max_blocks_per_seq, L,
                              h, Hkv, D, num_blocks, block_size, K, V);
        if (rc != ORACLE_OK) {
#pragma omp critical
            status = rc;
        } else {
            const uint16_t* qrow = q + ((size_t)t * Hq + hq) * D;
            for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(qrow[d]);
            attend_row(qd, K, V, L, D, scale, scores, out + ((size_t)t * Hq + hq) * D,
                       lse + (size_t)t * Hq + hq);
        }
        free(K);
        free(V);
        free(qd);
        free(scores);
    }
    return status;
}

/* Dense contiguous attention for one (query row, K, V) -- the same step the
 * paged functions end in, exposed so tests can compare paged against contiguous
 * on identical data. q: [D] bf16; K, V: [L][D] doubles. */
void oracle_dense_row(const uint16_t* q, const double* K, const double* V, int L, int D,
                      double scale, double* out, double* lse) {
    double* qd = (double*)malloc(sizeof(double) * D);
    double* scores = (double*)malloc(sizeof(double) * ((size_t)L + 1));
    for (int d = 0; d < D; ++d) qd[d] = oracle_bf16_to_f64(q[d]);
    attend_row(qd, K, V, L, D, scale, scores, out, lse);
    free(qd);
    free(scores);
}

/* 1 when this build runs the per-(sequence, head) loops on OpenMP threads. */
int oracle_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}
