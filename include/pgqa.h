/*
 * pgqa.h -- C ABI of the paged grouped-query attention library (libpgqa.so).
 *
 * Attention over a paged KV cache, as the LLM-serving pages on PagedAttention
 * and FlashAttention describe it:
 *  - "Llama 4 inference speed-up: FlashAttention-3 + PagedAttention + vLLM"
 *    (rkmt.cn), sec. 3.1: the KV cache is a logical address space cut into
 *    fixed 16-token pages; a page table maps logical page numbers to physical
 *    block numbers (int32, -1 = unallocated); sec. 2.4: variable-length batches
 *    given by cumulative sequence lengths, causal masking, outputs out and the
 *    log-sum-exp.
 *  - "PageAttention + FlashAttention, the golden combination" (lpnh.cn),
 *    sec. 2.1: per-request block tables, block_size 16, copy-on-write sharing
 *    of a prompt's blocks between sequences.
 *  - "LLM inference surgery log" (xdnf.cn), sec. 3.1: an int32 block table per
 *    sequence and a pre-allocated pool of KV blocks updated in place at decode.
 *  - "LLaMA structure and inference performance" (wmrh.cn), sec. 2.1: grouped-
 *    query attention (query heads of one group share one K/V head); sec. 3.1:
 *    scores Q.K^T * scale, mask, softmax in float32, weighted sum of V.
 *
 * Conventions shared by every call
 *  - Tensors are dense, row-major, in DEVICE memory owned by the caller. The
 *    library never allocates, frees or keeps a pointer past the call, and it
 *    keeps no state between calls other than a host-side cache of TMA tensor
 *    descriptors keyed by (address, shape).
 *  - The KV cache is two tensors, k_cache and v_cache, each
 *      [num_blocks][num_kv_heads][block_size][head_dim]
 *    so one (block, kv-head) page of block_size x head_dim elements is
 *    contiguous (4 KB for bf16 at 16 x 128). Element type cache_dtype:
 *      PGQA_DTYPE_BF16  bfloat16
 *      PGQA_DTYPE_E4M3  FP8 E4M3 codes (OCP OFP8); the real value of a code in
 *                       kv-head h is E4M3(code) * scale[h], with separate fp32
 *                       k_scale[num_kv_heads] and v_scale[num_kv_heads].
 *  - Logical token j of sequence s is row j % block_size of physical block
 *    block_tables[s * max_blocks_per_seq + j / block_size]. Entries at or past
 *    ceil(context_len / block_size) are never read and may hold -1.
 *  - Query head hq uses kv-head hq / (num_q_heads / num_kv_heads).
 *  - scores are scale * q.k (times k_scale[h] for E4M3); lse is the natural
 *    log of the sum of exp(score) over the attended keys.
 *  - All calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and run on the current CUDA device.
 *  - The kernels launch programmatically: a call's kernel may start while the
 *    stream's previous kernel finishes, and waits for it before touching q, K/V
 *    rows, the caches, out, lse or the workspace. The decode calls read
 *    block_tables and context_lens BEFORE that wait, so the kernel enqueued right
 *    before a decode call must not write them if it releases its dependents early
 *    (griddepcontrol.launch_dependents / cudaTriggerProgrammaticLaunchCompletion).
 *    Copies, and kernels that do not release early (ordinary kernels), are fully
 *    ordered; no kernel of this library writes either array.
 *  - Supported now: head_dim 64 or 128, bf16 q/out; block_size 8, 16 or 32
 *    and 1 <= num_q_heads / num_kv_heads <= 8 for decode (bf16 or E4M3 cache);
 *    block_size 16 and any group size for prefill (bf16 or E4M3 cache); any
 *    block_size for kv_cache_write.
 *
 * Errors
 *  - Argument errors found on the host return a negative pgqa_status_t and
 *    launch nothing.
 *  - Errors found on the device never fault: a block id < 0 or >= num_blocks
 *    inside a context, or a slot past the pool, is PGQA_EBADINDEX; a context
 *    longer than max_context_len or than the block table is PGQA_EINVAL. The
 *    kernel skips the affected rows (attention rows are written as out = 0,
 *    lse = -inf) and, when dev_status is non-NULL, stores the first such code
 *    into *dev_status (a device int the caller zeroes; later errors do not
 *    overwrite it). A bounded wait inside a kernel that gives up stores
 *    PGQA_ETIMEOUT the same way.
 */
#ifndef PGQA_H
#define PGQA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int pgqa_status_t;

#define PGQA_OK 0
#define PGQA_EINVAL (-1)        /* null pointer, negative size, inconsistent shapes, misalignment */
#define PGQA_EUNSUPPORTED (-2)  /* valid request this build does not implement */
#define PGQA_ENOWORKSPACE (-3)  /* workspace_bytes smaller than the matching *_workspace_size */
#define PGQA_ECUDA (-4)         /* a CUDA runtime call or kernel launch failed */
#define PGQA_EBADINDEX (-5)     /* device: block id or slot out of range */
#define PGQA_ETIMEOUT (-6)      /* device: a bounded wait on a barrier gave up */

#define PGQA_DTYPE_BF16 0
#define PGQA_DTYPE_E4M3 1

#define PGQA_ABI_VERSION 1

/* ABI version of the loaded library (PGQA_ABI_VERSION it was built with). */
int pgqa_abi_version(void);

/* Static, NUL-terminated description of a status code. Never NULL. */
const char* pgqa_status_string(pgqa_status_t status);

/*
 * Failure-detection aid (the pages have no counterpart; it exists so that the bounded
 * waits can be tested without faulting a GPU). Every wait inside the decode kernels
 * (pgqa_paged_attention_decode and its window, append and noalloc forms) is bounded: the
 * consumer and merge warps' barrier waits and the producer's wait for free stages give
 * up after 2 s by default, store PGQA_ETIMEOUT in *dev_status and let the kernel end.
 * This sets that limit, in nanoseconds, for the decode launches made after it on any
 * device (0 restores the 2 s default); a very short limit makes those waits run out.
 * The producer's final wait for its own copies in flight always keeps the 2 s limit, so
 * no copy can land after a thread block exits. After a call that reported
 * PGQA_ETIMEOUT the call's outputs are undefined and its workspace must be zero-filled
 * again before reuse. Host only; a process-wide setting (not synchronised with launches
 * made concurrently from other host threads).
 */
void pgqa_set_decode_wait_limit_ns(uint64_t ns);

/* Bytes of KV cache for `num_layers` layers of `tokens` cached tokens:
 * 2 (K and V) * layers * tokens * kv-heads * head_dim * element size
 * ("LLaMA structure and inference performance", sec. 5, sizes a 4K-context
 * 32-layer cache at about 2.1 GB for 32 heads and about 0.5 GB for 8 kv-heads).
 * Returns -1 for a negative argument or an unknown dtype. Host only. */
int64_t pgqa_kv_cache_bytes(int num_layers, int64_t tokens, int num_kv_heads, int head_dim,
                            int cache_dtype);

/*
 * Scatter new K/V rows into the paged cache (the in-place update at decode of
 * "LLM inference surgery log", sec. 3.1; slot = physical block * block_size +
 * row, from the page-table description of the rkmt.cn article, sec. 3.1).
 *
 *   key, value    [num_tokens][num_kv_heads][head_dim] bf16, read.
 *   slot_mapping  [num_tokens] int64, read. slot < 0: token skipped.
 *                 Otherwise block = slot / block_size (must be < num_blocks),
 *                 row = slot % block_size. Two tokens must not share a slot.
 *   k_cache, v_cache  the cache described above, written at those slots only.
 *   cache_dtype   PGQA_DTYPE_BF16: bit-exact copy.
 *                 PGQA_DTYPE_E4M3: code = E4M3 round-to-nearest-even, saturated
 *                 to +-448, of float(x) / scale[h] (binary32 division);
 *                 k_scale / v_scale [num_kv_heads] fp32 device arrays, read.
 *                 Must be NULL for bf16.
 *   dev_status    optional device int, see "Errors".
 * head_dim must be a multiple of 8; key/value 16-byte aligned.
 */
pgqa_status_t pgqa_kv_cache_write(const void* key, const void* value,
                                  const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                                  int head_dim, void* k_cache, void* v_cache, int num_blocks,
                                  int block_size, int cache_dtype, const float* k_scale,
                                  const float* v_scale, int* dev_status, void* stream);

/*
 * Gather the pages of each sequence into contiguous K and V (a debugging and
 * testing aid that exercises exactly the block-table addressing the attention
 * kernels use).
 *
 *   k_out, v_out  [num_seqs][num_kv_heads][max_context_len][head_dim] in the
 *                 cache's element type, written: rows j < context_lens[s] are a
 *                 bit-exact copy of the cache; rows past it are zero.
 * Other arguments as for pgqa_paged_attention_decode.
 */
pgqa_status_t pgqa_paged_kv_gather(const void* k_cache, const void* v_cache, int cache_dtype,
                                   const int32_t* block_tables, int max_blocks_per_seq,
                                   const int32_t* context_lens, int num_seqs, int num_kv_heads,
                                   int head_dim, int num_blocks, int block_size,
                                   int max_context_len, void* k_out, void* v_out,
                                   int* dev_status, void* stream);

/*
 * Grid of paged decode (host logic, no device access): the number of CTAs the
 * decode kernel launches on a device with `num_sms` multiprocessors for this
 * head_dim and cache dtype. Each CTA owns an equal share of all cached pages of
 * the batch (laid end to end in (sequence, kv-head) order), so ragged context
 * lengths cannot unbalance the GPU. Returns PGQA_EINVAL on a bad argument.
 */
int pgqa_decode_grid_size(int num_sms, int head_dim, int cache_dtype);

/* Workspace bytes pgqa_paged_attention_decode needs on the current device for
 * these sizes (any cache dtype): one ticket counter per (sequence, kv-head) and
 * two partial-result slots of 8 x head_dim floats per CTA. max_context_len does
 * not change it. */
size_t pgqa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                  int max_context_len);

/*
 * Paged decode attention: one new query token per sequence attends to its
 * whole cached context ("LLaMA structure and inference performance", sec. 3.1
 * steps 2-6 with repeat_kv as the index map of sec. 2.1, read through the block
 * table of the rkmt.cn article, sec. 3.1). Each KV byte is read once: one
 * thread block serves all query heads of a kv-head.
 *
 *   out           [num_seqs][num_q_heads][head_dim] bf16, written
 *                 (fp32 accumulation, rounded to nearest even).
 *   lse           [num_seqs][num_q_heads] fp32, written; may be NULL.
 *   q             [num_seqs][num_q_heads][head_dim] bf16, read.
 *   block_tables  [num_seqs][max_blocks_per_seq] int32, read.
 *   context_lens  [num_seqs] int32, read; 0 gives out = 0, lse = -inf.
 *   block_size    8, 16 or 32 tokens (PGQA_EUNSUPPORTED otherwise); the kernel
 *                 reads 16-token pages: half a 32-token block, or two 8-token
 *                 blocks whose ids are checked separately.
 *   scale         softmax scale (usually 1/sqrt(head_dim)).
 *   cache_dtype, k_scale, v_scale   as for pgqa_kv_cache_write.
 *   max_context_len  an upper bound on context_lens; a longer context is a
 *                 device error.
 *   workspace     device scratch of at least pgqa_decode_workspace_size()
 *                 bytes, 256-byte aligned, ZERO-FILLED before its first use;
 *                 every call that completes leaves it ready for the next call.
 *                 Calls that share one workspace must not overlap in time.
 * k_cache/v_cache must be 16-byte aligned, q/out 16-byte aligned.
 */
pgqa_status_t pgqa_paged_attention_decode(void* out, float* lse, const void* q,
                                          const void* k_cache, const void* v_cache,
                                          const int32_t* block_tables, int max_blocks_per_seq,
                                          const int32_t* context_lens, int num_seqs,
                                          int num_q_heads, int num_kv_heads, int head_dim,
                                          int num_blocks, int block_size, float scale,
                                          int cache_dtype, const float* k_scale,
                                          const float* v_scale, int max_context_len,
                                          void* workspace, size_t workspace_bytes,
                                          int* dev_status, void* stream);

/*
 * Sliding-window paged decode: as pgqa_paged_attention_decode, but a context of L
 * keys attends only to its last `window` keys, L-window .. L-1 (the sliding-window
 * mask of "PageAttention + FlashAttention, the golden combination", sec. 4.1:
 * query i sees keys i-W+1 .. i). Only the pages holding those keys are read.
 *   window        >= 1 (PGQA_EINVAL otherwise); a window of at least the context
 *                 is plain decode.
 * Every other argument, the workspace (pgqa_decode_workspace_size) and the error
 * behaviour are as for pgqa_paged_attention_decode.
 */
pgqa_status_t pgqa_paged_attention_decode_window(
    void* out, float* lse, const void* q, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, int block_size,
    float scale, int window, int cache_dtype, const float* k_scale, const float* v_scale,
    int max_context_len, void* workspace, size_t workspace_bytes, int* dev_status, void* stream);

/* Size of the library-owned scratch array used by
 * pgqa_paged_attention_decode_noalloc (8 MiB on each GPU where it has been set up). */
#define PGQA_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/*
 * pgqa_paged_attention_decode_noalloc -- the same paged decode attention as
 * pgqa_paged_attention_decode, for callers that cannot allocate device memory.
 * The pages have no counterpart for this entry point; it exists for users of the
 * library: a serving engine that sizes its KV block pool to fill the GPU's free
 * memory at start-up (so a later cudaMalloc fails), or a plugin hosted inside
 * another framework whose device memory belongs to that framework's allocator,
 * has nowhere to get the split-K workspace from.
 *
 * Arguments are those of pgqa_paged_attention_decode without the workspace; the
 * caller still passes every input and output. The split-K scratch is a static
 * device array of PGQA_NOALLOC_SCRATCH_BYTES owned by the library:
 *  - per-device set-up: the first call on a device, with that device current,
 *    looks up the array's device address (cudaGetSymbolAddress) and loads the
 *    decode kernels there. Under the CUDA runtime's lazy module loading (the
 *    default) that is also when the device allocates the array and the kernels'
 *    code, so make this first call BEFORE filling the device's free memory, and
 *    before any stream capture. A call with num_seqs == 0 (the other pointers may
 *    be NULL) does only this set-up and enqueues nothing; later calls on that
 *    device allocate nothing;
 *  - arguments are checked on the host first: a call that returns an error has
 *    enqueued nothing; sizes whose workspace (pgqa_decode_workspace_size) exceeds
 *    the array are rejected with PGQA_ENOWORKSPACE;
 *  - each call clears the array's merge counters with cudaMemsetAsync on
 *    `stream`, then launches the decode kernel; it never calls cudaMalloc,
 *    cudaFree or any allocating routine;
 *  - all calls share the one array, so calls that overlap on the GPU (other
 *    streams, other host threads) race and must be serialised by the caller.
 */
pgqa_status_t pgqa_paged_attention_decode_noalloc(void* out, float* lse, const void* q,
                                                  const void* k_cache, const void* v_cache,
                                                  const int32_t* block_tables,
                                                  int max_blocks_per_seq,
                                                  const int32_t* context_lens, int num_seqs,
                                                  int num_q_heads, int num_kv_heads, int head_dim,
                                                  int num_blocks, int block_size, float scale,
                                                  int cache_dtype, const float* k_scale,
                                                  const float* v_scale, int max_context_len,
                                                  int* dev_status, void* stream);

/*
 * One decode step with the append fused in: the new token of every sequence is
 * written into the cache and attended in one launch. context_lens[b] counts the new
 * token; its K and V rows go to position L-1 of sequence b, i.e. block
 * block_tables[b][(L-1) / block_size], row (L-1) % block_size: exactly what
 * pgqa_kv_cache_write writes for a slot mapping pointing there (bf16 copy, or the
 * same E4M3 codes), and the attention then reads it as pgqa_paged_attention_decode
 * does (the page-cache update then attention of the surgery-log article, sec. 3.1,
 * and the LLaMA-structure article's decode step, sec. 3.1).
 *   key, value    [num_seqs][num_kv_heads][head_dim] bf16, read; 16-byte aligned.
 *   k_cache, v_cache  read and written.
 * A sequence whose length is invalid (a device error, as for
 * pgqa_paged_attention_decode) or 0 gets no append; a bad block id for position L-1
 * is PGQA_EBADINDEX and nothing is written there. Every other argument, the
 * workspace and the error behaviour are as for pgqa_paged_attention_decode.
 */
pgqa_status_t pgqa_paged_attention_decode_append(
    void* out, float* lse, const void* q, const void* key, const void* value, void* k_cache,
    void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* context_lens, int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
    int num_blocks, int block_size, float scale, int cache_dtype, const float* k_scale,
    const float* v_scale, int max_context_len, void* workspace, size_t workspace_bytes,
    int* dev_status, void* stream);

/* Most new tokens per sequence pgqa_paged_attention_decode_multi takes. */
#define PGQA_MAX_DECODE_TOKENS 8

/* Workspace bytes pgqa_paged_attention_decode_multi needs on the current device for
 * these sizes (any cache dtype and block size): as for pgqa_decode_workspace_size, with
 * partial-result slots for the q_len x group query rows of a (sequence, kv-head); or the
 * prefill workspace when those rows are more than 32 (see below). 0 on a bad argument. */
size_t pgqa_decode_multi_workspace_size(int num_seqs, int q_len, int num_q_heads,
                                        int num_kv_heads, int head_dim);

/*
 * Multi-token paged decode: q_len new tokens per sequence attend to the cached context,
 * each causally -- speculative verification of draft tokens (the rkmt.cn article's
 * speculative decoding, sec. 4.2, drafts several tokens per step) as the varlen call
 * with per-sequence query and key lengths of sec. 2.4, every chunk q_len long. The
 * drafts' K/V must already be in the cache (pgqa_kv_cache_write): context_lens[b]
 * counts them, and token t of sequence b attends keys 0 .. context_lens[b] - q_len + t
 * (bottom-right causal alignment), read through its block table.
 *
 *   out           [num_seqs][q_len][num_q_heads][head_dim] bf16, written.
 *   lse           [num_seqs][q_len][num_q_heads] fp32, written; may be NULL.
 *   q             [num_seqs][q_len][num_q_heads][head_dim] bf16, read.
 *   q_len         1 .. PGQA_MAX_DECODE_TOKENS (PGQA_EINVAL below, PGQA_EUNSUPPORTED above).
 *   context_lens  [num_seqs] int32, read: 0 (nothing to attend: out = 0, lse = -inf) or
 *                 at least q_len (a shorter context is a device error, PGQA_EINVAL).
 *   workspace     at least pgqa_decode_multi_workspace_size() bytes, 256-byte aligned,
 *                 ZERO-FILLED before its first use; every call that completes leaves
 *                 it ready for the next call.
 * Every other argument and the error behaviour are as for pgqa_paged_attention_decode.
 * The q_len x (num_q_heads / num_kv_heads) query rows of a (sequence, kv-head) share
 * every page read when they are at most 32 (the decode kernel); above that the prefill
 * kernel runs the call (block_size 16 only, else PGQA_EUNSUPPORTED; scale > 0).
 */
pgqa_status_t pgqa_paged_attention_decode_multi(
    void* out, float* lse, const void* q, int q_len, const void* k_cache, const void* v_cache,
    const int32_t* block_tables, int max_blocks_per_seq, const int32_t* context_lens,
    int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int num_blocks, int block_size,
    float scale, int cache_dtype, const float* k_scale, const float* v_scale, int max_context_len,
    void* workspace, size_t workspace_bytes, int* dev_status, void* stream);

/* Workspace bytes pgqa_paged_prefill_varlen needs (33024: the ticket counters the
 * CTAs take work items with, and the longest-first item tables each call rebuilds). */
size_t pgqa_prefill_workspace_size(int num_seqs, int num_q_heads, int max_seqlen);

/*
 * Causal variable-length prefill over the paged cache (the varlen call with
 * cumulative lengths, causal=True, returning out and lse, of the rkmt.cn
 * article, sec. 2.4; keys read through the block tables of sec. 3.1).
 * The prompt's K/V must already be in the cache (pgqa_kv_cache_write).
 *
 *   out           [T][num_q_heads][head_dim] bf16, written; T = cu_seqlens[num_seqs].
 *   lse           [T][num_q_heads] fp32, written; may be NULL.
 *   q             [T][num_q_heads][head_dim] bf16, read.
 *   num_tokens    T; must equal cu_seqlens[num_seqs] (checked on the device).
 *   cu_seqlens    [num_seqs + 1] int32, read: sequence i owns tokens
 *                 cu_seqlens[i] .. cu_seqlens[i+1]-1; the token at position p
 *                 of sequence i attends to keys 0..p of sequence i.
 *   max_seqlen    an upper bound on the sequence lengths (at most 262144).
 *   block_tables  [num_seqs][max_blocks_per_seq] int32, read.
 *   num_seqs      at most 4096.
 *   scale         must be > 0.
 *   workspace     device scratch of at least pgqa_prefill_workspace_size()
 *                 bytes, 16-byte aligned; its first 256 bytes ZERO-FILLED before
 *                 its first use (every call that completes leaves them zero).
 *                 Calls sharing a workspace must not overlap in time.
 * bf16 cache (an E4M3 one: pgqa_paged_prefill_varlen_e4m3); q/out/k_cache/v_cache
 * 16-byte aligned. Inconsistent cu_seqlens (negative lengths, a length above max_seqlen or beyond the block
 * table, a last entry other than num_tokens) are a device error (PGQA_EINVAL in
 * *dev_status); nothing is written for the sequences concerned.
 */
pgqa_status_t pgqa_paged_prefill_varlen(void* out, float* lse, const void* q, int num_tokens,
                                        const void* k_cache, const void* v_cache,
                                        const int32_t* block_tables, int max_blocks_per_seq,
                                        const int32_t* cu_seqlens, int num_seqs, int max_seqlen,
                                        int num_q_heads, int num_kv_heads, int head_dim,
                                        int num_blocks, int block_size, float scale,
                                        void* workspace, size_t workspace_bytes,
                                        int* dev_status, void* stream);

/*
 * Chunked prefill over a cached prefix: the varlen call of the rkmt.cn article,
 * sec. 2.4, with separate query and key lengths (its cu_seqlens_q / cu_seqlens_k),
 * keys read through the block tables of sec. 3.1. Sequence i's new tokens (its
 * chunk, cu_seqlens_q[i] .. cu_seqlens_q[i+1]-1, Lq of them) are the last Lq of the
 * Lk = seq_lens_k[i] tokens in its cache, so chunk position p attends to keys
 * 0 .. Lk-Lq+p (bottom-right causal alignment; Lk = Lq is
 * pgqa_paged_prefill_varlen). The chunk's own K/V must already be in the cache
 * (pgqa_kv_cache_write). Speculative verification (a few draft tokens per
 * sequence) is the case Lq = 2..6.
 *
 *   cu_seqlens_q  [num_seqs + 1] int32, read: the chunks in q / out / lse.
 *   seq_lens_k    [num_seqs] int32, read: Lk per sequence, Lq <= Lk <= max_seqlen_k.
 *   max_seqlen_q  an upper bound on the chunk lengths (at most 262144).
 *   max_seqlen_k  an upper bound on Lk (at most 2^26).
 * Every other argument, the workspace and the error behaviour are as for
 * pgqa_paged_prefill_varlen; a sequence with Lk < Lq, Lk above max_seqlen_k or
 * beyond its block table is a device error (PGQA_EINVAL).
 */
pgqa_status_t pgqa_paged_prefill_varlen_kv(void* out, float* lse, const void* q, int num_tokens,
                                           const void* k_cache, const void* v_cache,
                                           const int32_t* block_tables, int max_blocks_per_seq,
                                           const int32_t* cu_seqlens_q, const int32_t* seq_lens_k,
                                           int num_seqs, int max_seqlen_q, int max_seqlen_k,
                                           int num_q_heads, int num_kv_heads, int head_dim,
                                           int num_blocks, int block_size, float scale,
                                           void* workspace, size_t workspace_bytes,
                                           int* dev_status, void* stream);

/*
 * Prefill over an E4M3 cache: pgqa_paged_prefill_varlen_kv over a cache written by
 * pgqa_kv_cache_write with cache_dtype PGQA_DTYPE_E4M3 (the FP8 cache the rkmt.cn
 * article pairs with GQA, ch. 1; stored value = code * scale_h per kv-head).
 *   seq_lens_k    [num_seqs] int32 as for pgqa_paged_prefill_varlen_kv, or NULL for
 *                 no cached prefix (Lk = Lq; max_seqlen_k is then ignored).
 *   k_scale, v_scale  [num_kv_heads] fp32 device arrays, read; every entry must be
 *                 positive and finite (else PGQA_EINVAL in *dev_status).
 * Arithmetic: the codes are widened exactly to f16 and q is rounded to f16 (exact
 * for |q| in [2^-14, 65504]); scores and the output accumulate in fp32, P is
 * rounded to f16 for the P V product; out is rounded to bf16.
 * Every other argument, the workspace and the error behaviour are as for
 * pgqa_paged_prefill_varlen_kv.
 */
pgqa_status_t pgqa_paged_prefill_varlen_e4m3(
    void* out, float* lse, const void* q, int num_tokens, const void* k_cache,
    const void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
    const int32_t* cu_seqlens_q, const int32_t* seq_lens_k, int num_seqs, int max_seqlen_q,
    int max_seqlen_k, int num_q_heads, int num_kv_heads, int head_dim, int num_blocks,
    int block_size, float scale, const float* k_scale, const float* v_scale, void* workspace,
    size_t workspace_bytes, int* dev_status, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* PGQA_H */
