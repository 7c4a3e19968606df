"""paged_kv_gqa_10_gb300 -- paged grouped-query attention for GB300 (sm_103a).

A thin ctypes binding over ``libpgqa.so`` (the C ABI declared in
``include/pgqa.h``). Every function here only marshals arguments: tensors
become device pointers and sizes, the current torch CUDA stream becomes the
launch stream, and a non-zero status becomes a ``PgqaError``. All computation
runs in the library's CUDA kernels; there is no other path. The first call
raises ImportError if the library has not been built
(``python -m paged_kv_gqa_10_gb300.build``).

Functions (same names as the C entry points, without the ``pgqa_`` prefix):
  kv_cache_write, paged_kv_gather,
  paged_attention_decode, paged_attention_decode_append,
  paged_attention_decode_window, paged_attention_decode_noalloc,
  paged_attention_decode_multi,
  paged_prefill_varlen, paged_prefill_varlen_kv, paged_prefill_varlen_e4m3,
  decode_workspace_size, decode_multi_workspace_size, decode_grid_size,
  prefill_workspace_size, kv_cache_bytes,
  set_decode_wait_limit_ns, status_string, abi_version.
"""
import ctypes
import os

import torch

__all__ = [
    "PgqaError", "BF16", "E4M3", "kv_cache_write", "paged_kv_gather",
    "paged_attention_decode", "paged_attention_decode_append", "paged_attention_decode_window",
    "paged_attention_decode_noalloc", "paged_attention_decode_multi", "paged_prefill_varlen",
    "paged_prefill_varlen_kv",
    "paged_prefill_varlen_e4m3", "decode_workspace_size", "decode_multi_workspace_size",
    "decode_grid_size",
    "prefill_workspace_size", "kv_cache_bytes", "set_decode_wait_limit_ns", "status_string",
    "abi_version",
    "library_path", "lib",
]

BF16 = 0
E4M3 = 1
ABI_VERSION = 1
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024
MAX_DECODE_TOKENS = 8

OK, EINVAL, EUNSUPPORTED, ENOWORKSPACE, ECUDA, EBADINDEX, ETIMEOUT = 0, -1, -2, -3, -4, -5, -6

_HERE = os.path.dirname(os.path.abspath(__file__))
_LIB_PATH = os.path.join(_HERE, "libpgqa.so")


class PgqaError(RuntimeError):
    def __init__(self, status, what):
        self.status = status
        super().__init__(f"{what}: {status_string(status)} ({status})")


def _load():
    if not os.path.exists(_LIB_PATH):
        raise ImportError(
            f"{_LIB_PATH} is missing: build it with `python -m paged_kv_gqa_10_gb300.build` "
            "(there is no fallback implementation)")
    lib = ctypes.CDLL(_LIB_PATH)
    P, I, I64, F, SZ = (ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_float,
                        ctypes.c_size_t)
    sig = {
        "pgqa_abi_version": ([], I),
        "pgqa_status_string": ([I], ctypes.c_char_p),
        "pgqa_set_decode_wait_limit_ns": ([ctypes.c_uint64], None),
        "pgqa_kv_cache_bytes": ([I, I64, I, I, I], I64),
        "pgqa_kv_cache_write": ([P, P, P, I, I, I, P, P, I, I, I, P, P, P, P], I),
        "pgqa_paged_kv_gather": ([P, P, I, P, I, P, I, I, I, I, I, I, P, P, P, P], I),
        "pgqa_decode_grid_size": ([I, I, I], I),
        "pgqa_decode_workspace_size": ([I, I, I, I, I], SZ),
        "pgqa_paged_attention_decode": ([P, P, P, P, P, P, I, P, I, I, I, I, I, I, F, I, P, P,
                                         I, P, SZ, P, P], I),
        "pgqa_paged_attention_decode_window": ([P, P, P, P, P, P, I, P, I, I, I, I, I, I, F, I,
                                                I, P, P, I, P, SZ, P, P], I),
        "pgqa_paged_attention_decode_append": ([P, P, P, P, P, P, P, P, I, P, I, I, I, I, I,
                                                I, F, I, P, P, I, P, SZ, P, P], I),
        "pgqa_paged_attention_decode_noalloc": ([P, P, P, P, P, P, I, P, I, I, I, I, I, I, F,
                                                 I, P, P, I, P, P], I),
        "pgqa_decode_multi_workspace_size": ([I, I, I, I, I], SZ),
        "pgqa_paged_attention_decode_multi": ([P, P, P, I, P, P, P, I, P, I, I, I, I, I, I, F,
                                               I, P, P, I, P, SZ, P, P], I),
        "pgqa_prefill_workspace_size": ([I, I, I], SZ),
        "pgqa_paged_prefill_varlen": ([P, P, P, I, P, P, P, I, P, I, I, I, I, I, I, I, F, P,
                                       SZ, P, P], I),
        "pgqa_paged_prefill_varlen_kv": ([P, P, P, I, P, P, P, I, P, P, I, I, I, I, I, I, I, I,
                                          F, P, SZ, P, P], I),
        "pgqa_paged_prefill_varlen_e4m3": ([P, P, P, I, P, P, P, I, P, P, I, I, I, I, I, I, I,
                                            I, F, P, P, P, SZ, P, P], I),
    }
    for name, (args, res) in sig.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    if lib.pgqa_abi_version() != ABI_VERSION:
        raise ImportError("libpgqa ABI version mismatch; rebuild the library")
    return lib


_lib = None


def __getattr__(name):
    if name == "lib":
        return _handle()
    raise AttributeError(name)


def _handle():
    """The loaded ctypes library (loaded on first use)."""
    global _lib
    if _lib is None:
        _lib = _load()
    return _lib


def library_path() -> str:
    return _LIB_PATH


def abi_version() -> int:
    return _handle().pgqa_abi_version()


def status_string(status: int) -> str:
    return _handle().pgqa_status_string(status).decode()


def set_decode_wait_limit_ns(ns: int) -> None:
    """Limit, in nanoseconds, of the decode kernels' bounded waits for the launches that
    follow (0 restores the 2 s default); a failure-detection testing aid, see
    pgqa_set_decode_wait_limit_ns in include/pgqa.h."""
    if int(ns) < 0:
        raise ValueError("ns must be >= 0")
    _handle().pgqa_set_decode_wait_limit_ns(int(ns))


# ------------------------------------------------------------------ helpers

def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t, name, dtype=None):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise TypeError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} has dtype {t.dtype}, expected {dtype}")
    return t


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _cache_dtype(cache):
    if cache.dtype == torch.bfloat16:
        return BF16
    if cache.dtype in (torch.uint8, getattr(torch, "float8_e4m3fn", torch.uint8)):
        return E4M3
    raise TypeError(f"cache dtype {cache.dtype} is neither bfloat16 nor E4M3 bytes")


def _check(rc, what):
    if rc != OK:
        raise PgqaError(rc, what)


# ------------------------------------------------------------------- C ABI

def kv_cache_bytes(num_layers, tokens, num_kv_heads, head_dim, cache_dtype=BF16) -> int:
    return _handle().pgqa_kv_cache_bytes(num_layers, tokens, num_kv_heads, head_dim, cache_dtype)


def decode_grid_size(num_sms, head_dim=128, cache_dtype=BF16):
    """CTAs the decode kernel launches on a device with num_sms SMs."""
    n = _handle().pgqa_decode_grid_size(num_sms, head_dim, cache_dtype)
    if n < 0:
        raise PgqaError(n, "decode_grid_size")
    return n


def decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim, max_context_len) -> int:
    return _handle().pgqa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                                max_context_len)


def decode_multi_workspace_size(num_seqs, q_len, num_q_heads, num_kv_heads, head_dim) -> int:
    return int(_handle().pgqa_decode_multi_workspace_size(num_seqs, q_len, num_q_heads,
                                                          num_kv_heads, head_dim))


def prefill_workspace_size(num_seqs, num_q_heads, max_seqlen) -> int:
    return _handle().pgqa_prefill_workspace_size(num_seqs, num_q_heads, max_seqlen)


def kv_cache_write(key, value, slot_mapping, k_cache, v_cache, k_scale=None, v_scale=None,
                   dev_status=None, stream=None):
    """key/value [T, Hkv, D] bf16; slot_mapping [T] int64; caches [NB, Hkv, bs, D]."""
    _dev(key, "key", torch.bfloat16)
    _dev(value, "value", torch.bfloat16)
    _dev(slot_mapping, "slot_mapping", torch.int64)
    _dev(k_cache, "k_cache")
    _dev(v_cache, "v_cache")
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    _dev(dev_status, "dev_status", torch.int32)
    T, Hkv, D = key.shape
    NB, _, bs, _ = k_cache.shape
    rc = _handle().pgqa_kv_cache_write(_ptr(key), _ptr(value), _ptr(slot_mapping), T, Hkv, D,
                                       _ptr(k_cache), _ptr(v_cache), NB, bs,
                                       _cache_dtype(k_cache), _ptr(k_scale), _ptr(v_scale),
                                       _ptr(dev_status), _stream(stream))
    _check(rc, "kv_cache_write")


def paged_kv_gather(k_cache, v_cache, block_tables, context_lens, max_context_len, k_out, v_out,
                    dev_status=None, stream=None):
    """k_out/v_out [B, Hkv, max_context_len, D] in the cache dtype."""
    for t, n in ((k_cache, "k_cache"), (v_cache, "v_cache"), (k_out, "k_out"), (v_out, "v_out")):
        _dev(t, n)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    _dev(dev_status, "dev_status", torch.int32)
    NB, Hkv, bs, D = k_cache.shape
    B = context_lens.shape[0]
    rc = _handle().pgqa_paged_kv_gather(_ptr(k_cache), _ptr(v_cache), _cache_dtype(k_cache),
                                        _ptr(block_tables), block_tables.shape[1],
                                        _ptr(context_lens), B, Hkv, D, NB, bs, max_context_len,
                                        _ptr(k_out), _ptr(v_out), _ptr(dev_status),
                                        _stream(stream))
    _check(rc, "paged_kv_gather")


def paged_attention_decode(out, lse, q, k_cache, v_cache, block_tables, context_lens, scale,
                           max_context_len, k_scale=None, v_scale=None, workspace=None,
                           dev_status=None, stream=None):
    """out [B, Hq, D] bf16 and lse [B, Hq] fp32 (or None) are written.
    workspace: a zero-initialised uint8 CUDA tensor of at least
    decode_workspace_size(...) bytes."""
    _dev(out, "out", torch.bfloat16)
    _dev(lse, "lse", torch.float32)
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache")
    _dev(v_cache, "v_cache")
    _dev(block_tables, "block_tables", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    _dev(workspace, "workspace")
    _dev(dev_status, "dev_status", torch.int32)
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _handle().pgqa_paged_attention_decode(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, NB, bs, float(scale),
        _cache_dtype(k_cache), _ptr(k_scale), _ptr(v_scale), int(max_context_len),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(rc, "paged_attention_decode")


def paged_attention_decode_append(out, lse, q, key, value, k_cache, v_cache, block_tables,
                                  context_lens, scale, max_context_len, k_scale=None,
                                  v_scale=None, workspace=None, dev_status=None, stream=None):
    """One decode step with the append fused in: key/value [B, Hkv, D] bf16 (the new
    token of every sequence) go to position context_lens[b] - 1 of each cache, then
    attention over the whole context. Other arguments as for paged_attention_decode."""
    _dev(out, "out", torch.bfloat16)
    _dev(lse, "lse", torch.float32)
    _dev(q, "q", torch.bfloat16)
    _dev(key, "key", torch.bfloat16)
    _dev(value, "value", torch.bfloat16)
    _dev(k_cache, "k_cache")
    _dev(v_cache, "v_cache")
    _dev(block_tables, "block_tables", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    _dev(workspace, "workspace")
    _dev(dev_status, "dev_status", torch.int32)
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _handle().pgqa_paged_attention_decode_append(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(key), _ptr(value), _ptr(k_cache), _ptr(v_cache),
        _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, NB, bs,
        float(scale), _cache_dtype(k_cache), _ptr(k_scale), _ptr(v_scale), int(max_context_len),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(rc, "paged_attention_decode_append")


def paged_attention_decode_window(out, lse, q, k_cache, v_cache, block_tables, context_lens,
                                  scale, window, max_context_len, k_scale=None, v_scale=None,
                                  workspace=None, dev_status=None, stream=None):
    """Sliding-window decode: each context's last `window` keys only. Arguments as for
    paged_attention_decode."""
    _dev(out, "out", torch.bfloat16)
    _dev(lse, "lse", torch.float32)
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache")
    _dev(v_cache, "v_cache")
    _dev(block_tables, "block_tables", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    _dev(workspace, "workspace")
    _dev(dev_status, "dev_status", torch.int32)
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _handle().pgqa_paged_attention_decode_window(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, NB, bs, float(scale),
        int(window), _cache_dtype(k_cache), _ptr(k_scale), _ptr(v_scale), int(max_context_len),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(rc, "paged_attention_decode_window")


def paged_attention_decode_noalloc(out, lse, q, k_cache, v_cache, block_tables, context_lens,
                                   scale, max_context_len, k_scale=None, v_scale=None,
                                   dev_status=None, stream=None):
    """paged_attention_decode for callers that cannot allocate device memory: the
    split-K scratch is a fixed 8 MiB array owned by the library (see
    pgqa_paged_attention_decode_noalloc in include/pgqa.h). The first call on a device
    loads that array and the decode kernels there (make it before filling the device's
    memory; the C function called with num_seqs = 0 does only that). Calls that overlap
    on the GPU race on that array."""
    _dev(out, "out", torch.bfloat16)
    _dev(lse, "lse", torch.float32)
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache")
    _dev(v_cache, "v_cache")
    _dev(block_tables, "block_tables", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    _dev(dev_status, "dev_status", torch.int32)
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    rc = _handle().pgqa_paged_attention_decode_noalloc(
        _ptr(out), _ptr(lse), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, NB, bs, float(scale),
        _cache_dtype(k_cache), _ptr(k_scale), _ptr(v_scale), int(max_context_len),
        _ptr(dev_status), _stream(stream))
    _check(rc, "paged_attention_decode_noalloc")


def paged_attention_decode_multi(out, lse, q, k_cache, v_cache, block_tables, context_lens,
                                 scale, max_context_len, k_scale=None, v_scale=None,
                                 workspace=None, dev_status=None, stream=None):
    """Multi-token decode (speculative verification): q and out [B, q_len, Hq, D] bf16,
    lse [B, q_len, Hq] fp32 (or None); token t of sequence b attends keys
    0 .. context_lens[b] - q_len + t."""
    _dev(out, "out", torch.bfloat16)
    _dev(lse, "lse", torch.float32)
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache")
    _dev(v_cache, "v_cache")
    _dev(block_tables, "block_tables", torch.int32)
    _dev(context_lens, "context_lens", torch.int32)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    _dev(workspace, "workspace")
    _dev(dev_status, "dev_status", torch.int32)
    B, T, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _handle().pgqa_paged_attention_decode_multi(
        _ptr(out), _ptr(lse), _ptr(q), T, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(context_lens), B, Hq, Hkv, D, NB, bs, float(scale),
        _cache_dtype(k_cache), _ptr(k_scale), _ptr(v_scale), int(max_context_len),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(rc, "paged_attention_decode_multi")


def paged_prefill_varlen(out, lse, q, k_cache, v_cache, block_tables, cu_seqlens, max_seqlen,
                         scale, workspace=None, dev_status=None, stream=None):
    """out [T, Hq, D] bf16 and lse [T, Hq] fp32 (or None) are written."""
    _dev(out, "out", torch.bfloat16)
    _dev(lse, "lse", torch.float32)
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache", torch.bfloat16)
    _dev(v_cache, "v_cache", torch.bfloat16)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(cu_seqlens, "cu_seqlens", torch.int32)
    _dev(workspace, "workspace")
    _dev(dev_status, "dev_status", torch.int32)
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    S = cu_seqlens.shape[0] - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _handle().pgqa_paged_prefill_varlen(
        _ptr(out), _ptr(lse), _ptr(q), T, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(cu_seqlens), S, int(max_seqlen), Hq, Hkv, D, NB, bs,
        float(scale), _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(rc, "paged_prefill_varlen")


def paged_prefill_varlen_kv(out, lse, q, k_cache, v_cache, block_tables, cu_seqlens_q, seq_lens_k,
                            max_seqlen_q, max_seqlen_k, scale, workspace=None, dev_status=None,
                            stream=None):
    """Prefill over a cached prefix: each sequence's chunk (cu_seqlens_q) is the last
    Lq of its seq_lens_k cached tokens. out [T, Hq, D] bf16 and lse [T, Hq] fp32 (or
    None) are written."""
    _dev(out, "out", torch.bfloat16)
    _dev(lse, "lse", torch.float32)
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache", torch.bfloat16)
    _dev(v_cache, "v_cache", torch.bfloat16)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _dev(seq_lens_k, "seq_lens_k", torch.int32)
    _dev(workspace, "workspace")
    _dev(dev_status, "dev_status", torch.int32)
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    S = cu_seqlens_q.shape[0] - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _handle().pgqa_paged_prefill_varlen_kv(
        _ptr(out), _ptr(lse), _ptr(q), T, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(cu_seqlens_q), _ptr(seq_lens_k), S, int(max_seqlen_q),
        int(max_seqlen_k), Hq, Hkv, D, NB, bs, float(scale), _ptr(workspace), ws_bytes,
        _ptr(dev_status), _stream(stream))
    _check(rc, "paged_prefill_varlen_kv")


def paged_prefill_varlen_e4m3(out, lse, q, k_cache, v_cache, block_tables, cu_seqlens_q,
                              seq_lens_k, max_seqlen_q, max_seqlen_k, scale, k_scale, v_scale,
                              workspace=None, dev_status=None, stream=None):
    """Prefill over an E4M3 cache (uint8 codes, per-kv-head k_scale / v_scale [Hkv]
    fp32). seq_lens_k None: no cached prefix (whole-sequence causal prefill, and
    max_seqlen_k is ignored); else as paged_prefill_varlen_kv."""
    _dev(out, "out", torch.bfloat16)
    _dev(lse, "lse", torch.float32)
    _dev(q, "q", torch.bfloat16)
    _dev(k_cache, "k_cache", torch.uint8)
    _dev(v_cache, "v_cache", torch.uint8)
    _dev(block_tables, "block_tables", torch.int32)
    _dev(cu_seqlens_q, "cu_seqlens_q", torch.int32)
    _dev(seq_lens_k, "seq_lens_k", torch.int32)
    _dev(k_scale, "k_scale", torch.float32)
    _dev(v_scale, "v_scale", torch.float32)
    _dev(workspace, "workspace")
    _dev(dev_status, "dev_status", torch.int32)
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = k_cache.shape
    S = cu_seqlens_q.shape[0] - 1
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    rc = _handle().pgqa_paged_prefill_varlen_e4m3(
        _ptr(out), _ptr(lse), _ptr(q), T, _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
        block_tables.shape[1], _ptr(cu_seqlens_q), _ptr(seq_lens_k), S, int(max_seqlen_q),
        int(max_seqlen_k), Hq, Hkv, D, NB, bs, float(scale), _ptr(k_scale), _ptr(v_scale),
        _ptr(workspace), ws_bytes, _ptr(dev_status), _stream(stream))
    _check(rc, "paged_prefill_varlen_e4m3")
