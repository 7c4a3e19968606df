"""fp64 CPU oracle for paged grouped-query attention -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package. The CUDA library never imports it, and
it imports nothing from the CUDA library: the two share only the seeded input
generators in ``workloads``.

The arithmetic lives in ``oracle.c`` (plain C, IEEE double, loops in the order
of the definitions); this module is argument marshalling with numpy.
Inputs are numpy arrays (or CPU torch tensors, converted here):
bf16 data is passed as its uint16 bit pattern, E4M3 data as uint8 codes.
"""
import contextlib
import ctypes
import os

import numpy as np

from . import build as _build

BF16 = 0
E4M3 = 1


def _bind(path):
    lib = ctypes.CDLL(path)
    P = ctypes.c_void_p
    I = ctypes.c_int
    I64 = ctypes.c_int64
    D = ctypes.c_double
    lib.oracle_bf16_to_f64.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_f64.restype = D
    lib.oracle_e4m3_to_f64.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_f64.restype = D
    lib.oracle_e4m3_from_f32.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_from_f32.restype = ctypes.c_uint8
    lib.oracle_kv_cache_write.argtypes = [P, P, P, I, I, I, P, P, I, I, I, P, P]
    lib.oracle_kv_cache_write.restype = I
    lib.oracle_gather_kv.argtypes = [P, P, I, P, P, P, I, I, I, I, I, I, I, P, P]
    lib.oracle_gather_kv.restype = I
    lib.oracle_paged_decode.argtypes = [P, P, P, I, P, P, P, I, P, I, I, I, I, I, I, D, P, P, I]
    lib.oracle_paged_decode.restype = I
    lib.oracle_paged_prefill.argtypes = [P, P, P, I, P, P, P, I, P, I, I, I, I, I, I, D, P, I64,
                                         P, P, I]
    lib.oracle_paged_prefill.restype = I
    lib.oracle_paged_prefill_kv.argtypes = [P, P, P, I, P, P, P, I, P, P, I, I, I, I, I, I, D, P,
                                            I64, P, P, I]
    lib.oracle_paged_prefill_kv.restype = I
    lib.oracle_paged_decode_window.argtypes = [P, P, P, I, P, P, P, I, P, I, I, I, I, I, I, D, I,
                                               P, P, I]
    lib.oracle_paged_decode_window.restype = I
    lib.oracle_dense_row.argtypes = [P, P, P, I, I, D, P, P]
    lib.oracle_dense_row.restype = None
    lib.oracle_has_openmp.argtypes = []
    lib.oracle_has_openmp.restype = I
    return lib


_default = None


def _load():
    global _default
    if _default is None:
        _default = _bind(_build.build())
    return _default


@contextlib.contextmanager
def use_library(path):
    """Run the calls inside the ``with`` block against another build of the
    oracle (the planted-mistake tests load mutated copies this way)."""
    global _default
    old = _load()
    _default = _bind(path)
    try:
        yield
    finally:
        _default = old


def _np(x, dtype=None):
    """numpy view of a CPU tensor / array; bf16 tensors become uint16 bit patterns."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if x.dtype == torch.bfloat16:
                x = x.view(torch.int16).numpy().view(np.uint16)
            elif x.dtype == getattr(torch, "float8_e4m3fn", None):
                x = x.view(torch.uint8).numpy()
            else:
                x = x.numpy()
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if dtype is not None and x.dtype != dtype:
        raise TypeError(f"expected {np.dtype(dtype)}, got {x.dtype}")
    return x


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _check(rc, what):
    if rc != 0:
        raise ValueError(f"oracle {what} returned {rc}")


def default_threads():
    return os.cpu_count() or 1


def has_openmp() -> bool:
    return bool(_load().oracle_has_openmp())


def bf16_to_f64(bits: int) -> float:
    return _load().oracle_bf16_to_f64(bits)


def e4m3_to_f64(code: int) -> float:
    return _load().oracle_e4m3_to_f64(code)


def e4m3_from_f32(x: float) -> int:
    return int(_load().oracle_e4m3_from_f32(x))


def kv_cache_write(key, value, slot_mapping, k_cache, v_cache, dtype=BF16, k_scale=None,
                   v_scale=None):
    """Scatter key/value [T, Hkv, D] (bf16) into copies of k_cache/v_cache
    [NB, Hkv, bs, D] by slot; returns the new (k_cache, v_cache) numpy arrays."""
    key, value = _np(key, np.uint16), _np(value, np.uint16)
    slots = _np(slot_mapping, np.int64)
    elem = np.uint16 if dtype == BF16 else np.uint8
    kc, vc = _np(k_cache, elem).copy(), _np(v_cache, elem).copy()
    ks = None if k_scale is None else _np(k_scale, np.float32)
    vs = None if v_scale is None else _np(v_scale, np.float32)
    T, Hkv, D = key.shape
    NB, _, bs, _ = kc.shape
    rc = _load().oracle_kv_cache_write(_ptr(key), _ptr(value), _ptr(slots), T, Hkv, D, _ptr(kc),
                                       _ptr(vc), NB, bs, dtype, _ptr(ks), _ptr(vs))
    _check(rc, "kv_cache_write")
    return kc, vc


def gather_kv(k_cache, v_cache, block_table_row, L, h, dtype=BF16, k_scale=None, v_scale=None):
    """Contiguous (K, V) [L, D] float64 of kv-head h for one sequence."""
    elem = np.uint16 if dtype == BF16 else np.uint8
    kc, vc = _np(k_cache, elem), _np(v_cache, elem)
    bt = _np(block_table_row, np.int32)
    ks = None if k_scale is None else _np(k_scale, np.float32)
    vs = None if v_scale is None else _np(v_scale, np.float32)
    NB, Hkv, bs, D = kc.shape
    K = np.zeros((max(L, 1), D), np.float64)
    V = np.zeros((max(L, 1), D), np.float64)
    rc = _load().oracle_gather_kv(_ptr(kc), _ptr(vc), dtype, _ptr(ks), _ptr(vs), _ptr(bt),
                                  bt.shape[-1], L, h, Hkv, D, NB, bs, _ptr(K), _ptr(V))
    _check(rc, "gather_kv")
    return K[:L], V[:L]


def paged_decode(q, k_cache, v_cache, block_tables, context_lens, scale, dtype=BF16,
                 k_scale=None, v_scale=None, threads=None):
    """Decode attention: returns (out [B, Hq, D] float64, lse [B, Hq] float64)."""
    q = _np(q, np.uint16)
    elem = np.uint16 if dtype == BF16 else np.uint8
    kc, vc = _np(k_cache, elem), _np(v_cache, elem)
    bt, cl = _np(block_tables, np.int32), _np(context_lens, np.int32)
    ks = None if k_scale is None else _np(k_scale, np.float32)
    vs = None if v_scale is None else _np(v_scale, np.float32)
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = kc.shape
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = _load().oracle_paged_decode(_ptr(q), _ptr(kc), _ptr(vc), dtype, _ptr(ks), _ptr(vs),
                                     _ptr(bt), bt.shape[1], _ptr(cl), B, Hq, Hkv, D, NB, bs,
                                     float(scale), _ptr(out), _ptr(lse),
                                     threads or default_threads())
    _check(rc, "paged_decode")
    return out, lse


def paged_prefill(q, k_cache, v_cache, block_tables, cu_seqlens, scale, rows=None,
                  dtype=BF16, k_scale=None, v_scale=None, threads=None):
    """Causal varlen prefill. rows: optional int array [n, 2] of (token, q_head).
    Returns (out [T, Hq, D], lse [T, Hq]) float64; rows not computed stay NaN."""
    q = _np(q, np.uint16)
    elem = np.uint16 if dtype == BF16 else np.uint8
    kc, vc = _np(k_cache, elem), _np(v_cache, elem)
    bt, cu = _np(block_tables, np.int32), _np(cu_seqlens, np.int32)
    ks = None if k_scale is None else _np(k_scale, np.float32)
    vs = None if v_scale is None else _np(v_scale, np.float32)
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = kc.shape
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, np.int32).reshape(-1, 2))
    n_rows = 0 if r is None else r.shape[0]
    out = np.full((T, Hq, D), np.nan, np.float64)
    lse = np.full((T, Hq), np.nan, np.float64)
    rc = _load().oracle_paged_prefill(_ptr(q), _ptr(kc), _ptr(vc), dtype, _ptr(ks), _ptr(vs),
                                      _ptr(bt), bt.shape[1], _ptr(cu), len(cu) - 1, Hq, Hkv, D, NB,
                                      bs, float(scale), _ptr(r), n_rows, _ptr(out), _ptr(lse),
                                      threads or default_threads())
    _check(rc, "paged_prefill")
    return out, lse


def paged_decode_window(q, k_cache, v_cache, block_tables, context_lens, scale, window,
                        dtype=BF16, k_scale=None, v_scale=None, threads=None):
    """Sliding-window decode: each context's last `window` keys only. Returns
    (out [B, Hq, D] float64, lse [B, Hq] float64)."""
    q = _np(q, np.uint16)
    elem = np.uint16 if dtype == BF16 else np.uint8
    kc, vc = _np(k_cache, elem), _np(v_cache, elem)
    bt, cl = _np(block_tables, np.int32), _np(context_lens, np.int32)
    ks = None if k_scale is None else _np(k_scale, np.float32)
    vs = None if v_scale is None else _np(v_scale, np.float32)
    B, Hq, D = q.shape
    NB, Hkv, bs, _ = kc.shape
    out = np.zeros((B, Hq, D), np.float64)
    lse = np.zeros((B, Hq), np.float64)
    rc = _load().oracle_paged_decode_window(_ptr(q), _ptr(kc), _ptr(vc), dtype, _ptr(ks),
                                            _ptr(vs), _ptr(bt), bt.shape[1], _ptr(cl), B, Hq, Hkv,
                                            D, NB, bs, float(scale), int(window), _ptr(out),
                                            _ptr(lse), threads or default_threads())
    _check(rc, "paged_decode_window")
    return out, lse


def paged_prefill_kv(q, k_cache, v_cache, block_tables, cu_seqlens_q, seq_lens_k, scale,
                     rows=None, dtype=BF16, k_scale=None, v_scale=None, threads=None):
    """Chunked prefill over a cached prefix: sequence i's chunk (cu_seqlens_q) is the
    last Lq of its seq_lens_k[i] cached tokens; query i of a chunk sees keys
    0..Lk-Lq+i. rows: optional int array [n, 2] of (token, q_head).
    Returns (out [T, Hq, D], lse [T, Hq]) float64; rows not computed stay NaN."""
    q = _np(q, np.uint16)
    elem = np.uint16 if dtype == BF16 else np.uint8
    kc, vc = _np(k_cache, elem), _np(v_cache, elem)
    bt, cu = _np(block_tables, np.int32), _np(cu_seqlens_q, np.int32)
    lk = _np(seq_lens_k, np.int32)
    ks = None if k_scale is None else _np(k_scale, np.float32)
    vs = None if v_scale is None else _np(v_scale, np.float32)
    T, Hq, D = q.shape
    NB, Hkv, bs, _ = kc.shape
    r = None if rows is None else np.ascontiguousarray(np.asarray(rows, np.int32).reshape(-1, 2))
    n_rows = 0 if r is None else r.shape[0]
    out = np.full((T, Hq, D), np.nan, np.float64)
    lse = np.full((T, Hq), np.nan, np.float64)
    rc = _load().oracle_paged_prefill_kv(_ptr(q), _ptr(kc), _ptr(vc), dtype, _ptr(ks), _ptr(vs),
                                         _ptr(bt), bt.shape[1], _ptr(cu), _ptr(lk), len(cu) - 1,
                                         Hq, Hkv, D, NB, bs, float(scale), _ptr(r), n_rows,
                                         _ptr(out), _ptr(lse), threads or default_threads())
    _check(rc, "paged_prefill_kv")
    return out, lse


def dense_row(q_row, K, V, scale):
    """Attention of one bf16 query row [D] over contiguous float64 K, V [L, D]."""
    q_row = _np(q_row, np.uint16)
    K = np.ascontiguousarray(K, np.float64)
    V = np.ascontiguousarray(V, np.float64)
    L, D = K.shape
    out = np.zeros(D, np.float64)
    lse = ctypes.c_double()
    _load().oracle_dense_row(_ptr(q_row), _ptr(K), _ptr(V), L, D, float(scale), _ptr(out),
                             ctypes.byref(lse))
    return out, lse.value
