"""The no-allocation decode entry point (collected last on purpose).

pgqa_paged_attention_decode_noalloc serves callers that cannot allocate device
memory -- e.g. an engine whose KV pool already fills the GPU, or a plugin whose
device memory belongs to a host framework's allocator -- by keeping the split-K
scratch in a fixed library-owned array. These tests call it through the C ABI
and check it against the regular entry point (which takes a caller-allocated
workspace), on two calls in a row, with the parity tolerances of the other
tests; and check that sizes beyond the array are refused without a launch."""
import ctypes

import pytest
import torch

import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import LSE_ATOL, OUT_ATOL, OUT_RTOL, DecodeRun

pytestmark = pytest.mark.gpu


def _noalloc(run, status=None):
    inp = run.inp
    B, Hq, D = inp.q.shape
    NB, Hkv, bs, _ = inp.k_cache.shape
    out = torch.full_like(run.out, 3.0)
    lse = torch.full_like(run.lse, 3.0)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = pgqa.lib.pgqa_paged_attention_decode_noalloc(
        P(out), P(lse), P(run.q), P(run.kc), P(run.vc), P(run.bt), inp.block_tables.shape[1],
        P(run.cl), B, Hq, Hkv, D, NB, bs, inp.scale, pgqa._cache_dtype(run.kc), P(run.ks),
        P(run.vs), run.max_ctx, P(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out, lse


def _close(a_out, a_lse, b_out, b_lse):
    diff = (a_out.float() - b_out.float()).abs()
    assert torch.all(diff <= OUT_ATOL + OUT_RTOL * b_out.float().abs()), float(diff.max())
    assert torch.all((a_lse - b_lse).abs() <= LSE_ATOL)


@pytest.mark.parametrize("cache_dtype", ["bf16", "e4m3"])
def test_noalloc_matches_workspace_entry_point_twice(cache_dtype):
    if cache_dtype == "bf16":
        inp = workloads.llama3_8b_decode()
    else:
        inp = workloads.make_decode([3000, 1500, 4096, 17] * 4, 32, 4, 128, 4096, seed=11,
                                    cache_dtype="e4m3")
    run = DecodeRun(inp)
    need = pgqa.decode_workspace_size(inp.num_seqs, inp.num_q_heads, inp.num_kv_heads,
                                      inp.head_dim, inp.max_context_len)
    assert 0 < need <= pgqa.NOALLOC_SCRATCH_BYTES  # the scratch path is exercised
    run.decode()                                   # regular entry point, caller workspace
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    for _ in range(2):
        rc, out, lse = _noalloc(run, status)
        assert rc == pgqa.OK, pgqa.status_string(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        _close(out, lse, run.out, run.lse)


def test_noalloc_rejects_sizes_beyond_its_scratch():
    # grow the batch until the workspace (one ticket per (sequence, kv-head) plus the
    # partial slots) exceeds the fixed array; the inputs are valid -- empty contexts,
    # so a launch would only write zeros -- but no launch must happen
    Hq, Hkv, D = 8, 8, 64
    B = 1 << 14
    while pgqa.decode_workspace_size(B, Hq, Hkv, D, 16) <= pgqa.NOALLOC_SCRATCH_BYTES:
        B *= 2
        assert B < 1 << 22
    kc = torch.zeros((1, Hkv, 16, D), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((B, 1), dtype=torch.int32, device="cuda")
    inp = workloads.DecodeInputs(q=torch.zeros((B, Hq, D), dtype=torch.bfloat16, device="cuda"),
                                 k_cache=kc, v_cache=kc, block_tables=bt,
                                 context_lens=torch.zeros((B,), dtype=torch.int32, device="cuda"),
                                 scale=0.1)
    run = DecodeRun(inp)
    rc, out, _ = _noalloc(run)
    torch.cuda.synchronize()
    assert rc == pgqa.ENOWORKSPACE
    assert torch.all(out == 3.0)  # nothing was launched
