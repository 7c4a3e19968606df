"""The no-allocation decode entry point (collected last on purpose).

pgqa_paged_attention_decode_noalloc serves callers that cannot allocate device
memory -- e.g. an engine whose KV pool already fills the GPU, or a plugin whose
device memory belongs to a host framework's allocator -- by keeping the split-K
scratch in a fixed library-owned array. These tests call it through the C ABI
and check it against the regular entry point (which takes a caller-allocated
workspace) on two calls in a row: both run the same kernel on the same grid and
split, so the results must be bit-identical (which also shows that the counter
clearing leaves no state behind). They also check that invalid arguments and
sizes beyond the array are refused with nothing enqueued, and, in a fresh
process, that once the per-device set-up is done the calls allocate nothing."""
import ctypes
import os
import subprocess
import sys
import textwrap

import pytest
import torch

import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import DecodeRun

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _noalloc(run, status=None, num_q_heads=None):
    inp = run.inp
    B, Hq, D = inp.q.shape
    NB, Hkv, bs, _ = inp.k_cache.shape
    out = torch.full_like(run.out, 3.0)
    lse = torch.full_like(run.lse, 3.0)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    rc = pgqa.lib.pgqa_paged_attention_decode_noalloc(
        P(out), P(lse), P(run.q), P(run.kc), P(run.vc), P(run.bt), inp.block_tables.shape[1],
        P(run.cl), B, Hq if num_q_heads is None else num_q_heads, Hkv, D, NB, bs, inp.scale,
        pgqa._cache_dtype(run.kc), P(run.ks), P(run.vs), run.max_ctx, P(status),
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    return rc, out, lse


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
        assert torch.equal(out, run.out) and torch.equal(lse, run.lse)


def test_noalloc_invalid_arguments_enqueue_nothing():
    """A call the host checks refuse (here a group of 16 query heads per kv-head, above
    the supported 8) returns its error and enqueues nothing: out keeps its fill, and the
    next valid call still gives the regular entry point's result bit for bit."""
    inp = workloads.tiny_decode()
    run = DecodeRun(inp)
    run.decode()
    rc, out, lse = _noalloc(run, num_q_heads=16 * inp.num_kv_heads)
    torch.cuda.synchronize()
    assert rc == pgqa.EUNSUPPORTED
    assert torch.all(out == 3.0) and torch.all(lse == 3.0)
    rc, out, lse = _noalloc(run)
    torch.cuda.synchronize()
    assert rc == pgqa.OK
    assert torch.equal(out, run.out) and torch.equal(lse, run.lse)


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


# Run in a fresh process with lazy module loading: every input is allocated first, then
# the set-up call (num_seqs = 0) is made and free device memory is read around it and
# around a series of real calls at several batch sizes and both cache types.
_FRESH = textwrap.dedent("""
    import ctypes, sys
    sys.path[:0] = [{root!r}, {tests!r}]
    import torch
    import paged_kv_gqa_10_gb300 as pgqa
    import workloads
    from parity import DecodeRun
    runs = [DecodeRun(workloads.llama3_8b_decode()), DecodeRun(workloads.tiny_decode()),
            DecodeRun(workloads.make_decode([700, 33, 2048] * 3, 32, 4, 128, 2048, seed=5,
                                            cache_dtype="e4m3"))]
    outs = [(torch.empty_like(r.out), torch.empty_like(r.lse)) for r in runs]
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    lib = pgqa.lib
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    free0 = torch.cuda.mem_get_info()[0]
    rc = lib.pgqa_paged_attention_decode_noalloc(None, None, None, None, None, None, 0, None,
                                                 0, 32, 8, 128, 1, 16, 0.1, 0, None, None, 0,
                                                 None, None)
    assert rc == 0, rc
    torch.cuda.synchronize()
    free1 = torch.cuda.mem_get_info()[0]
    for rep in range(3):
        for r, (o, l) in zip(runs, outs):
            inp = r.inp
            B, Hq, D = inp.q.shape
            NB, Hkv, bs, _ = inp.k_cache.shape
            rc = lib.pgqa_paged_attention_decode_noalloc(
                P(o), P(l), P(r.q), P(r.kc), P(r.vc), P(r.bt), inp.block_tables.shape[1],
                P(r.cl), B, Hq, Hkv, D, NB, bs, inp.scale, pgqa._cache_dtype(r.kc), P(r.ks),
                P(r.vs), r.max_ctx, P(status), None)
            assert rc == 0, rc
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    free2 = torch.cuda.mem_get_info()[0]
    print("SETUP", free0 - free1, "CALLS", free1 - free2)
""")


def test_noalloc_allocates_nothing_after_setup():
    script = _FRESH.format(root=ROOT, tests=os.path.join(ROOT, "tests"))
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    r = subprocess.run([sys.executable, "-c", script], capture_output=True, text=True, env=env,
                       timeout=600)
    assert r.returncode == 0, r.stdout + r.stderr
    line = [s for s in r.stdout.splitlines() if s.startswith("SETUP")][-1].split()
    setup, calls = int(line[1]), int(line[3])
    # the set-up call loads the array (and the decode kernels) on the device ...
    assert setup >= pgqa.NOALLOC_SCRATCH_BYTES, line
    # ... and no later call takes any device memory
    assert calls == 0, line
