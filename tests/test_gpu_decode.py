"""Paged decode on the GPU against the fp64 oracle, element by element.

Covers the five workloads (tiny; Llama-3-8B; 70B bf16 and E4M3; prefix sharing),
each as one decode step (append the new token's K/V, then attend), plus ragged
and degenerate contexts, every group size the kernel takes, head_dim 64,
forced split counts, repeat calls (the split-merge counters reset themselves),
and device-detected bad indices."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import (DecodeRun, assert_attention_close, bits, oracle_cache_after_append,
                    oracle_decode)

pytestmark = pytest.mark.gpu


def _step_and_check(inp, max_context_len=None, what=""):
    run = DecodeRun(inp, max_context_len)
    run.append()
    run.decode()
    assert run.status_code() == 0
    kc, vc = oracle_cache_after_append(inp)
    assert np.array_equal(bits(run.kc), kc) and np.array_equal(bits(run.vc), vc), "append"
    ref_out, ref_lse = oracle_decode(inp, kc, vc)
    err = assert_attention_close(run.out, run.lse, ref_out, ref_lse, what or inp.name)
    return run, ref_out, ref_lse, err


@pytest.fixture(scope="module")
def llama8b():
    return workloads.llama3_8b_decode()


def test_tiny_decode():
    _step_and_check(workloads.tiny_decode())


def test_llama3_8b_decode(llama8b):
    _step_and_check(llama8b)


def test_70b_decode_bf16():
    _step_and_check(workloads.llama70b_decode())


def test_70b_decode_e4m3():
    _step_and_check(workloads.llama70b_decode(cache_dtype="e4m3"))


def test_prefix_sharing_decode():
    inp = workloads.prefix_sharing_decode()
    # the appended token lies past the shared prefix, so sharing stays copy-on-write safe
    assert all(L - 1 >= 4096 for L in inp.context_lens.tolist())
    _step_and_check(inp)


def test_repeat_calls_identical(llama8b):
    """The split-merge ticket counters must return to zero after every call."""
    run = DecodeRun(llama8b)
    run.decode()
    first = run.out.clone(), run.lse.clone()
    for _ in range(3):
        run.decode()
    assert run.status_code() == 0
    assert torch.equal(first[0], run.out) and torch.equal(first[1], run.lse)
    if run.ws is not None:
        nctr = llama8b.num_seqs * llama8b.num_kv_heads
        assert int(run.ws[: 4 * nctr].view(torch.int32).abs().sum()) == 0


@pytest.mark.parametrize("G", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_contexts_and_groups(G, D):
    lens = [1, 2, 15, 16, 17, 31, 32, 33, 127, 128, 129, 300, 1000]
    Hkv = 2
    inp = workloads.make_decode(lens, G * Hkv, Hkv, D, 256, seed=100 + G * 7 + D)
    _step_and_check(inp, what=f"G={G} D={D}")


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_contexts_e4m3(G, D):
    lens = [1, 7, 16, 17, 40, 257, 999]
    inp = workloads.make_decode(lens, G * 2, 2, D, 256, seed=200 + G + D, cache_dtype="e4m3")
    _step_and_check(inp, what=f"e4m3 G={G} D={D}")


@pytest.mark.parametrize("B", [193, 500])
@pytest.mark.parametrize("cache_dtype", ["bf16", "e4m3"])
def test_more_sequences_than_one_plan_pass(B, cache_dtype):
    """The kernel's range plan scans the context lengths 192 sequences at a time: with
    more, the unit holding a range's first page is found in a later pass."""
    g = np.random.default_rng(B)
    lens = [int(x) for x in g.integers(1, 400, size=B)]
    nb = sum(-(-L // 16) for L in lens) + 16
    inp = workloads.make_decode(lens, 8, 2, 128, nb, seed=B, cache_dtype=cache_dtype)
    _step_and_check(inp, what=f"B={B} {cache_dtype}")


@pytest.mark.parametrize("max_ctx_factor", [1, 2, 8])
def test_split_counts_agree(max_ctx_factor):
    """Inflating max_context_len changes the split plan, not the result."""
    lens = [130, 700, 2049, 64]
    inp = workloads.make_decode(lens, 8, 2, 128, 512, seed=300)
    _step_and_check(inp, max_context_len=inp.max_context_len * max_ctx_factor)


def test_single_key_returns_v_exactly():
    inp = workloads.make_decode([1, 1, 1], 8, 2, 128, 16, seed=400)
    run = DecodeRun(inp)
    run.decode()
    assert run.status_code() == 0
    G = 4
    for b in range(3):
        for hq in range(8):
            pbn = int(inp.block_tables[b, 0])
            assert torch.equal(run.out[b, hq].cpu(), inp.v_cache[pbn, hq // G, 0])
    ref_out, ref_lse = oracle_decode(inp)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse)


def test_empty_context():
    inp = workloads.make_decode([0, 20], 4, 2, 128, 16, seed=500)
    run = DecodeRun(inp)
    run.out.fill_(7)
    run.decode()
    assert run.status_code() == 0
    assert torch.all(run.out[0] == 0) and torch.all(torch.isneginf(run.lse[0]))
    ref_out, ref_lse = oracle_decode(inp)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse)


@pytest.mark.parametrize("bad", [-1, 10 ** 6])
def test_bad_block_id_is_reported_not_faulted(bad):
    lens = [200, 300, 50]
    inp = workloads.make_decode(lens, 8, 2, 128, 64, seed=600)
    inp.block_tables[1, 5] = bad
    run = DecodeRun(inp)
    run.decode()
    assert run.status_code() == pgqa.EBADINDEX
    assert torch.all(run.out[1] == 0) and torch.all(torch.isneginf(run.lse[1]))
    good = [0, 2]
    inp.block_tables[1, 5] = 0
    ref_out, ref_lse = oracle_decode(inp)
    assert_attention_close(run.out[good], run.lse[good], ref_out[good], ref_lse[good])


def test_context_longer_than_bound_is_reported():
    inp = workloads.make_decode([100, 40], 4, 2, 128, 32, seed=700)
    run = DecodeRun(inp, max_context_len=64)
    run.decode()
    assert run.status_code() == pgqa.EINVAL
    assert torch.all(run.out[0] == 0)
    ref_out, ref_lse = oracle_decode(inp)
    assert_attention_close(run.out[1:], run.lse[1:], ref_out[1:], ref_lse[1:])


def test_no_lse_output():
    inp = workloads.tiny_decode()
    run = DecodeRun(inp)
    pgqa.paged_attention_decode(run.out, None, run.q, run.kc, run.vc, run.bt, run.cl, inp.scale,
                                run.max_ctx, workspace=run.ws, dev_status=run.status)
    assert run.status_code() == 0
    ref_out, _ = oracle_decode(inp)
    assert_attention_close(run.out, None, ref_out, None)


def test_workspace_too_small_is_rejected():
    inp = workloads.make_decode([2000] * 4, 8, 2, 128, 600, seed=800)
    run = DecodeRun(inp)
    assert run.ws is not None
    with pytest.raises(pgqa.PgqaError) as e:
        pgqa.paged_attention_decode(run.out, run.lse, run.q, run.kc, run.vc, run.bt, run.cl,
                                    inp.scale, run.max_ctx, workspace=run.ws[:16])
    assert e.value.status == pgqa.ENOWORKSPACE
