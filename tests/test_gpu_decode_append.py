"""One decode step with the append fused in, on the GPU.

The fused call writes each sequence's new token at position L-1 and attends the whole
context in one launch. Checked: the caches bit for bit against the oracle's cache
write with the step's slot mapping, out / lse against the oracle's decode of that
cache, and bit-identity with the two-call path (cache write, then decode) on the same
inputs, over ragged contexts (one key, page and block edges), every group size,
head_dim 64 and 128, block sizes 8, 16 and 32, the E4M3 cache and the full
Llama-3-8B-shaped batch. A bad block id at position L-1 is reported and nothing is
written for it."""
import numpy as np
import pytest
import torch

import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import (DecodeRun, assert_attention_close, bits, dev, oracle_cache_after_append,
                    oracle_decode)

pytestmark = pytest.mark.gpu

LENS = [1, 2, 7, 8, 9, 15, 16, 17, 31, 32, 33, 100, 257, 1000]


def fused(run):
    inp = run.inp
    pgqa.paged_attention_decode_append(run.out, run.lse, run.q, dev(inp.step_key),
                                       dev(inp.step_value), run.kc, run.vc, run.bt, run.cl,
                                       inp.scale, run.max_ctx, k_scale=run.ks, v_scale=run.vs,
                                       workspace=run.ws, dev_status=run.status)


def _check(inp, what):
    run = DecodeRun(inp)
    fused(run)
    assert run.status_code() == 0
    kc, vc = oracle_cache_after_append(inp)
    assert np.array_equal(bits(run.kc), kc) and np.array_equal(bits(run.vc), vc), "cache"
    ref_out, ref_lse = oracle_decode(inp, kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, what)
    # the two-call path on a fresh copy gives the same bits
    two = DecodeRun(inp)
    two.append()
    two.decode()
    assert two.status_code() == 0
    assert torch.equal(two.out, run.out) and torch.equal(two.lse, run.lse), "fused vs two calls"
    assert np.array_equal(bits(two.kc), bits(run.kc)) and np.array_equal(bits(two.vc), bits(run.vc))
    return run


@pytest.mark.parametrize("bs", [8, 16, 32])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_contexts(bs, G, D):
    inp = workloads.make_decode(LENS, G * 2, 2, D, 1024, seed=800 + bs + G + D, block_size=bs)
    _check(inp, f"fused append bs={bs} G={G} D={D}")


@pytest.mark.parametrize("bs", [8, 16, 32])
def test_e4m3(bs):
    inp = workloads.make_decode(LENS, 8, 2, 128, 1024, seed=830 + bs, cache_dtype="e4m3",
                                block_size=bs)
    _check(inp, f"fused append e4m3 bs={bs}")


def test_llama3_8b_batch():
    _check(workloads.llama3_8b_decode(), "fused append, Llama-3-8B batch")


def test_bad_block_at_the_new_position_is_reported():
    inp = workloads.make_decode([100, 40], 8, 2, 128, 64, seed=850)
    run = DecodeRun(inp)
    before_k, before_v = run.kc.clone(), run.vc.clone()
    run.bt[0, (100 - 1) // 16] = -1            # the block holding key 99
    fused(run)
    assert run.status_code() == pgqa.EBADINDEX
    kc, vc = oracle_cache_after_append(inp)
    ref_out, ref_lse = oracle_decode(inp, kc, vc)
    assert_attention_close(run.out[1:], run.lse[1:], ref_out[1:], ref_lse[1:])
    assert torch.all(run.out[0] == 0) and torch.all(torch.isneginf(run.lse[0]))
    # sequence 1's row is written; sequence 0's block is not a valid one: nothing else
    # changed
    s1 = int(inp.step_slots[1])
    blk, row = s1 // 16, s1 % 16
    changed = (run.kc.view(torch.int16) != before_k.view(torch.int16)).nonzero()
    assert changed.numel() > 0 and torch.all(changed[:, 0] == blk) and torch.all(changed[:, 2] == row)


def test_missing_rows_are_rejected():
    inp = workloads.tiny_decode()
    run = DecodeRun(inp)
    with pytest.raises(pgqa.PgqaError):
        pgqa.paged_attention_decode_append(run.out, run.lse, run.q, None, None, run.kc, run.vc,
                                           run.bt, run.cl, inp.scale, run.max_ctx,
                                           workspace=run.ws, dev_status=run.status)
