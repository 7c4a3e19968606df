"""Paged decode with 8- and 32-token blocks on the GPU against the fp64 oracle.

The kernel works on 16-token pages: a 32-token block holds two of them, a 16-token
page spans two 8-token blocks (two independent block ids). Ragged contexts around
8-, 16- and 32-token edges, every group size, head_dim 64 and 128, the E4M3 cache,
with and without a sliding window, and a bad block id in the second 8-token half of
a page, which is reported, not faulted."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import (DecodeRun, assert_attention_close, bits, oracle_cache_after_append,
                    oracle_decode)

pytestmark = pytest.mark.gpu

LENS = [1, 7, 8, 9, 15, 16, 17, 31, 32, 33, 100, 257, 1000]


def _step(inp, window=None, what=""):
    run = DecodeRun(inp)
    run.append()
    if window is None:
        run.decode()
    else:
        pgqa.paged_attention_decode_window(run.out, run.lse, run.q, run.kc, run.vc, run.bt,
                                           run.cl, inp.scale, window, run.max_ctx,
                                           k_scale=run.ks, v_scale=run.vs, workspace=run.ws,
                                           dev_status=run.status)
    assert run.status_code() == 0
    kc, vc = oracle_cache_after_append(inp)
    assert np.array_equal(bits(run.kc), kc) and np.array_equal(bits(run.vc), vc), "append"
    if window is None:
        ref_out, ref_lse = oracle_decode(inp, kc, vc)
    else:
        dt = oracle.BF16 if inp.cache_dtype == "bf16" else oracle.E4M3
        ref_out, ref_lse = oracle.paged_decode_window(inp.q, kc, vc, inp.block_tables,
                                                      inp.context_lens, inp.scale, window,
                                                      dtype=dt, k_scale=inp.k_scale,
                                                      v_scale=inp.v_scale)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, what)
    return run


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_block_sizes_ragged(bs, G, D):
    inp = workloads.make_decode(LENS, G * 2, 2, D, 1024, seed=700 + bs + G + D, block_size=bs)
    _step(inp, what=f"bs={bs} G={G} D={D}")


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("D", [64, 128])
def test_block_sizes_e4m3(bs, D):
    inp = workloads.make_decode(LENS, 8, 2, D, 1024, seed=720 + bs + D, cache_dtype="e4m3",
                                block_size=bs)
    _step(inp, what=f"e4m3 bs={bs} D={D}")


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("window", [5, 40])
def test_block_sizes_with_window(bs, window):
    inp = workloads.make_decode(LENS, 8, 2, 128, 1024, seed=730 + bs + window, block_size=bs)
    _step(inp, window=window, what=f"bs={bs} W={window}")


def test_block8_bad_id_in_second_half_is_reported():
    inp = workloads.make_decode([100, 40], 8, 2, 128, 64, seed=740, block_size=8)
    run = DecodeRun(inp)
    run.append()
    torch.cuda.synchronize()
    run.bt[0, 3] = -1                           # block 3 = keys 24..31: page 1's second half
    run.decode()
    assert run.status_code() == pgqa.EBADINDEX
    kc, vc = oracle_cache_after_append(inp)
    ref_out, ref_lse = oracle_decode(inp, kc, vc)
    # sequence 1 is untouched; sequence 0 is written as out = 0, lse = -inf
    assert_attention_close(run.out[1:], run.lse[1:], ref_out[1:], ref_lse[1:])
    assert torch.all(run.out[0] == 0) and torch.all(torch.isneginf(run.lse[0]))


def test_block_size_64_is_unsupported():
    inp = workloads.make_decode([40], 4, 2, 128, 16, seed=750, block_size=64)
    run = DecodeRun(inp)
    with pytest.raises(pgqa.PgqaError):
        run.decode()
