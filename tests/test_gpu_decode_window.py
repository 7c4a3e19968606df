"""Sliding-window paged decode on the GPU against the fp64 oracle.

A context of L keys attends to its last W keys only. Ragged contexts around page
(16) and window edges, windows that are not multiples of a page (the first page
read is cut inside), a window of one key (the output is that key's V row exactly),
windows at least the context (plain decode, bit for bit), every group size, head_dim
64 and 128 and the E4M3 cache; one 70B-shaped batch at full size."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import DecodeRun, assert_attention_close, bits, oracle_cache_after_append

pytestmark = pytest.mark.gpu


def _window_step(inp, window, what=""):
    run = DecodeRun(inp)
    run.append()
    pgqa.paged_attention_decode_window(run.out, run.lse, run.q, run.kc, run.vc, run.bt, run.cl,
                                       inp.scale, window, run.max_ctx, k_scale=run.ks,
                                       v_scale=run.vs, workspace=run.ws, dev_status=run.status)
    assert run.status_code() == 0
    kc, vc = oracle_cache_after_append(inp)
    assert np.array_equal(bits(run.kc), kc) and np.array_equal(bits(run.vc), vc), "append"
    dt = oracle.BF16 if inp.cache_dtype == "bf16" else oracle.E4M3
    ref_out, ref_lse = oracle.paged_decode_window(inp.q, kc, vc, inp.block_tables,
                                                  inp.context_lens, inp.scale, window, dtype=dt,
                                                  k_scale=inp.k_scale, v_scale=inp.v_scale)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, what or f"window {window}")
    return run


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
@pytest.mark.parametrize("window", [1, 7, 16, 37, 128, 500])
def test_ragged_contexts_windows(G, D, window):
    lens = [1, 2, 15, 16, 17, 33, 128, 129, 300, 1000, 4000]
    Hkv = 2
    inp = workloads.make_decode(lens, G * Hkv, Hkv, D, 512, seed=500 + G + D + window)
    _window_step(inp, window, f"G={G} D={D} W={window}")


@pytest.mark.parametrize("window", [5, 100])
@pytest.mark.parametrize("D", [64, 128])
def test_e4m3_windows(window, D):
    lens = [1, 7, 16, 17, 40, 257, 999]
    inp = workloads.make_decode(lens, 8, 2, D, 256, seed=600 + window + D, cache_dtype="e4m3")
    _window_step(inp, window, f"e4m3 W={window} D={D}")


def test_window_of_one_key_returns_its_value_exactly():
    inp = workloads.make_decode([40, 1, 17], 8, 2, 128, 64, seed=610)
    run = _window_step(inp, 1)
    kc, vc = oracle_cache_after_append(inp)
    G = 4
    for b, L in enumerate(inp.context_lens.tolist()):
        for hq in range(8):
            assert torch.equal(run.out[b, hq].cpu(), inp.step_value[b, hq // G]), (b, hq)


def test_window_covering_the_context_is_plain_decode():
    inp = workloads.make_decode([100, 513, 7], 8, 2, 128, 128, seed=620)
    run = _window_step(inp, 100000)
    out2, lse2 = torch.zeros_like(run.out), torch.zeros_like(run.lse)
    ws2 = torch.zeros_like(run.ws)
    pgqa.paged_attention_decode(out2, lse2, run.q, run.kc, run.vc, run.bt, run.cl, inp.scale,
                                run.max_ctx, workspace=ws2, dev_status=run.status)
    assert run.status_code() == 0
    assert torch.equal(out2, run.out) and torch.equal(lse2, run.lse)


def test_70b_shaped_window_2048():
    _window_step(workloads.llama70b_decode(), 2048, "70B W=2048")


def test_zero_window_is_rejected():
    inp = workloads.tiny_decode()
    run = DecodeRun(inp)
    with pytest.raises(pgqa.PgqaError):
        pgqa.paged_attention_decode_window(run.out, run.lse, run.q, run.kc, run.vc, run.bt, run.cl,
                                           inp.scale, 0, run.max_ctx, workspace=run.ws,
                                           dev_status=run.status)
