"""Prefill over an E4M3 cache on the GPU against the fp64 oracle.

The batch's K/V go into an E4M3 cache through the cache-write kernel (codes checked
bit for bit against the oracle's quantiser, per-kv-head scales amax / 448), then the
E4M3 prefill attends them. Small cases compare every row: whole sequences with
lengths on both sides of the tile (128) and page (16) edges, and chunks over cached
prefixes (speculative verification included), for every group size, head_dim 64 and
128. At full size (16 sequences, lengths uniform on [128, 2048], 32 query / 8 kv
heads, head_dim 128; and the cached-prefix batch) the oracle checks sampled rows.
A bad block id and a scale that is not positive are reported, not faulted."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import assert_attention_close, bits, dev

pytestmark = pytest.mark.gpu


class E4M3Run:
    def __init__(self, inp):
        self.inp = inp
        self.chunked = isinstance(inp, workloads.ChunkedPrefillInputs)
        kc, vc, ks, vs = workloads.e4m3_prefill_cache(inp)
        self.kc0, self.vc0, self.ks_host, self.vs_host = kc, vc, ks, vs
        self.kc, self.vc, self.ks, self.vs = dev(kc), dev(vc), dev(ks), dev(vs)
        self.q, self.bt = dev(inp.q), dev(inp.block_tables)
        if self.chunked:
            self.cu, self.lk = dev(inp.cu_seqlens_q), dev(inp.seq_lens_k)
            self.max_q, self.max_k = inp.max_seqlen_q, inp.max_seqlen_k
        else:
            self.cu, self.lk = dev(inp.cu_seqlens), None
            self.max_q, self.max_k = inp.max_seqlen, 0
        T, Hq, D = inp.q.shape
        self.out = torch.full((T, Hq, D), 5.0, dtype=torch.bfloat16, device="cuda")
        self.lse = torch.full((T, Hq), 5.0, dtype=torch.float32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.ws = torch.zeros(pgqa.prefill_workspace_size(inp.num_seqs, Hq, self.max_q),
                              dtype=torch.uint8, device="cuda")

    def write(self):
        pgqa.kv_cache_write(dev(self.inp.key), dev(self.inp.value), dev(self.inp.slot_mapping),
                            self.kc, self.vc, k_scale=self.ks, v_scale=self.vs,
                            dev_status=self.status)

    def prefill(self, out=None, lse=None):
        pgqa.paged_prefill_varlen_e4m3(self.out if out is None else out,
                                       self.lse if lse is None else lse, self.q, self.kc,
                                       self.vc, self.bt, self.cu, self.lk, self.max_q, self.max_k,
                                       self.inp.scale, self.ks, self.vs, workspace=self.ws,
                                       dev_status=self.status)

    def status_code(self):
        torch.cuda.synchronize()
        return int(self.status.item())

    def oracle_cache(self):
        return oracle.kv_cache_write(self.inp.key, self.inp.value, self.inp.slot_mapping,
                                     self.kc0, self.vc0, dtype=oracle.E4M3,
                                     k_scale=self.ks_host, v_scale=self.vs_host)

    def oracle_rows(self, kc, vc, rows=None):
        inp = self.inp
        if self.chunked:
            return oracle.paged_prefill_kv(inp.q, kc, vc, inp.block_tables, inp.cu_seqlens_q,
                                           inp.seq_lens_k, inp.scale, rows=rows,
                                           dtype=oracle.E4M3, k_scale=self.ks_host,
                                           v_scale=self.vs_host)
        return oracle.paged_prefill(inp.q, kc, vc, inp.block_tables, inp.cu_seqlens, inp.scale,
                                    rows=rows, dtype=oracle.E4M3, k_scale=self.ks_host,
                                    v_scale=self.vs_host)


def _run(inp):
    run = E4M3Run(inp)
    run.write()
    run.prefill()
    assert run.status_code() == 0
    kc, vc = run.oracle_cache()
    assert np.array_equal(bits(run.kc), kc) and np.array_equal(bits(run.vc), vc), "cache codes"
    return run, kc, vc


def _sample(cu, T, Hq, n, seed):
    g = np.random.default_rng(seed)
    rows = set()
    for i in range(len(cu) - 1):
        for t in (cu[i], cu[i + 1] - 1, cu[i] + 127, cu[i] + 128):
            if cu[i] <= t < cu[i + 1]:
                rows.add((t, int(g.integers(Hq))))
    while len(rows) < n:
        rows.add((int(g.integers(T)), int(g.integers(Hq))))
    return np.array(sorted(rows), np.int32)


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_whole_sequences_full_compare(G, D):
    lens = [1, 15, 16, 17, 127, 128, 129, 300, 64]
    nb = sum(-(-L // 16) for L in lens) + 8
    inp = workloads.make_prefill(lens, 2 * G, 2, D, nb, seed=400 + G + D)
    run, kc, vc = _run(inp)
    ref_out, ref_lse = run.oracle_rows(kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, f"e4m3 G={G} D={D}")


@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_chunks_full_compare(G, D):
    lens_q = [1, 5, 17, 127, 128, 129, 64]
    lens_k = [1, 300, 150, 130, 256, 400, 700]
    nb = sum(-(-L // 16) for L in lens_k) + 8
    inp = workloads.make_chunked_prefill(lens_k, lens_q, 2 * G, 2, D, nb, seed=420 + G + D)
    run, kc, vc = _run(inp)
    ref_out, ref_lse = run.oracle_rows(kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, f"e4m3 chunks G={G} D={D}")


def test_speculative_verification_full_compare():
    lens_k = [37, 256, 513, 1000, 64, 129]
    nb = sum(-(-L // 16) for L in lens_k) + 8
    inp = workloads.make_chunked_prefill(lens_k, [5] * len(lens_k), 32, 8, 128, nb, seed=440)
    run, kc, vc = _run(inp)
    ref_out, ref_lse = run.oracle_rows(kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, "e4m3 speculative verification")


def test_varlen_workload_sampled_rows():
    inp = workloads.varlen_prefill()
    run, kc, vc = _run(inp)
    T, Hq, _ = inp.q.shape
    rows = _sample(inp.cu_seqlens.tolist(), T, Hq, 1500, 5)
    ref_out, ref_lse = run.oracle_rows(kc, vc, rows=rows)
    t, h = rows[:, 0], rows[:, 1]
    assert_attention_close(run.out[t, h], run.lse[t, h], ref_out[t, h], ref_lse[t, h],
                           "e4m3 varlen prefill sampled rows")


def test_chunked_workload_sampled_rows():
    inp = workloads.chunked_prefill()
    run, kc, vc = _run(inp)
    T, Hq, _ = inp.q.shape
    rows = _sample(inp.cu_seqlens_q.tolist(), T, Hq, 800, 6)
    ref_out, ref_lse = run.oracle_rows(kc, vc, rows=rows)
    t, h = rows[:, 0], rows[:, 1]
    assert_attention_close(run.out[t, h], run.lse[t, h], ref_out[t, h], ref_lse[t, h],
                           "e4m3 chunked prefill sampled rows")


def test_repeat_calls_are_identical():
    lens = [700, 130, 5]
    nb = sum(-(-L // 16) for L in lens) + 8
    run, _, _ = _run(workloads.make_prefill(lens, 8, 2, 128, nb, seed=450))
    out2, lse2 = torch.zeros_like(run.out), torch.zeros_like(run.lse)
    run.prefill(out2, lse2)
    assert run.status_code() == 0
    assert torch.equal(out2, run.out) and torch.equal(lse2, run.lse)
    assert torch.all(run.ws[:256] == 0)


def test_bad_block_id_is_reported_not_faulted():
    lens = [200, 300]
    inp = workloads.make_prefill(lens, 4, 2, 128, 64, seed=460)
    run = E4M3Run(inp)
    run.write()
    torch.cuda.synchronize()
    run.bt[1, 3] = -1               # page 3 of sequence 1 (keys 48..63)
    run.prefill()
    assert run.status_code() == pgqa.EBADINDEX
    kc, vc = run.oracle_cache()
    ref_out, ref_lse = run.oracle_rows(kc, vc)
    a = lens[0]
    assert_attention_close(run.out[:a], run.lse[:a], ref_out[:a], ref_lse[:a])
    assert torch.all(run.out[a:] == 0) and torch.all(torch.isneginf(run.lse[a:]))


def test_nonpositive_scale_is_reported():
    inp = workloads.make_prefill([40, 7], 4, 2, 128, 16, seed=470)
    run = E4M3Run(inp)
    run.write()
    torch.cuda.synchronize()
    run.ks[1] = 0.0
    run.prefill()
    assert run.status_code() == pgqa.EINVAL


def test_grouped_rows_speculative_e4m3():
    lens_k = [37, 256, 513, 1000, 64, 129]
    nb = sum(-(-L // 16) for L in lens_k) + 8
    inp = workloads.make_chunked_prefill(lens_k, [5] * len(lens_k), 32, 8, 128, nb, seed=480)
    run, kc, vc = _run(inp)
    ref_out, ref_lse = run.oracle_rows(kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, "e4m3 grouped rows")
