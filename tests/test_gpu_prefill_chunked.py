"""Prefill over a cached prefix (chunked prefill, speculative verification) on the GPU
against the fp64 oracle.

Sequence i caches Lk tokens; its chunk is the last Lq of them, and chunk position p
attends to keys 0..Lk-Lq+p. Small cases are compared in full, with prefixes that are
not multiples of the 128-token tile (so the masked keys of a query tile spread over
two key tiles), chunks of 1..6 tokens (speculative verification) and chunks that
cross tile and page edges, for every group size. At full size the oracle checks
sampled rows (always including each chunk's first and last row). Properties: a
chunk's rows equal the same rows of a prefill over the whole sequence (two GPU
calls, within the tolerance), the last row equals a decode step over the whole
context, and Lk = Lq reproduces the varlen prefill bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import assert_attention_close, bits, dev

pytestmark = pytest.mark.gpu


class ChunkRun:
    def __init__(self, inp, max_seqlen_q=None, max_seqlen_k=None):
        self.inp = inp
        self.kc, self.vc = dev(inp.k_cache), dev(inp.v_cache)
        self.q = dev(inp.q)
        self.bt = dev(inp.block_tables)
        self.cu, self.lk = dev(inp.cu_seqlens_q), dev(inp.seq_lens_k)
        T, Hq, D = inp.q.shape
        self.out = torch.full((T, Hq, D), 5.0, dtype=torch.bfloat16, device="cuda")
        self.lse = torch.full((T, Hq), 5.0, dtype=torch.float32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.ws = torch.zeros(pgqa.prefill_workspace_size(inp.num_seqs, Hq, inp.max_seqlen_q),
                              dtype=torch.uint8, device="cuda")
        self.max_q = max_seqlen_q if max_seqlen_q is not None else inp.max_seqlen_q
        self.max_k = max_seqlen_k if max_seqlen_k is not None else inp.max_seqlen_k

    def write(self):
        pgqa.kv_cache_write(dev(self.inp.key), dev(self.inp.value), dev(self.inp.slot_mapping),
                            self.kc, self.vc, dev_status=self.status)

    def prefill(self):
        pgqa.paged_prefill_varlen_kv(self.out, self.lse, self.q, self.kc, self.vc, self.bt,
                                     self.cu, self.lk, self.max_q, self.max_k, self.inp.scale,
                                     workspace=self.ws, dev_status=self.status)

    def status_code(self):
        torch.cuda.synchronize()
        return int(self.status.item())


def oracle_cache(inp):
    return oracle.kv_cache_write(inp.key, inp.value, inp.slot_mapping, inp.k_cache, inp.v_cache)


def oracle_rows(inp, kc, vc, rows=None):
    return oracle.paged_prefill_kv(inp.q, kc, vc, inp.block_tables, inp.cu_seqlens_q,
                                   inp.seq_lens_k, inp.scale, rows=rows)


def _case(lens_k, lens_q, Hq, Hkv, D, seed):
    nb = sum(-(-L // 16) for L in lens_k) + 8
    inp = workloads.make_chunked_prefill(lens_k, lens_q, Hq, Hkv, D, nb, seed)
    run = ChunkRun(inp)
    run.write()
    run.prefill()
    assert run.status_code() == 0
    kc, vc = oracle_cache(inp)
    return inp, run, kc, vc


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_chunks_full_compare(G, D):
    # prefixes off the tile grid, chunks across tile and page edges, single tokens
    lens_q = [1, 2, 5, 6, 17, 127, 128, 129, 200, 64]
    lens_k = [1, 300, 133, 6, 150, 130, 256, 400, 333, 700]
    inp, run, kc, vc = _case(lens_k, lens_q, 2 * G, 2, D, seed=300 + G + D)
    ref_out, ref_lse = oracle_rows(inp, kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, f"G={G} D={D}")


@pytest.mark.parametrize("G", [1, 4])
def test_empty_chunks_in_the_batch(G):
    """Sequences with a cached prefix but no new token take no work and report
    nothing; the other chunks match the oracle (G = 4: the grouped-rows layout)."""
    inp, run, kc, vc = _case([40, 300, 17, 129, 5], [0, 5, 0, 3, 0], 2 * G, 2, 128,
                             seed=310 + G)
    ref_out, ref_lse = oracle_rows(inp, kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, f"empty chunks G={G}")


def test_speculative_verification_full_compare():
    lens_k = [37, 256, 513, 1000, 64, 129]
    inp, run, kc, vc = _case(lens_k, [5] * len(lens_k), 32, 8, 128, seed=320)
    ref_out, ref_lse = oracle_rows(inp, kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, "speculative verification")


@pytest.fixture(scope="module")
def chunked():
    inp = workloads.chunked_prefill()
    run = ChunkRun(inp)
    run.write()
    run.prefill()
    assert run.status_code() == 0
    kc, vc = oracle_cache(inp)
    return inp, run, kc, vc


def test_chunked_workload_cache_and_sampled_rows(chunked):
    inp, run, kc, vc = chunked
    assert np.array_equal(bits(run.kc), kc) and np.array_equal(bits(run.vc), vc)
    g = np.random.default_rng(3)
    T, Hq, _ = inp.q.shape
    rows = set()
    cu = inp.cu_seqlens_q.tolist()
    for i in range(len(cu) - 1):
        for t in (cu[i], cu[i + 1] - 1, cu[i] + 127, cu[i] + 128):
            if cu[i] <= t < cu[i + 1]:
                rows.add((t, int(g.integers(Hq))))
    while len(rows) < 1500:
        rows.add((int(g.integers(T)), int(g.integers(Hq))))
    rows = np.array(sorted(rows), np.int32)
    ref_out, ref_lse = oracle_rows(inp, kc, vc, rows=rows)
    t, h = rows[:, 0], rows[:, 1]
    assert_attention_close(run.out[t, h], run.lse[t, h], ref_out[t, h], ref_lse[t, h],
                           "chunked prefill sampled rows")


def test_chunk_rows_equal_whole_sequence_prefill():
    """Two GPU calls over the same cache: the whole sequences as one prefill, and only
    their last tokens as chunks; the chunks' rows agree within the tolerance."""
    lens = [700, 300, 129]
    chunk = [200, 57, 129]
    nb = sum(-(-L // 16) for L in lens) + 8
    inp = workloads.make_chunked_prefill(lens, lens, 8, 2, 128, nb, seed=330)
    full = ChunkRun(inp)
    full.write()
    full.prefill()
    assert full.status_code() == 0
    cuk = [0] + np.cumsum(lens).tolist()
    sel = torch.cat([torch.arange(cuk[i + 1] - n, cuk[i + 1]) for i, n in enumerate(chunk)])
    part = workloads.ChunkedPrefillInputs(
        q=inp.q[sel], key=inp.key, value=inp.value, slot_mapping=inp.slot_mapping,
        cu_seqlens_q=torch.tensor([0] + np.cumsum(chunk).tolist(), dtype=torch.int32),
        seq_lens_k=inp.seq_lens_k, block_tables=inp.block_tables, k_cache=inp.k_cache,
        v_cache=inp.v_cache, scale=inp.scale)
    run = ChunkRun(part)
    run.kc, run.vc = full.kc, full.vc
    run.prefill()
    assert run.status_code() == 0
    sel_d = sel.cuda()
    ref = full.out[sel_d].float().cpu().double().numpy()
    assert_attention_close(run.out, run.lse, ref, full.lse[sel_d].cpu().double().numpy(),
                           "chunk vs whole-sequence prefill")


def test_last_row_equals_decode():
    lens_k, lens_q = [900, 131, 40], [3, 130, 40]
    inp, run, kc, vc = _case(lens_k, lens_q, 16, 4, 128, seed=340)
    cu = inp.cu_seqlens_q.tolist()
    last = [cu[i + 1] - 1 for i in range(len(lens_k))]
    out = torch.empty((len(lens_k), 16, 128), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((len(lens_k), 16), dtype=torch.float32, device="cuda")
    ws = torch.zeros(pgqa.decode_workspace_size(len(lens_k), 16, 4, 128, max(lens_k)),
                     dtype=torch.uint8, device="cuda")
    pgqa.paged_attention_decode(out, lse, run.q[last].contiguous(), run.kc, run.vc, run.bt,
                                run.lk, inp.scale, max(lens_k), workspace=ws,
                                dev_status=run.status)
    assert run.status_code() == 0
    ref_o = out.float().cpu().double().numpy()
    ref_l = lse.cpu().double().numpy()
    assert_attention_close(run.out[last], run.lse[last], ref_o, ref_l, "chunk last row vs decode")


def test_without_prefix_matches_varlen_prefill_bitwise():
    lens = [300, 17, 128]
    nb = sum(-(-L // 16) for L in lens) + 8
    inp = workloads.make_chunked_prefill(lens, lens, 8, 2, 128, nb, seed=350)
    run = ChunkRun(inp)
    run.write()
    run.prefill()
    assert run.status_code() == 0
    out2 = torch.zeros_like(run.out)
    lse2 = torch.zeros_like(run.lse)
    ws = torch.zeros_like(run.ws)
    pgqa.paged_prefill_varlen(out2, lse2, run.q, run.kc, run.vc, run.bt, run.cu, max(lens),
                              inp.scale, workspace=ws, dev_status=run.status)
    assert run.status_code() == 0
    assert torch.equal(out2, run.out) and torch.equal(lse2, run.lse)


def test_key_length_shorter_than_chunk_is_reported():
    lens_k, lens_q = [100, 50], [20, 10]
    nb = sum(-(-L // 16) for L in lens_k) + 8
    inp = workloads.make_chunked_prefill(lens_k, lens_q, 4, 2, 128, nb, seed=360)
    inp.seq_lens_k[1] = 5                       # Lk < Lq
    run = ChunkRun(inp)
    run.write()
    run.prefill()
    assert run.status_code() == pgqa.EINVAL


@pytest.mark.parametrize("G,lens_q", [(4, [1, 5, 64, 17, 33, 2]), (8, [1, 6, 32, 9, 31, 2])])
def test_grouped_rows_layout(G, lens_q):
    """Chunks of at most 256/G tokens for groups of 4 or 8 take the grouped layout (a
    tile holds G/2 heads of every token of the chunk): every row against the oracle,
    chunk lengths up to the layout's limit, prefixes across tile edges."""
    lens_k = [1, 300, 64, 129, 700, 2]
    inp, run, kc, vc = _case(lens_k, lens_q, 2 * G, 2, 128, seed=370 + G)
    ref_out, ref_lse = oracle_rows(inp, kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, f"grouped rows G={G}")


@pytest.mark.parametrize("G", [4, 8])
def test_grouped_rows_whole_sequences(G):
    """The plain varlen prefill with every sequence within the grouped layout's limit."""
    lens = [1, 17, 256 // G, 5]
    nb = sum(-(-L // 16) for L in lens) + 8
    inp = workloads.make_chunked_prefill(lens, lens, 2 * G, 2, 64, nb, seed=380 + G)
    run = ChunkRun(inp)
    run.write()
    pgqa.paged_prefill_varlen(run.out, run.lse, run.q, run.kc, run.vc, run.bt, run.cu, max(lens),
                              inp.scale, workspace=run.ws, dev_status=run.status)
    assert run.status_code() == 0
    kc, vc = oracle_cache(inp)
    ref_out, ref_lse = oracle_rows(inp, kc, vc)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, f"grouped whole sequences G={G}")
