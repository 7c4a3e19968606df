"""Multi-token paged decode (speculative verification) on the GPU against the fp64 oracle.

pgqa_paged_attention_decode_multi takes q_len new tokens per sequence, already written
into the cache: token t of a sequence with L cached tokens attends keys 0 .. L - q_len + t.
The oracle is the chunked-prefill one (each sequence's chunk is its last q_len tokens).
Small cases are compared in full for q_len 1-8, every group size, head_dim 64 and 128,
bf16 and E4M3 caches and 8/16/32-token blocks, with contexts that end on and off page
edges and contexts equal to q_len: up to 8 query rows per (sequence, kv-head) run the
decode kernel as a plain decode does, up to 32 its row-split form, and more run on the
prefill kernel; the same comparisons cover all three.
Also: repeat calls are bit-identical (the split-merge counters reset themselves), empty
and too-short contexts, and the full speculative-verification batch on sampled rows."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import assert_attention_close, dev

pytestmark = pytest.mark.gpu


class MultiRun:
    """A speculative-verification batch on the GPU: the cache written with every token
    (drafts included), then one multi-token decode call."""

    def __init__(self, lens_k, q_len, Hq, Hkv, D, seed, block_size=16, e4m3=False):
        nb = sum(-(-L // block_size) for L in lens_k) + 8
        self.inp = inp = workloads.make_chunked_prefill(lens_k, [min(q_len, L) for L in lens_k],
                                                        Hq, Hkv, D, nb, seed,
                                                        block_size=block_size)
        self.q_len, self.e4m3 = q_len, e4m3
        B = len(lens_k)
        if e4m3:
            kc, vc, ks, vs = workloads.e4m3_prefill_cache(inp)
            self.kc0, self.vc0, self.ks0, self.vs0 = kc, vc, ks, vs
        else:
            self.kc0, self.vc0, self.ks0, self.vs0 = inp.k_cache, inp.v_cache, None, None
        self.kc, self.vc = dev(self.kc0), dev(self.vc0)
        self.ks, self.vs = dev(self.ks0), dev(self.vs0)
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        pgqa.kv_cache_write(dev(inp.key), dev(inp.value), dev(inp.slot_mapping), self.kc, self.vc,
                            k_scale=self.ks, v_scale=self.vs, dev_status=self.status)
        # q: the chunks of q_len tokens (a sequence shorter than q_len is padded; such a
        # sequence is an error case the tests check separately)
        T, _, _ = inp.q.shape
        self.q = torch.zeros((B, q_len, Hq, D), dtype=torch.bfloat16, device="cuda")
        cu = inp.cu_seqlens_q.tolist()
        for b in range(B):
            n = cu[b + 1] - cu[b]
            self.q[b, q_len - n:] = dev(inp.q[cu[b]:cu[b + 1]])
        self.bt = dev(inp.block_tables)
        self.cl = dev(inp.seq_lens_k)
        self.out = torch.full((B, q_len, Hq, D), 5.0, dtype=torch.bfloat16, device="cuda")
        self.lse = torch.full((B, q_len, Hq), 5.0, dtype=torch.float32, device="cuda")
        n = pgqa.decode_multi_workspace_size(B, q_len, Hq, Hkv, D)
        self.ws = torch.zeros(max(n, 256), dtype=torch.uint8, device="cuda")
        self.max_ctx = max(lens_k)

    def decode(self):
        pgqa.paged_attention_decode_multi(self.out, self.lse, self.q, self.kc, self.vc, self.bt,
                                          self.cl, self.inp.scale, self.max_ctx,
                                          k_scale=self.ks, v_scale=self.vs, workspace=self.ws,
                                          dev_status=self.status)

    def status_code(self):
        torch.cuda.synchronize()
        return int(self.status.item())

    def reference(self):
        inp = self.inp
        dt = oracle.E4M3 if self.e4m3 else oracle.BF16
        kc, vc = oracle.kv_cache_write(inp.key, inp.value, inp.slot_mapping, self.kc0, self.vc0,
                                       dtype=dt, k_scale=self.ks0, v_scale=self.vs0)
        return oracle.paged_prefill_kv(inp.q, kc, vc, inp.block_tables, inp.cu_seqlens_q,
                                       inp.seq_lens_k, inp.scale, dtype=dt, k_scale=self.ks0,
                                       v_scale=self.vs0)

    def compare(self, what):
        ref_out, ref_lse = self.reference()
        B, q_len, Hq, D = self.out.shape
        assert_attention_close(self.out.view(B * q_len, Hq, D), self.lse.view(B * q_len, Hq),
                               ref_out, ref_lse, what)


LENS = [8, 16, 17, 31, 32, 33, 100, 257, 640, 1000]


@pytest.mark.parametrize("q_len", [1, 2, 3, 5, 6, 8])
@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_multi_token_full_compare(q_len, G, D):
    Hkv = 2
    run = MultiRun(LENS, q_len, G * Hkv, Hkv, D, seed=400 + 10 * q_len + G + D)
    run.decode()
    assert run.status_code() == 0
    run.compare(f"q_len={q_len} G={G} D={D}")


@pytest.mark.parametrize("q_len", [2, 5, 6])
@pytest.mark.parametrize("G", [1, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_multi_token_e4m3(q_len, G, D):
    Hkv = 2
    run = MultiRun(LENS, q_len, G * Hkv, Hkv, D, seed=500 + 10 * q_len + G + D, e4m3=True)
    run.decode()
    assert run.status_code() == 0
    run.compare(f"E4M3 q_len={q_len} G={G} D={D}")


@pytest.mark.parametrize("bs", [8, 32])
@pytest.mark.parametrize("q_len,G", [(5, 4), (3, 8), (8, 2)])
def test_multi_token_block_sizes(bs, q_len, G):
    run = MultiRun(LENS, q_len, 2 * G, 2, 128, seed=600 + bs + q_len + G, block_size=bs)
    run.decode()
    assert run.status_code() == 0
    run.compare(f"block {bs} q_len={q_len} G={G}")


def test_more_rows_than_the_decode_kernel_needs_16_token_blocks():
    run = MultiRun(LENS, 5, 16, 2, 128, seed=650, block_size=32)  # 5 x 8 = 40 rows
    with pytest.raises(pgqa.PgqaError) as e:
        run.decode()
    assert e.value.status == pgqa.EUNSUPPORTED


def test_repeat_calls_identical_and_counters_reset():
    run = MultiRun([300, 1000, 77, 4096, 512] * 4, 5, 32, 8, 128, seed=660)
    run.decode()
    first = run.out.clone(), run.lse.clone()
    for _ in range(3):
        run.decode()
    assert run.status_code() == 0
    assert torch.equal(first[0], run.out) and torch.equal(first[1], run.lse)
    nctr = 20 * 8  # a ticket per unit
    assert int(run.ws[: 4 * nctr].view(torch.int32).abs().sum()) == 0
    run.compare("repeat calls")


@pytest.mark.parametrize("q_len,G", [(2, 4), (5, 4)])
def test_unit_parts_where_a_draft_sees_no_key(q_len, G):
    """Contexts of 33 tokens: a unit is 3 pages and the last holds key 32 alone, which
    the earlier drafts do not attend. The stream-K ranges (at least 8 pages) cut units,
    so some thread block's part of a unit is that last page only, where those rows see
    no key: its partial must be zero with lse -inf, not NaN (both the plain scheme, 8
    rows, and the row-split form, 20 rows)."""
    run = MultiRun([33] * 300, q_len, 2 * G, 2, 128, seed=680 + q_len)
    run.decode()
    assert run.status_code() == 0
    run.compare(f"parts without keys q_len={q_len} G={G}")


def test_empty_and_too_short_contexts():
    """A context of 0 gives out = 0 and lse = -inf for all its tokens; a context shorter
    than q_len is a device error for that sequence (PGQA_EINVAL), written the same way;
    the other sequences are unaffected."""
    q_len = 4
    run = MultiRun([40, 300, 129], q_len, 8, 2, 128, seed=670)
    ref_out, ref_lse = run.reference()
    cl = run.cl.clone()
    run.cl[0] = 0
    run.cl[2] = 3
    run.decode()
    assert run.status_code() == pgqa.EINVAL
    for b in (0, 2):
        assert torch.all(run.out[b] == 0) and torch.all(torch.isinf(run.lse[b]))
    B, _, Hq, D = run.out.shape
    got = run.out[1].view(q_len, Hq, D)
    assert_attention_close(got, run.lse[1], ref_out[q_len:2 * q_len], ref_lse[q_len:2 * q_len],
                           "the valid sequence")
    run.cl.copy_(cl)


def test_speculative_verification_batch_sampled_rows():
    """The bench's speculative-verification batch (64 sequences, contexts U[256, 1024], 5
    tokens each, 32/8 heads, head_dim 128) against the oracle on sampled rows, always
    including every sequence's first and last token."""
    inp = workloads.speculative_verify()
    B = inp.num_seqs
    lens = inp.seq_lens_k.tolist()
    run = MultiRun(lens, 5, 32, 8, 128, seed=8)
    # the workload's own draws (same seed path) for the inputs
    run.inp = inp
    kc, vc = dev(inp.k_cache), dev(inp.v_cache)
    pgqa.kv_cache_write(dev(inp.key), dev(inp.value), dev(inp.slot_mapping), kc, vc,
                        dev_status=run.status)
    run.kc, run.vc, run.kc0, run.vc0 = kc, vc, inp.k_cache, inp.v_cache
    run.q = dev(inp.q).view(B, 5, 32, 128)
    run.bt, run.cl = dev(inp.block_tables), dev(inp.seq_lens_k)
    run.decode()
    assert run.status_code() == 0
    g = np.random.default_rng(5)
    rows = set()
    for b in range(B):
        rows.add((5 * b, int(g.integers(32))))
        rows.add((5 * b + 4, int(g.integers(32))))
    while len(rows) < 600:
        rows.add((int(g.integers(5 * B)), int(g.integers(32))))
    rows = np.array(sorted(rows), np.int32)
    okc, ovc = oracle.kv_cache_write(inp.key, inp.value, inp.slot_mapping, inp.k_cache,
                                     inp.v_cache)
    ref_out, ref_lse = oracle.paged_prefill_kv(inp.q, okc, ovc, inp.block_tables,
                                               inp.cu_seqlens_q, inp.seq_lens_k, inp.scale,
                                               rows=rows)
    t, h = rows[:, 0], rows[:, 1]
    out = run.out.view(5 * B, 32, 128)
    lse = run.lse.view(5 * B, 32)
    assert_attention_close(out[t, h], lse[t, h], ref_out[t, h], ref_lse[t, h], "spec batch")
