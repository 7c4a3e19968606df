"""Causal varlen paged prefill on the GPU against the fp64 oracle.

The full workload (16 sequences, lengths uniform on [128, 2048], 32 query / 8 kv
heads, head_dim 128) is written into the paged cache by the GPU kernel, checked
bit for bit against the oracle's scatter, then attended; the oracle checks
sampled rows (a few thousand (token, head) pairs, always including each
sequence's first and last token). Small cases are compared in full, with lengths
on both sides of every tile (128) and page (16) edge. Properties that hold at any
size are checked at full size: keys after a query's position have bit-exactly no
effect, and a sequence's first token returns its V row exactly."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import assert_attention_close, bits, dev

pytestmark = pytest.mark.gpu


class PrefillRun:
    def __init__(self, inp, max_seqlen=None):
        self.inp = inp
        self.kc, self.vc = dev(inp.k_cache), dev(inp.v_cache)
        self.q = dev(inp.q)
        self.bt, self.cu = dev(inp.block_tables), dev(inp.cu_seqlens)
        T, Hq, D = inp.q.shape
        self.out = torch.full((T, Hq, D), 5.0, dtype=torch.bfloat16, device="cuda")
        self.lse = torch.full((T, Hq), 5.0, dtype=torch.float32, device="cuda")
        self.status = torch.zeros(1, dtype=torch.int32, device="cuda")
        self.ws = torch.zeros(pgqa.prefill_workspace_size(inp.num_seqs, Hq, inp.max_seqlen),
                              dtype=torch.uint8, device="cuda")
        self.max_seqlen = max_seqlen if max_seqlen is not None else inp.max_seqlen

    def write(self):
        pgqa.kv_cache_write(dev(self.inp.key), dev(self.inp.value), dev(self.inp.slot_mapping),
                            self.kc, self.vc, dev_status=self.status)

    def prefill(self):
        pgqa.paged_prefill_varlen(self.out, self.lse, self.q, self.kc, self.vc, self.bt, self.cu,
                                  self.max_seqlen, self.inp.scale, workspace=self.ws,
                                  dev_status=self.status)

    def status_code(self):
        torch.cuda.synchronize()
        return int(self.status.item())


def oracle_cache(inp):
    return oracle.kv_cache_write(inp.key, inp.value, inp.slot_mapping, inp.k_cache, inp.v_cache)


def sample_rows(inp, n, seed):
    g = np.random.default_rng(seed)
    T, Hq, _ = inp.q.shape
    rows = set()
    cu = inp.cu_seqlens.tolist()
    for i in range(len(cu) - 1):
        for t in (cu[i], cu[i + 1] - 1, cu[i] + 127, cu[i] + 128):
            if cu[i] <= t < cu[i + 1]:
                rows.add((t, int(g.integers(Hq))))
    while len(rows) < n:
        rows.add((int(g.integers(T)), int(g.integers(Hq))))
    return np.array(sorted(rows), np.int32)


@pytest.fixture(scope="module")
def varlen():
    inp = workloads.varlen_prefill()
    run = PrefillRun(inp)
    run.write()
    run.prefill()
    assert run.status_code() == 0
    kc, vc = oracle_cache(inp)
    return inp, run, kc, vc


def test_kv_write_then_cache_matches_oracle(varlen):
    inp, run, kc, vc = varlen
    assert np.array_equal(bits(run.kc), kc) and np.array_equal(bits(run.vc), vc)


def test_varlen_prefill_sampled_rows(varlen):
    inp, run, kc, vc = varlen
    rows = sample_rows(inp, 3000, seed=1)
    ref_out, ref_lse = oracle.paged_prefill(inp.q, kc, vc, inp.block_tables, inp.cu_seqlens,
                                            inp.scale, rows=rows)
    t, h = rows[:, 0], rows[:, 1]
    assert_attention_close(run.out[t, h], run.lse[t, h], ref_out[t, h], ref_lse[t, h],
                           "varlen prefill sampled rows")


def test_first_token_returns_v_exactly(varlen):
    inp, run, kc, vc = varlen
    G = inp.q.shape[1] // inp.key.shape[1]
    for i, start in enumerate(inp.cu_seqlens[:-1].tolist()):
        for hq in range(inp.q.shape[1]):
            assert torch.equal(run.out[start, hq].cpu(), inp.value[start, hq // G])


def test_future_keys_have_no_effect(varlen):
    """Perturbing K/V after position p leaves rows 0..p bit-identical."""
    inp, run, _, _ = varlen
    i = int(np.argmax(inp.seq_lens))
    start, L = int(inp.cu_seqlens[i]), inp.seq_lens[i]
    cut = L // 2 + 5
    g = torch.Generator().manual_seed(77)
    key2, val2 = inp.key.clone(), inp.value.clone()
    key2[start + cut + 1:start + L] = torch.randn(key2[start + cut + 1:start + L].shape,
                                                  generator=g).to(torch.bfloat16) * 4
    val2[start + cut + 1:start + L] = torch.randn(val2[start + cut + 1:start + L].shape,
                                                  generator=g).to(torch.bfloat16) * 4
    run2 = PrefillRun(inp)
    pgqa.kv_cache_write(dev(key2), dev(val2), dev(inp.slot_mapping), run2.kc, run2.vc,
                        dev_status=run2.status)
    run2.prefill()
    assert run2.status_code() == 0
    a, b = start, start + cut + 1
    assert torch.equal(run.out[a:b], run2.out[a:b]) and torch.equal(run.lse[a:b], run2.lse[a:b])
    assert not torch.equal(run.out[b:start + L], run2.out[b:start + L])


def _full_case(lens, Hq, Hkv, D, seed):
    nb = sum(-(-L // 16) for L in lens) + 8
    inp = workloads.make_prefill(lens, Hq, Hkv, D, nb, seed)
    run = PrefillRun(inp)
    run.write()
    run.prefill()
    assert run.status_code() == 0
    kc, vc = oracle_cache(inp)
    ref_out, ref_lse = oracle.paged_prefill(inp.q, kc, vc, inp.block_tables, inp.cu_seqlens,
                                            inp.scale)
    return run, ref_out, ref_lse


@pytest.mark.parametrize("G", [1, 2, 4, 8])
@pytest.mark.parametrize("D", [64, 128])
def test_ragged_lengths_full_compare(G, D):
    lens = [1, 2, 15, 16, 17, 127, 128, 129, 255, 256, 300]
    run, ref_out, ref_lse = _full_case(lens, 2 * G, 2, D, seed=40 + G + D)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, f"G={G} D={D}")


def test_empty_sequences_in_the_batch():
    """Sequences with no token (repeated cu_seqlens values, at the start, in the
    middle and at the end) take no work, report nothing, and every other row is the
    oracle's."""
    run, ref_out, ref_lse = _full_case([0, 17, 0, 130, 1, 0], 8, 2, 128, seed=60)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse, "empty sequences")


def test_one_long_sequence_full_compare():
    run, ref_out, ref_lse = _full_case([1000], 4, 1, 128, seed=50)
    assert_attention_close(run.out, run.lse, ref_out, ref_lse)


def test_repeat_calls_reuse_the_workspace():
    """The ticket counters are left zero: a second call on the same workspace gives
    the same bits, and the counters end zero."""
    lens = [700, 3, 129, 400, 256]
    inp = workloads.make_prefill(lens, 8, 2, 128, 128, seed=65)
    run = PrefillRun(inp)
    run.write()
    run.prefill()
    assert run.status_code() == 0
    out1, lse1 = run.out.clone(), run.lse.clone()
    run.out.fill_(7.0)
    run.prefill()
    assert run.status_code() == 0
    assert torch.equal(run.out, out1) and torch.equal(run.lse, lse1)
    assert not torch.any(run.ws[:256])


def test_max_seqlen_upper_bound_is_enough():
    """max_seqlen only sizes the grid: a larger bound gives the same result."""
    lens = [130, 40, 257]
    inp = workloads.make_prefill(lens, 8, 2, 128, 64, seed=60)
    r1 = PrefillRun(inp)
    r1.write()
    r1.prefill()
    r2 = PrefillRun(inp, max_seqlen=1024)
    r2.write()
    r2.prefill()
    assert r1.status_code() == 0 and r2.status_code() == 0
    assert torch.equal(r1.out, r2.out) and torch.equal(r1.lse, r2.lse)


def test_bad_block_id_is_reported_not_faulted():
    lens = [200, 300]
    inp = workloads.make_prefill(lens, 4, 2, 128, 64, seed=70)
    run = PrefillRun(inp)
    run.write()
    torch.cuda.synchronize()
    run.bt[1, 3] = -1               # page 3 of sequence 1 (keys 48..63)
    run.prefill()
    assert run.status_code() == pgqa.EBADINDEX
    kc, vc = oracle_cache(inp)
    ref_out, ref_lse = oracle.paged_prefill(inp.q, kc, vc, inp.block_tables, inp.cu_seqlens,
                                            inp.scale)
    a = lens[0]
    # sequence 0 is untouched
    assert_attention_close(run.out[:a], run.lse[:a], ref_out[:a], ref_lse[:a])
    # every tile of sequence 1 reads page 3: its rows are 0 / -inf
    assert torch.all(run.out[a:] == 0) and torch.all(torch.isneginf(run.lse[a:]))


def test_inconsistent_lengths_are_reported():
    lens = [100, 50]
    inp = workloads.make_prefill(lens, 4, 2, 128, 32, seed=80)
    run = PrefillRun(inp, max_seqlen=64)   # too small a bound
    run.write()
    run.prefill()
    assert run.status_code() == pgqa.EINVAL
