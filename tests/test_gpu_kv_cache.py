"""KV-cache scatter and page gather on the GPU: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import paged_kv_gqa_10_gb300 as pgqa
import workloads
from parity import bits, dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def prefill_inputs():
    return workloads.varlen_prefill()


def test_kv_cache_write_bf16_prefill_workload(prefill_inputs):
    p = prefill_inputs
    kc, vc = dev(p.k_cache), dev(p.v_cache)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pgqa.kv_cache_write(dev(p.key), dev(p.value), dev(p.slot_mapping), kc, vc, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ok, ov = oracle.kv_cache_write(p.key, p.value, p.slot_mapping, p.k_cache, p.v_cache)
    assert np.array_equal(bits(kc), ok) and np.array_equal(bits(vc), ov)


@pytest.mark.parametrize("D", [64, 128])
def test_kv_cache_write_e4m3(D):
    T, Hkv, NB = 3000, 8, 256
    g = torch.Generator().manual_seed(D)
    key = (torch.randn((T, Hkv, D), generator=g) * 3).to(torch.bfloat16)
    value = torch.randn((T, Hkv, D), generator=g).to(torch.bfloat16)
    key[0, 0, :4] = torch.tensor([1e6, -1e6, 0.0, -0.0])          # saturation and signed zero
    slots = torch.randperm(NB * 16, generator=g)[:T].to(torch.int64)
    slots[::97] = -1
    ks = (torch.rand(Hkv, generator=g) * 0.05 + 0.001).to(torch.float32)
    vs = (torch.rand(Hkv, generator=g) * 0.05 + 0.001).to(torch.float32)
    kc0 = torch.randint(0, 256, (NB, Hkv, 16, D), generator=g, dtype=torch.uint8)
    vc0 = torch.randint(0, 256, (NB, Hkv, 16, D), generator=g, dtype=torch.uint8)
    kc, vc = dev(kc0), dev(vc0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pgqa.kv_cache_write(dev(key), dev(value), dev(slots), kc, vc, k_scale=dev(ks),
                        v_scale=dev(vs), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ok, ov = oracle.kv_cache_write(key, value, slots, kc0, vc0, dtype=oracle.E4M3, k_scale=ks,
                                   v_scale=vs)
    assert np.array_equal(kc.cpu().numpy(), ok) and np.array_equal(vc.cpu().numpy(), ov)


@pytest.mark.parametrize("D,bs,e4m3", [(128, 8, False), (64, 32, False), (128, 32, True),
                                       (96, 16, False), (128, 12, False), (64, 12, True)])
def test_kv_cache_write_block_sizes_and_head_dims(D, bs, e4m3):
    """Power-of-two block sizes at head_dim 64/128 take the 32-bit index kernel, the
    rest (block size 12, head_dim 96) the general one: both bit-exact."""
    T, Hkv, NB = 1500, 4, 480
    g = torch.Generator().manual_seed(D * 100 + bs)
    key = (torch.randn((T, Hkv, D), generator=g) * 2).to(torch.bfloat16)
    value = torch.randn((T, Hkv, D), generator=g).to(torch.bfloat16)
    slots = torch.randperm(NB * bs, generator=g)[:T].to(torch.int64)
    slots[::53] = -1
    if e4m3:
        ks = (torch.rand(Hkv, generator=g) * 0.05 + 0.001).to(torch.float32)
        vs = (torch.rand(Hkv, generator=g) * 0.05 + 0.001).to(torch.float32)
        kc0 = torch.randint(0, 256, (NB, Hkv, bs, D), generator=g, dtype=torch.uint8)
        vc0 = torch.randint(0, 256, (NB, Hkv, bs, D), generator=g, dtype=torch.uint8)
    else:
        ks = vs = None
        kc0 = torch.randn((NB, Hkv, bs, D), generator=g).to(torch.bfloat16)
        vc0 = torch.randn((NB, Hkv, bs, D), generator=g).to(torch.bfloat16)
    kc, vc = dev(kc0), dev(vc0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pgqa.kv_cache_write(dev(key), dev(value), dev(slots), kc, vc, k_scale=dev(ks),
                        v_scale=dev(vs), dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ok, ov = oracle.kv_cache_write(key, value, slots, kc0, vc0,
                                   dtype=oracle.E4M3 if e4m3 else oracle.BF16, k_scale=ks,
                                   v_scale=vs)
    if e4m3:
        assert np.array_equal(kc.cpu().numpy(), ok) and np.array_equal(vc.cpu().numpy(), ov)
    else:
        assert np.array_equal(bits(kc), ok) and np.array_equal(bits(vc), ov)


def test_kv_cache_write_bad_slot_reported():
    T, Hkv, D, NB = 64, 2, 128, 4
    key = torch.randn((T, Hkv, D)).to(torch.bfloat16)
    slots = torch.arange(T, dtype=torch.int64)
    slots[10] = NB * 16 + 3
    kc0 = torch.zeros((NB, Hkv, 16, D), dtype=torch.bfloat16)
    kc, vc = dev(kc0), dev(kc0)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pgqa.kv_cache_write(dev(key), dev(key), dev(slots), kc, vc, dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == pgqa.EBADINDEX
    good = slots.clone()
    good[10] = -1
    ok, _ = oracle.kv_cache_write(key, key, good, kc0, kc0)
    assert np.array_equal(bits(kc), ok)


@pytest.mark.parametrize("which", ["llama8b", "prefix", "e4m3"])
def test_paged_kv_gather_bit_exact(which):
    if which == "llama8b":
        inp = workloads.llama3_8b_decode()
    elif which == "prefix":
        inp = workloads.prefix_sharing_decode()
    else:
        inp = workloads.make_decode([5, 16, 17, 400], 8, 2, 128, 64, seed=9, cache_dtype="e4m3")
    B, Hkv, D, M = inp.num_seqs, inp.num_kv_heads, inp.head_dim, inp.max_context_len
    kc, vc = dev(inp.k_cache), dev(inp.v_cache)
    ko = torch.full((B, Hkv, M, D), 1, dtype=inp.k_cache.dtype, device="cuda")
    vo = torch.full_like(ko, 1)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pgqa.paged_kv_gather(kc, vc, dev(inp.block_tables), dev(inp.context_lens), M, ko, vo,
                         dev_status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    kb, vb = bits(ko), bits(vo)
    elem = np.uint16 if inp.cache_dtype == "bf16" else np.uint8
    src_k, src_v = bits(inp.k_cache), bits(inp.v_cache)
    for b, L in enumerate(inp.context_lens.tolist()):
        assert not kb[b, :, L:].any() and not vb[b, :, L:].any()
        for h in range(Hkv):
            # expected rows read straight off the source pool by the table definition
            j = np.arange(L)
            pbn = inp.block_tables[b].numpy()[j // 16]
            assert np.array_equal(kb[b, h, :L], src_k[pbn, h, j % 16].astype(elem))
            assert np.array_equal(vb[b, h, :L], src_v[pbn, h, j % 16].astype(elem))
        if b < 4 and inp.cache_dtype == "bf16":
            K, V = oracle.gather_kv(inp.k_cache, inp.v_cache, inp.block_tables[b], L, 0)
            got = ko[b, 0, :L].float().cpu().double().numpy()
            assert np.array_equal(got, K)
