"""Pins for the fp64 oracle: checks against things other than the oracle itself.

Each ``pin_*`` function raises AssertionError when the oracle currently loaded
(``oracle.use_library`` can swap in another build) disagrees with:
  - a library routine that computes the same quantity a different way
    (torch's scaled_dot_product_attention in float64, torch's float8 cast,
    numpy fancy-index assignment for the scatter),
  - a closed form or invariant the definitions fix (weights sum to 1, a single
    key returns V, q = 0 gives uniform weights, future keys have no effect,
    LSE-weighted merge of disjoint key ranges equals the whole),
  - an independent pure-Python brute force with ``math.fsum`` on tiny inputs,
  - values printed in a published format table (tests/golden/).
They are plain functions (not pytest tests) so the planted-mistake test can run
them against mutated oracle builds; ``test_oracle_pins.py`` runs them as tests.
"""
import math
import os

import numpy as np
import torch
import torch.nn.functional as F

import oracle as O

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
BS = 16


# ----------------------------------------------------------------- helpers

def bf16(x) -> torch.Tensor:
    return torch.as_tensor(x, dtype=torch.float32).to(torch.bfloat16)


def rand_bf16(shape, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(shape, generator=g).to(torch.bfloat16)


def identity_pool(K, V, lens, nan_tail=True):
    """Pack per-sequence contiguous K/V (lists of [Hkv, L, D] bf16) into a pool
    with sequence b in consecutive blocks, using only reshape/permute (the layout
    definition [NB, Hkv, bs, D]); returns (k_cache, v_cache, block_tables)."""
    Hkv, _, D = K[0].shape
    nbs = [-(-L // BS) for L in lens]
    total = sum(nbs)
    kc = torch.full((total, Hkv, BS, D), float("nan") if nan_tail else 0.0, dtype=torch.bfloat16)
    vc = kc.clone()
    table = torch.full((len(lens), max(nbs + [1])), -1, dtype=torch.int32)
    base = 0
    for b, L in enumerate(lens):
        n = nbs[b]
        pad = n * BS - L
        kp = torch.cat([K[b], torch.full((Hkv, pad, D), float("nan"), dtype=torch.bfloat16)], 1)
        vp = torch.cat([V[b], torch.full((Hkv, pad, D), float("nan"), dtype=torch.bfloat16)], 1)
        kc[base:base + n] = kp.reshape(Hkv, n, BS, D).permute(1, 0, 2, 3)
        vc[base:base + n] = vp.reshape(Hkv, n, BS, D).permute(1, 0, 2, 3)
        table[b, :n] = torch.arange(base, base + n, dtype=torch.int32)
        base += n
    return kc, vc, table


def shuffle_pool(kc, vc, table, seed):
    """The same logical contents with physical blocks relabelled by a permutation."""
    g = torch.Generator().manual_seed(seed)
    nb = kc.shape[0]
    perm = torch.randperm(nb, generator=g)           # new id of old block i
    kc2 = torch.empty_like(kc)
    vc2 = torch.empty_like(vc)
    kc2[perm] = kc
    vc2[perm] = vc
    t2 = table.clone()
    m = table >= 0
    t2[m] = perm[table[m].long()].to(torch.int32)
    return kc2, vc2, t2


def sdpa_rows(q, K, V, scale, causal=False):
    """torch SDPA in float64. q [H, Lq, D], K/V [H, L, D] (already one K/V per head)."""
    return F.scaled_dot_product_attention(q.double()[None], K.double()[None], V.double()[None],
                                          is_causal=causal, scale=scale)[0]


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    if not np.allclose(a, b, rtol=rtol, atol=atol, equal_nan=False):
        err = float(np.max(np.nan_to_num(np.abs(a - b), nan=np.inf))) if a.size else 0.0
        raise AssertionError(f"{what}: max abs diff {err}")


def _decode_case(lens, Hq, Hkv, D, seed):
    K = [rand_bf16((Hkv, L, D), seed * 10 + b) for b, L in enumerate(lens)]
    V = [rand_bf16((Hkv, L, D), seed * 10 + 5 + b) for b, L in enumerate(lens)]
    q = rand_bf16((len(lens), Hq, D), seed * 10 + 9)
    return q, K, V


# ----------------------------------------------------------- number formats

def pin_e4m3_golden():
    with open(os.path.join(GOLDEN, "e4m3_values.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            code, val = line.split()
            got = O.e4m3_to_f64(int(code, 16))
            if val == "nan":
                assert math.isnan(got), (code, got)
            else:
                want = float(val)
                assert got == want and math.copysign(1, got) == math.copysign(1, want), \
                    (code, got, want)


def pin_e4m3_roundtrip():
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        v = O.e4m3_to_f64(c)
        assert O.e4m3_from_f32(v) == c, (hex(c), v)


def pin_e4m3_vs_torch_cast():
    """RNE ties-to-even on every midpoint and a dense sweep, against torch's cast
    (which agrees with satfinite below the first value past 448 + half an ulp)."""
    vals = [O.e4m3_to_f64(c) for c in range(0x7F)]
    mids = [(a + b) / 2 for a, b in zip(vals[:-1], vals[1:])]
    sweep = np.linspace(-460, 460, 20001).tolist()
    small = (np.linspace(-0.03, 0.03, 4001)).tolist()
    xs = np.array(mids + [-m for m in mids] + sweep + small, np.float32)
    want = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    for x, w in zip(xs.tolist(), want.tolist()):
        got = O.e4m3_from_f32(x)
        assert got == w, (x, hex(got), hex(w))


def pin_e4m3_saturation():
    assert O.e4m3_from_f32(500.0) == 0x7E
    assert O.e4m3_from_f32(-1e30) == 0xFE
    assert O.e4m3_from_f32(float("inf")) == 0x7E
    assert O.e4m3_from_f32(449.0) == 0x7E


def pin_bf16_widening():
    g = np.random.default_rng(7)
    bits = g.integers(0, 1 << 16, 4000, dtype=np.int64).astype(np.uint16)
    want = torch.from_numpy(bits.view(np.int16)).view(torch.bfloat16).double().numpy()
    got = np.array([O.bf16_to_f64(int(b)) for b in bits])
    fin = np.isfinite(want)
    assert np.array_equal(got[fin], want[fin])
    assert np.array_equal(np.isnan(got), np.isnan(want))


# ------------------------------------------------------------ cache write

def pin_kv_write_bf16_scatter():
    NB, Hkv, D, T = 6, 3, 8, 40
    key = rand_bf16((T, Hkv, D), 1)
    val = rand_bf16((T, Hkv, D), 2)
    g = torch.Generator().manual_seed(3)
    slots = torch.randperm(NB * BS, generator=g)[:T].to(torch.int64)
    slots[5] = -1
    kc0 = rand_bf16((NB, Hkv, BS, D), 4)
    vc0 = rand_bf16((NB, Hkv, BS, D), 5)
    kc, vc = O.kv_cache_write(key, val, slots, kc0, vc0)
    want_k = kc0.clone()
    want_v = vc0.clone()
    s = slots[slots >= 0]
    want_k[s // BS, :, s % BS, :] = key[slots >= 0]
    want_v[s // BS, :, s % BS, :] = val[slots >= 0]
    assert np.array_equal(kc, want_k.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(vc, want_v.view(torch.int16).numpy().view(np.uint16))


def pin_kv_write_e4m3():
    NB, Hkv, D, T = 4, 2, 16, 30
    key = rand_bf16((T, Hkv, D), 11) * 3
    val = rand_bf16((T, Hkv, D), 12)
    slots = torch.arange(T, dtype=torch.int64) * 2
    ks = torch.tensor([0.0123, 0.5], dtype=torch.float32)
    vs = torch.tensor([0.031, 0.007], dtype=torch.float32)
    kc0 = torch.zeros((NB, Hkv, BS, D), dtype=torch.uint8)
    kc, vc = O.kv_cache_write(key, val, slots, kc0, kc0.clone(), dtype=O.E4M3, k_scale=ks,
                              v_scale=vs)
    s = slots
    for src, sc, got in ((key, ks, kc), (val, vs, vc)):
        x = (src.float() / sc.view(1, -1, 1)).clamp(-448, 448)   # binary32 division
        codes = x.to(torch.float8_e4m3fn).view(torch.uint8)
        want = torch.zeros_like(kc0)
        want[s // BS, :, s % BS, :] = codes
        assert np.array_equal(got, want.numpy())


def pin_kv_write_skip_and_range():
    NB, Hkv, D = 2, 1, 4
    key = rand_bf16((2, Hkv, D), 21)
    kc0 = torch.zeros((NB, Hkv, BS, D), dtype=torch.bfloat16)
    kc, _ = O.kv_cache_write(key, key, torch.tensor([-1, -7]), kc0, kc0)
    assert not kc.any()
    try:
        O.kv_cache_write(key, key, torch.tensor([0, NB * BS]), kc0, kc0)
    except ValueError:
        pass
    else:
        raise AssertionError("slot past the pool accepted")


# ------------------------------------------------------------ page gather

def pin_gather_identity_layout():
    lens = [37, 16, 5]
    Hkv, D = 3, 8
    _, K, V = _decode_case(lens, Hkv, Hkv, D, 31)
    kc, vc, table = identity_pool(K, V, lens)
    kc, vc, table = shuffle_pool(kc, vc, table, 32)
    for b, L in enumerate(lens):
        for h in range(Hkv):
            Kg, Vg = O.gather_kv(kc, vc, table[b], L, h)
            assert np.array_equal(Kg, K[b][h].double().numpy())
            assert np.array_equal(Vg, V[b][h].double().numpy())


def pin_bad_block_index():
    lens = [20]
    _, K, V = _decode_case(lens, 2, 2, 8, 41)
    kc, vc, table = identity_pool(K, V, lens)
    q = rand_bf16((1, 2, 8), 42)
    t = torch.cat([table, torch.full((1, 2), -1, dtype=torch.int32)], 1)
    O.paged_decode(q, kc, vc, t, torch.tensor([20], dtype=torch.int32), 0.3)  # -1 past L: fine
    for bad in (-1, kc.shape[0]):
        t2 = t.clone()
        t2[0, 1] = bad
        try:
            O.paged_decode(q, kc, vc, t2, torch.tensor([20], dtype=torch.int32), 0.3)
        except ValueError:
            continue
        raise AssertionError(f"block id {bad} inside the context accepted")


# ------------------------------------------------------------------ decode

def pin_decode_vs_sdpa():
    """Paged decode == library attention on the contiguous K/V, with repeat_kv
    done by torch.repeat_interleave; pages relabelled by a random permutation."""
    lens = [37, 50, 1, 16]
    Hq, Hkv, D = 8, 2, 32
    scale = 1 / math.sqrt(D)
    q, K, V = _decode_case(lens, Hq, Hkv, D, 51)
    kc, vc, table = shuffle_pool(*identity_pool(K, V, lens), 52)
    out, lse = O.paged_decode(q, kc, vc, table, torch.tensor(lens, dtype=torch.int32), scale)
    G = Hq // Hkv
    for b, L in enumerate(lens):
        Kr = K[b].repeat_interleave(G, 0)
        Vr = V[b].repeat_interleave(G, 0)
        want = sdpa_rows(q[b][:, None, :], Kr, Vr, scale)[:, 0, :]
        _close(out[b], want.numpy(), 1e-11, 1e-12, "decode vs sdpa")
        s = torch.einsum("hd,hld->hl", q[b].double(), Kr.double()) * scale
        _close(lse[b], torch.logsumexp(s, -1).numpy(), 1e-12, 1e-12, "lse vs logsumexp")


def pin_decode_relabel_invariance():
    lens = [33, 64]
    q, K, V = _decode_case(lens, 4, 2, 16, 61)
    kc, vc, table = identity_pool(K, V, lens)
    cl = torch.tensor(lens, dtype=torch.int32)
    o1, l1 = O.paged_decode(q, kc, vc, table, cl, 0.25)
    o2, l2 = O.paged_decode(q, *shuffle_pool(kc, vc, table, 62), cl, 0.25)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


def pin_gqa_equals_repeated_mha():
    lens = [29]
    Hq, Hkv, D = 8, 2, 16
    q, K, V = _decode_case(lens, Hq, Hkv, D, 71)
    cl = torch.tensor(lens, dtype=torch.int32)
    og, lg = O.paged_decode(q, *identity_pool(K, V, lens), cl, 0.2)
    Kr = [K[0].repeat_interleave(Hq // Hkv, 0)]
    Vr = [V[0].repeat_interleave(Hq // Hkv, 0)]
    om, lm = O.paged_decode(q, *identity_pool(Kr, Vr, lens), cl, 0.2)
    assert np.array_equal(og, om) and np.array_equal(lg, lm)


def pin_weights_sum_to_one():
    lens = [45, 3]
    q, K, _ = _decode_case(lens, 4, 2, 16, 81)
    ones = [torch.ones_like(k) for k in K]
    out, _ = O.paged_decode(q, *identity_pool(K, ones, lens),
                            torch.tensor(lens, dtype=torch.int32), 0.7)
    _close(out, np.ones_like(out), 1e-13, 1e-13, "sum of weights")


def pin_single_key():
    q, K, V = _decode_case([1], 4, 2, 16, 91)
    out, lse = O.paged_decode(q, *identity_pool(K, V, [1]), torch.tensor([1], dtype=torch.int32),
                              0.5)
    for hq in range(4):
        h = hq // 2
        assert np.array_equal(out[0, hq], V[0][h, 0].double().numpy())
        s0 = 0.5 * math.fsum(float(a) * float(b) for a, b in zip(q[0, hq].double(),
                                                                  K[0][h, 0].double()))
        assert abs(lse[0, hq] - s0) <= 1e-13 * max(1.0, abs(s0)), (lse[0, hq], s0)


def pin_uniform_closed_form():
    lens = [23, 40]
    _, K, V = _decode_case(lens, 4, 2, 16, 101)
    q = torch.zeros((2, 4, 16), dtype=torch.bfloat16)
    out, lse = O.paged_decode(q, *identity_pool(K, V, lens), torch.tensor(lens, dtype=torch.int32),
                              0.3)
    for b, L in enumerate(lens):
        for hq in range(4):
            _close(out[b, hq], V[b][hq // 2].double().mean(0).numpy(), 1e-13, 1e-14, "mean V")
            assert abs(lse[b, hq] - math.log(L)) < 1e-13


def _brute_decode(q, K, V, scale):
    """Independent nested-loop attention with math.fsum (tiny inputs only)."""
    Hq = q.shape[0]
    Hkv, L, D = K.shape
    G = Hq // Hkv
    out = np.zeros((Hq, D))
    lse = np.zeros(Hq)
    for hq in range(Hq):
        h = hq // G
        s = [scale * math.fsum(float(q[hq, d]) * float(K[h, j, d]) for d in range(D))
             for j in range(L)]
        m = max(s)
        z = math.fsum(math.exp(x - m) for x in s)
        lse[hq] = m + math.log(z)
        w = [math.exp(x - lse[hq]) for x in s]
        for d in range(D):
            out[hq, d] = math.fsum(w[j] * float(V[h, j, d]) for j in range(L))
    return out, lse


def pin_bruteforce_tiny():
    lens = [7, 19]
    Hq, Hkv, D = 4, 2, 8
    q, K, V = _decode_case(lens, Hq, Hkv, D, 111)
    out, lse = O.paged_decode(q, *shuffle_pool(*identity_pool(K, V, lens), 112),
                              torch.tensor(lens, dtype=torch.int32), 0.35)
    for b in range(2):
        bo, bl = _brute_decode(q[b].double().numpy(), K[b].double().numpy(),
                               V[b].double().numpy(), 0.35)
        _close(out[b], bo, 1e-12, 1e-12, "brute out")
        _close(lse[b], bl, 1e-12, 1e-12, "brute lse")


def pin_split_merge_identity():
    """out and lse over disjoint key ranges, merged with weights exp(lse_i - lse),
    equal the whole: the identity split-K decoding relies on."""
    L, D = 70, 16
    q, K, V = _decode_case([L], 2, 1, D, 121)
    Kd, Vd = K[0][0].double().numpy(), V[0][0].double().numpy()
    full_o, full_l = O.dense_row(q[0, 0], Kd, Vd, 0.4)
    parts = [O.dense_row(q[0, 0], Kd[a:b], Vd[a:b], 0.4) for a, b in ((0, 16), (16, 48), (48, 70))]
    lses = np.array([p[1] for p in parts])
    tot = lses.max() + math.log(sum(math.exp(x - lses.max()) for x in lses))
    merged = sum(math.exp(p[1] - tot) * p[0] for p in parts)
    _close(merged, full_o, 1e-12, 1e-13, "merge out")
    assert abs(tot - full_l) < 1e-12


def pin_e4m3_decode_cache():
    """An E4M3 cache means code value * per-kv-head scale: paged decode on random
    codes equals library attention on the cache dequantised by torch's float8
    view, gathered with reshape/permute."""
    lens = [21, 34]
    Hq, Hkv, D = 4, 2, 16
    q = rand_bf16((2, Hq, D), 131)
    g = torch.Generator().manual_seed(132)
    nbs = [-(-L // BS) for L in lens]
    kc = torch.randint(0, 0x7F, (sum(nbs), Hkv, BS, D), generator=g, dtype=torch.uint8)
    kc |= torch.randint(0, 2, kc.shape, generator=g, dtype=torch.uint8) << 7
    kc[kc == 0xFF] = 0x80
    vc = kc.flip(0).clone()
    table = torch.tensor([[0, 1, -1], [2, 3, 4]], dtype=torch.int32)
    ks = torch.tensor([0.01, 0.02])
    vs = torch.tensor([0.03, 0.005])
    out, lse = O.paged_decode(q, kc, vc, table, torch.tensor(lens, dtype=torch.int32), 0.25,
                              dtype=O.E4M3, k_scale=ks, v_scale=vs)
    deq = lambda c, s: c.view(torch.float8_e4m3fn).double() * s.double().view(1, -1, 1, 1)
    kd, vd = deq(kc, ks), deq(vc, vs)
    for b, L in enumerate(lens):
        blocks = table[b, :nbs[b]].long()
        Kb = kd[blocks].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :L]
        Vb = vd[blocks].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :L]
        want = sdpa_rows(q[b][:, None, :], Kb.repeat_interleave(2, 0),
                         Vb.repeat_interleave(2, 0), 0.25)[:, 0, :]
        _close(out[b], want.numpy(), 1e-11, 1e-13, "e4m3 decode vs sdpa")


# ----------------------------------------------------------------- prefill

def _prefill_case(lens, Hq, Hkv, D, seed):
    T = sum(lens)
    q = rand_bf16((T, Hq, D), seed)
    K = [rand_bf16((Hkv, L, D), seed + 1 + b) for b, L in enumerate(lens)]
    V = [rand_bf16((Hkv, L, D), seed + 50 + b) for b, L in enumerate(lens)]
    cu = torch.tensor([0] + np.cumsum(lens).tolist(), dtype=torch.int32)
    return q, K, V, cu


def pin_prefill_vs_sdpa_causal():
    lens = [1, 17, 40]
    Hq, Hkv, D = 4, 2, 16
    q, K, V, cu = _prefill_case(lens, Hq, Hkv, D, 141)
    kc, vc, table = shuffle_pool(*identity_pool(K, V, lens), 142)
    out, lse = O.paged_prefill(q, kc, vc, table, cu, 0.25)
    for i, L in enumerate(lens):
        a = int(cu[i])
        qi = q[a:a + L].permute(1, 0, 2)                     # [Hq, L, D]
        Kr = K[i].repeat_interleave(Hq // Hkv, 0)
        Vr = V[i].repeat_interleave(Hq // Hkv, 0)
        want = sdpa_rows(qi, Kr, Vr, 0.25, causal=True).permute(1, 0, 2)
        _close(out[a:a + L], want.numpy(), 1e-11, 1e-12, "prefill vs sdpa")


def pin_prefill_causality():
    lens = [30]
    q, K, V, cu = _prefill_case(lens, 2, 1, 8, 151)
    o1, l1 = O.paged_prefill(q, *identity_pool(K, V, lens), cu, 0.3)
    t = 11
    K2 = [K[0].clone()]
    V2 = [V[0].clone()]
    K2[0][:, t + 1:] = rand_bf16(K2[0][:, t + 1:].shape, 152)
    V2[0][:, t + 1:] = rand_bf16(V2[0][:, t + 1:].shape, 153)
    o2, l2 = O.paged_prefill(q, *identity_pool(K2, V2, lens), cu, 0.3)
    assert np.array_equal(o1[:t + 1], o2[:t + 1]) and np.array_equal(l1[:t + 1], l2[:t + 1])
    assert not np.array_equal(o1[t + 1:], o2[t + 1:])


def pin_prefill_first_token_and_uniform():
    lens = [9, 12]
    Hq, Hkv, D = 2, 1, 8
    _, K, V, cu = _prefill_case(lens, Hq, Hkv, D, 161)
    q = torch.zeros((sum(lens), Hq, D), dtype=torch.bfloat16)
    out, lse = O.paged_prefill(q, *identity_pool(K, V, lens), cu, 0.3)
    for i, L in enumerate(lens):
        a = int(cu[i])
        for p in range(L):
            for hq in range(Hq):
                _close(out[a + p, hq], V[i][0, :p + 1].double().mean(0).numpy(), 1e-13, 1e-14,
                       "uniform prefill")
                assert abs(lse[a + p, hq] - math.log(p + 1)) < 1e-13
        assert np.array_equal(out[a, 0], V[i][0, 0].double().numpy())


def pin_prefill_rows_subset():
    lens = [20, 5]
    q, K, V, cu = _prefill_case(lens, 4, 2, 8, 171)
    pool = identity_pool(K, V, lens)
    full_o, full_l = O.paged_prefill(q, *pool, cu, 0.3)
    rows = [(0, 0), (19, 3), (20, 1), (24, 2)]
    so, sl = O.paged_prefill(q, *pool, cu, 0.3, rows=rows)
    for t, h in rows:
        assert np.array_equal(so[t, h], full_o[t, h]) and sl[t, h] == full_l[t, h]


# ------------------------------------------------------- sliding-window decode

def pin_window_vs_sdpa_mask():
    """torch SDPA with an explicit mask over the whole context: keys L-W..L-1 only."""
    lens, W = [40, 9, 100], 16
    Hq, Hkv, D = 4, 2, 16
    q, K, V = _decode_case(lens, Hq, Hkv, D, 221)
    kc, vc, table = shuffle_pool(*identity_pool(K, V, lens), 222)
    cl = torch.tensor(lens, dtype=torch.int32)
    out, lse = O.paged_decode_window(q, kc, vc, table, cl, 0.3, W)
    for b, L in enumerate(lens):
        Kr = K[b].repeat_interleave(Hq // Hkv, 0)
        Vr = V[b].repeat_interleave(Hq // Hkv, 0)
        mask = (torch.arange(L) >= L - W)[None, :]
        want = F.scaled_dot_product_attention(q[b][:, None].double()[None], Kr.double()[None],
                                              Vr.double()[None], attn_mask=mask,
                                              scale=0.3)[0][:, 0]
        _close(out[b], want.numpy(), 1e-11, 1e-12, "window decode vs sdpa")


def pin_window_is_decode_of_the_window():
    """A window over a long context equals plain decode of a cache that holds only the
    window's keys; a window at least the context is plain decode."""
    lens, W = [70, 23], 20
    Hq, Hkv, D = 4, 1, 8
    q, K, V = _decode_case(lens, Hq, Hkv, D, 231)
    pool = identity_pool(K, V, lens)
    cl = torch.tensor(lens, dtype=torch.int32)
    wo, wl = O.paged_decode_window(q, *pool, cl, 0.2, W)
    tails = [min(L, W) for L in lens]
    Kt = [K[b][:, L - n:] for b, (L, n) in enumerate(zip(lens, tails))]
    Vt = [V[b][:, L - n:] for b, (L, n) in enumerate(zip(lens, tails))]
    do, dl = O.paged_decode(q, *identity_pool(Kt, Vt, tails), torch.tensor(tails, dtype=torch.int32), 0.2)
    assert np.array_equal(wo, do) and np.array_equal(wl, dl)
    fo, fl = O.paged_decode(q, *pool, cl, 0.2)
    go, gl = O.paged_decode_window(q, *pool, cl, 0.2, max(lens))
    assert np.array_equal(fo, go) and np.array_equal(fl, gl)


def pin_window_of_one_is_last_value():
    lens = [5, 33]
    q, K, V = _decode_case(lens, 2, 1, 8, 241)
    out, lse = O.paged_decode_window(q, *identity_pool(K, V, lens),
                                     torch.tensor(lens, dtype=torch.int32), 0.5, 1)
    for b, L in enumerate(lens):
        for h in range(2):
            assert np.array_equal(out[b, h], V[b][0, L - 1].double().numpy())
            s = 0.5 * float((q[b, h].double() * K[b][0, L - 1].double()).sum())
            assert abs(lse[b, h] - s) < 1e-12


# ------------------------------------------- prefill over a cached prefix (chunked)

def _chunk_case(lens_k, lens_q, Hq, Hkv, D, seed):
    """Full per-sequence K/V of Lk tokens; queries for the last Lq of them."""
    K = [rand_bf16((Hkv, L, D), seed + 1 + b) for b, L in enumerate(lens_k)]
    V = [rand_bf16((Hkv, L, D), seed + 70 + b) for b, L in enumerate(lens_k)]
    q = rand_bf16((sum(lens_q), Hq, D), seed)
    cu = torch.tensor([0] + np.cumsum(lens_q).tolist(), dtype=torch.int32)
    return q, K, V, cu, torch.tensor(lens_k, dtype=torch.int32)


def pin_chunked_vs_sdpa_bottom_right():
    """torch SDPA with an explicit mask: chunk row i sees keys 0..Lk-Lq+i."""
    lens_k, lens_q = [23, 40, 5], [7, 1, 5]
    Hq, Hkv, D = 4, 2, 16
    q, K, V, cu, lk = _chunk_case(lens_k, lens_q, Hq, Hkv, D, 181)
    kc, vc, table = shuffle_pool(*identity_pool(K, V, lens_k), 182)
    out, lse = O.paged_prefill_kv(q, kc, vc, table, cu, lk, 0.25)
    for i, (Lk, Lq) in enumerate(zip(lens_k, lens_q)):
        a = int(cu[i])
        qi = q[a:a + Lq].permute(1, 0, 2)                     # [Hq, Lq, D]
        Kr = K[i].repeat_interleave(Hq // Hkv, 0)
        Vr = V[i].repeat_interleave(Hq // Hkv, 0)
        mask = torch.arange(Lk)[None, :] <= (Lk - Lq + torch.arange(Lq))[:, None]
        want = F.scaled_dot_product_attention(qi.double()[None], Kr.double()[None],
                                              Vr.double()[None], attn_mask=mask,
                                              scale=0.25)[0].permute(1, 0, 2)
        _close(out[a:a + Lq], want.numpy(), 1e-11, 1e-12, "chunked prefill vs sdpa")


def pin_chunked_equals_full_prefill_rows():
    """A chunk's rows are the same rows of a prefill over the whole sequence."""
    lens = [33, 18]
    lens_q = [9, 18]
    Hq, Hkv, D = 2, 1, 8
    qf, K, V, cuf = _prefill_case(lens, Hq, Hkv, D, 191)
    pool = identity_pool(K, V, lens)
    full_o, full_l = O.paged_prefill(qf, *pool, cuf, 0.3)
    rows = torch.cat([qf[int(cuf[i + 1]) - n:int(cuf[i + 1])] for i, n in enumerate(lens_q)])
    cu = torch.tensor([0] + np.cumsum(lens_q).tolist(), dtype=torch.int32)
    o, l = O.paged_prefill_kv(rows, *pool, cu, torch.tensor(lens, dtype=torch.int32), 0.3)
    for i, n in enumerate(lens_q):
        e = int(cuf[i + 1])
        assert np.array_equal(o[int(cu[i]):int(cu[i + 1])], full_o[e - n:e])
        assert np.array_equal(l[int(cu[i]):int(cu[i + 1])], full_l[e - n:e])


def pin_chunked_last_row_is_decode():
    """The last row of a chunk attends to the whole context: a decode step."""
    lens_k, lens_q = [50, 17], [4, 3]
    Hq, Hkv, D = 4, 2, 8
    q, K, V, cu, lk = _chunk_case(lens_k, lens_q, Hq, Hkv, D, 201)
    pool = identity_pool(K, V, lens_k)
    o, l = O.paged_prefill_kv(q, *pool, cu, lk, 0.2)
    last = torch.stack([q[int(cu[i + 1]) - 1] for i in range(len(lens_k))])
    do, dl = O.paged_decode(last, *pool, lk, 0.2)
    for i in range(len(lens_k)):
        t = int(cu[i + 1]) - 1
        _close(o[t], do[i], 1e-13, 1e-14, "chunk last row vs decode")
        _close(l[t], dl[i], 1e-13, 1e-14, "chunk last row lse vs decode")


def pin_chunked_without_prefix_is_prefill():
    lens = [12, 3]
    q, K, V, cu = _prefill_case(lens, 4, 2, 8, 211)
    pool = identity_pool(K, V, lens)
    o1, l1 = O.paged_prefill(q, *pool, cu, 0.3)
    o2, l2 = O.paged_prefill_kv(q, *pool, cu, torch.tensor(lens, dtype=torch.int32), 0.3)
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)


# ------------------------------------------------------- prefill over an E4M3 cache

def pin_e4m3_prefill_cache():
    """Both prefill functions over an E4M3 cache of random codes equal library
    attention (causal; bottom-right for the chunked form) on the cache dequantised
    by torch's float8 view with separate per-kv-head K and V scales."""
    lens_k, lens_q = [19, 40], [19, 6]
    Hq, Hkv, D = 4, 2, 16
    g = torch.Generator().manual_seed(231)
    nbs = [-(-L // BS) for L in lens_k]
    kc = torch.randint(0, 0x7F, (sum(nbs), Hkv, BS, D), generator=g, dtype=torch.uint8)
    kc |= torch.randint(0, 2, kc.shape, generator=g, dtype=torch.uint8) << 7
    kc[kc == 0xFF] = 0x80
    vc = kc.flip(0).clone()
    table = torch.tensor([[1, 0, -1], [3, 2, 4]], dtype=torch.int32)
    ks, vs = torch.tensor([0.01, 0.02]), torch.tensor([0.03, 0.005])
    deq = lambda c, s: c.view(torch.float8_e4m3fn).double() * s.double().view(1, -1, 1, 1)
    kd, vd = deq(kc, ks), deq(vc, vs)
    q = rand_bf16((sum(lens_q), Hq, D), 232)
    cu = torch.tensor([0] + np.cumsum(lens_q).tolist(), dtype=torch.int32)
    lk = torch.tensor(lens_k, dtype=torch.int32)
    out, lse = O.paged_prefill_kv(q, kc, vc, table, cu, lk, 0.25, dtype=O.E4M3, k_scale=ks,
                                  v_scale=vs)
    for i, (Lk, Lq) in enumerate(zip(lens_k, lens_q)):
        blocks = table[i, :nbs[i]].long()
        Kb = kd[blocks].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :Lk]
        Vb = vd[blocks].permute(1, 0, 2, 3).reshape(Hkv, -1, D)[:, :Lk]
        a = int(cu[i])
        qi = q[a:a + Lq].permute(1, 0, 2).double()
        mask = torch.arange(Lk)[None, :] <= (Lk - Lq + torch.arange(Lq))[:, None]
        want = F.scaled_dot_product_attention(qi[None], Kb.repeat_interleave(2, 0)[None],
                                              Vb.repeat_interleave(2, 0)[None], attn_mask=mask,
                                              scale=0.25)[0].permute(1, 0, 2)
        _close(out[a:a + Lq], want.numpy(), 1e-11, 1e-13, "e4m3 chunked prefill vs sdpa")
    # sequence 0 has no prefix: the whole-sequence form gives the same rows
    cu0 = torch.tensor([0, lens_k[0]], dtype=torch.int32)
    o0, l0 = O.paged_prefill(q[:lens_k[0]], kc, vc, table[:1], cu0, 0.25, dtype=O.E4M3,
                             k_scale=ks, v_scale=vs)
    assert np.array_equal(o0, out[:lens_k[0]]) and np.array_equal(l0, lse[:lens_k[0]])


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_") and callable(v)]


def run_all():
    """Names of the pins that fail against the currently loaded oracle."""
    failed = []
    for p in ALL_PINS:
        try:
            p()
        except Exception:  # noqa: BLE001 -- any failure counts
            failed.append(p.__name__)
    return failed
