"""Seeded synthetic inputs for paged grouped-query attention.

This module is shared, as data, by the CUDA tests/benchmark and by the CPU
oracle. It holds none of the attention arithmetic: it draws random numbers,
lays them out in the paged cache format and builds block tables, slot mappings
and cumulative lengths. Everything is generated on the CPU with a seeded
``torch.Generator`` so both sides see identical bytes.

Workload shapes follow the serving settings the pages describe: Llama-style
models with grouped-query heads (Llama-3-8B: 32 query / 8 kv heads; Llama-2-70B:
64 query heads in 8 groups), head_dim 128, 16-token blocks, block tables of
int32 physical block ids with -1 for unallocated entries, and copy-on-write
sharing of a common prompt's blocks.

Cache layout: ``[num_blocks, num_kv_heads, block_size, head_dim]`` for K and V
separately; one (block, kv-head) page is contiguous.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import List, Optional, Sequence

import torch

BLOCK_SIZE = 16


def _gen(seed: int) -> torch.Generator:
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    return g


def _randn_bf16(shape, g) -> torch.Tensor:
    return torch.randn(shape, generator=g, dtype=torch.float32).to(torch.bfloat16)


def e4m3_encode_with_scale(x: torch.Tensor):
    """Per-kv-head scaled E4M3 codes for a pool ``x`` [NB, Hkv, bs, D] (float32).

    scale_h = amax over head h / 448; stored code = E4M3(x / scale_h), produced by
    torch's float8 cast (used here only to manufacture input data)."""
    amax = x.abs().amax(dim=(0, 2, 3)).clamp_min(1e-12)
    scale = (amax / 448.0).to(torch.float32)
    codes = (x / scale.view(1, -1, 1, 1)).clamp(-448.0, 448.0).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8), scale


@dataclass
class DecodeInputs:
    """One paged-decode batch (all CPU tensors)."""
    q: torch.Tensor                 # [B, Hq, D] bf16
    k_cache: torch.Tensor           # [NB, Hkv, bs, D] bf16 or uint8 (E4M3 codes)
    v_cache: torch.Tensor
    block_tables: torch.Tensor      # [B, max_blocks] int32, -1 = unallocated
    context_lens: torch.Tensor      # [B] int32
    scale: float
    cache_dtype: str = "bf16"       # "bf16" | "e4m3"
    k_scale: Optional[torch.Tensor] = None   # [Hkv] float32 (E4M3 only)
    v_scale: Optional[torch.Tensor] = None
    # the new token of this decode step, appended at position context_len - 1
    step_key: Optional[torch.Tensor] = None    # [B, Hkv, D] bf16
    step_value: Optional[torch.Tensor] = None
    step_slots: Optional[torch.Tensor] = None  # [B] int64
    # extra block-table sets over disjoint physical blocks (same context lens)
    rotations: List[torch.Tensor] = field(default_factory=list)
    rotation_slots: List[torch.Tensor] = field(default_factory=list)
    name: str = ""

    @property
    def num_seqs(self):
        return self.q.shape[0]

    @property
    def num_q_heads(self):
        return self.q.shape[1]

    @property
    def head_dim(self):
        return self.q.shape[2]

    @property
    def num_kv_heads(self):
        return self.k_cache.shape[1]

    @property
    def num_blocks(self):
        return self.k_cache.shape[0]

    @property
    def block_size(self):
        return self.k_cache.shape[2]

    @property
    def max_context_len(self):
        return int(self.context_lens.max().item()) if self.context_lens.numel() else 0


@dataclass
class PrefillInputs:
    """One varlen causal prefill batch (all CPU tensors)."""
    q: torch.Tensor               # [T, Hq, D] bf16
    key: torch.Tensor             # [T, Hkv, D] bf16 (to be written into the cache)
    value: torch.Tensor
    slot_mapping: torch.Tensor    # [T] int64
    cu_seqlens: torch.Tensor      # [S + 1] int32
    block_tables: torch.Tensor    # [S, max_blocks] int32, -1 = unallocated
    k_cache: torch.Tensor         # [NB, Hkv, bs, D] bf16, initial (pre-write) contents
    v_cache: torch.Tensor
    scale: float
    name: str = ""

    @property
    def num_seqs(self):
        return self.cu_seqlens.numel() - 1

    @property
    def seq_lens(self):
        return (self.cu_seqlens[1:] - self.cu_seqlens[:-1]).tolist()

    @property
    def max_seqlen(self):
        return max(self.seq_lens) if self.num_seqs else 0


@dataclass
class ChunkedPrefillInputs:
    """A prefill over a cached prefix (all CPU tensors): sequence i has Lk = seq_lens_k[i]
    tokens, the last Lq of which are the new chunk (cu_seqlens_q); key/value hold all
    Lk tokens of every sequence, written into the cache through slot_mapping."""
    q: torch.Tensor               # [Tq, Hq, D] bf16, the chunks' queries
    key: torch.Tensor             # [Tk, Hkv, D] bf16, every cached token
    value: torch.Tensor
    slot_mapping: torch.Tensor    # [Tk] int64
    cu_seqlens_q: torch.Tensor    # [S + 1] int32
    seq_lens_k: torch.Tensor      # [S] int32
    block_tables: torch.Tensor    # [S, max_blocks] int32
    k_cache: torch.Tensor         # [NB, Hkv, bs, D] bf16, initial (pre-write) contents
    v_cache: torch.Tensor
    scale: float
    name: str = ""

    @property
    def num_seqs(self):
        return self.cu_seqlens_q.numel() - 1

    @property
    def lens_q(self):
        return (self.cu_seqlens_q[1:] - self.cu_seqlens_q[:-1]).tolist()

    @property
    def max_seqlen_q(self):
        return max(self.lens_q) if self.num_seqs else 0

    @property
    def max_seqlen_k(self):
        return int(self.seq_lens_k.max()) if self.num_seqs else 0


def _blocks_needed(L: int, bs: int) -> int:
    return (L + bs - 1) // bs


def _assign_tables(context_lens: Sequence[int], perm: torch.Tensor, start: int, bs: int,
                   max_blocks: int, prefix_group: int = 0, prefix_tokens: int = 0):
    """Block tables taking physical ids from ``perm`` in order, starting at
    ``start``. With prefix_group > 0, each run of ``prefix_group`` sequences shares
    the blocks of its first ``prefix_tokens`` tokens (copy-on-write sharing)."""
    B = len(context_lens)
    table = torch.full((B, max_blocks), -1, dtype=torch.int32)
    pos = start
    shared = None
    for b, L in enumerate(context_lens):
        n = _blocks_needed(L, bs)
        first = 0
        if prefix_group > 0:
            n_shared = prefix_tokens // bs
            if b % prefix_group == 0:
                shared = perm[pos:pos + n_shared].to(torch.int32)
                pos += n_shared
            table[b, :n_shared] = shared
            first = n_shared
        table[b, first:n] = perm[pos:pos + (n - first)].to(torch.int32)
        pos += n - first
    return table, pos


def _slots_for_positions(table: torch.Tensor, positions: Sequence[int], bs: int) -> torch.Tensor:
    slots = torch.empty(len(positions), dtype=torch.int64)
    for b, p in enumerate(positions):
        slots[b] = int(table[b, p // bs]) * bs + p % bs
    return slots


def _used_rows(tables: Sequence[torch.Tensor], lens: Sequence[int], bs: int):
    """{physical block: number of leading rows holding context} over all tables."""
    used = {}
    for table in tables:
        for b, L in enumerate(lens):
            for j in range(_blocks_needed(L, bs)):
                pbn = int(table[b, j])
                used[pbn] = max(used.get(pbn, 0), min(bs, L - j * bs))
    return used


def _fill_pool(shape, used: dict, g: torch.Generator, cache_dtype: str):
    """A pool whose referenced rows are N(0,1) draws and whose every other element
    is NaN (so a read outside a context poisons the result)."""
    nb, hkv, bs, d = shape
    blocks = sorted(used)
    idx = torch.tensor(blocks, dtype=torch.int64)
    rows = torch.tensor([used[b] for b in blocks], dtype=torch.int64)
    x = torch.randn((len(blocks), hkv, bs, d), generator=g, dtype=torch.float32)
    keep = (torch.arange(bs).view(1, 1, bs, 1) < rows.view(-1, 1, 1, 1))
    if cache_dtype == "bf16":
        pool = torch.full(shape, float("nan"), dtype=torch.bfloat16)
        pool[idx] = torch.where(keep, x, torch.nan).to(torch.bfloat16)
        return pool, None
    codes, scale = e4m3_encode_with_scale(torch.where(keep, x, 0.0))
    codes = torch.where(keep, codes, torch.tensor(0x7F, dtype=torch.uint8))
    pool = torch.full(shape, 0x7F, dtype=torch.uint8)
    pool[idx] = codes
    return pool, scale


def make_decode(context_lens: Sequence[int], num_q_heads: int, num_kv_heads: int, head_dim: int,
                num_blocks: int, seed: int, cache_dtype: str = "bf16", block_size: int = BLOCK_SIZE,
                prefix_group: int = 0, prefix_tokens: int = 0, rotations: int = 0,
                max_blocks: Optional[int] = None, name: str = "") -> DecodeInputs:
    if cache_dtype not in ("bf16", "e4m3"):
        raise ValueError(cache_dtype)
    g = _gen(seed)
    B = len(context_lens)
    need = max([_blocks_needed(L, block_size) for L in context_lens] + [1])
    max_blocks = max_blocks or need
    perm = torch.randperm(num_blocks, generator=g)
    tables = []
    pos = 0
    for _ in range(rotations + 1):
        t, pos = _assign_tables(context_lens, perm, pos, block_size, max_blocks, prefix_group,
                                prefix_tokens)
        if pos > num_blocks:
            raise ValueError("block pool too small")
        tables.append(t)
    used = _used_rows(tables, context_lens, block_size)
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    q = _randn_bf16((B, num_q_heads, head_dim), g)
    k_cache, k_scale = _fill_pool(shape, used, g, cache_dtype)
    v_cache, v_scale = _fill_pool(shape, used, g, cache_dtype)
    step_key = _randn_bf16((B, num_kv_heads, head_dim), g)
    step_value = _randn_bf16((B, num_kv_heads, head_dim), g)
    positions = [L - 1 for L in context_lens]
    inp = DecodeInputs(q=q, k_cache=k_cache, v_cache=v_cache, block_tables=tables[0],
                       context_lens=torch.tensor(list(context_lens), dtype=torch.int32),
                       scale=1.0 / math.sqrt(head_dim), cache_dtype=cache_dtype,
                       k_scale=k_scale, v_scale=v_scale, step_key=step_key,
                       step_value=step_value, name=name)
    if all(L > 0 for L in context_lens):
        inp.step_slots = _slots_for_positions(tables[0], positions, block_size)
        for t in tables[1:]:
            inp.rotations.append(t)
            inp.rotation_slots.append(_slots_for_positions(t, positions, block_size))
    return inp


def make_prefill(seq_lens: Sequence[int], num_q_heads: int, num_kv_heads: int, head_dim: int,
                 num_blocks: int, seed: int, block_size: int = BLOCK_SIZE,
                 name: str = "") -> PrefillInputs:
    """The cache starts as all-NaN: after the writes, only the rows the sequences
    own hold data, so a read of anything else poisons the result."""
    g = _gen(seed)
    S = len(seq_lens)
    T = int(sum(seq_lens))
    cu = torch.zeros(S + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(list(seq_lens), dtype=torch.int64), 0).to(torch.int32)
    q = _randn_bf16((T, num_q_heads, head_dim), g)
    key = _randn_bf16((T, num_kv_heads, head_dim), g)
    value = _randn_bf16((T, num_kv_heads, head_dim), g)
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    k_cache = torch.full(shape, float("nan"), dtype=torch.bfloat16)
    v_cache = torch.full(shape, float("nan"), dtype=torch.bfloat16)
    perm = torch.randperm(num_blocks, generator=g)
    max_blocks = max([_blocks_needed(L, block_size) for L in seq_lens] + [1])
    table, used = _assign_tables(seq_lens, perm, 0, block_size, max_blocks)
    if used > num_blocks:
        raise ValueError("block pool too small")
    slots = torch.empty(T, dtype=torch.int64)
    for i, L in enumerate(seq_lens):
        base = int(cu[i])
        p = torch.arange(L, dtype=torch.int64)
        slots[base:base + L] = table[i, p // block_size].to(torch.int64) * block_size + p % block_size
    return PrefillInputs(q=q, key=key, value=value, slot_mapping=slots, cu_seqlens=cu,
                         block_tables=table, k_cache=k_cache, v_cache=v_cache,
                         scale=1.0 / math.sqrt(head_dim), name=name)


def make_chunked_prefill(lens_k: Sequence[int], lens_q: Sequence[int], num_q_heads: int,
                         num_kv_heads: int, head_dim: int, num_blocks: int, seed: int,
                         block_size: int = BLOCK_SIZE, name: str = "") -> ChunkedPrefillInputs:
    """Sequence i caches lens_k[i] tokens; its new chunk is the last lens_q[i] of them.
    The cache starts all-NaN, so a read of a row no sequence owns poisons the result."""
    assert len(lens_k) == len(lens_q) and all(0 <= q <= k for k, q in zip(lens_k, lens_q))
    g = _gen(seed)
    S = len(lens_k)
    Tk, Tq = int(sum(lens_k)), int(sum(lens_q))
    cu = torch.zeros(S + 1, dtype=torch.int32)
    cu[1:] = torch.cumsum(torch.tensor(list(lens_q), dtype=torch.int64), 0).to(torch.int32)
    q = _randn_bf16((Tq, num_q_heads, head_dim), g)
    key = _randn_bf16((Tk, num_kv_heads, head_dim), g)
    value = _randn_bf16((Tk, num_kv_heads, head_dim), g)
    shape = (num_blocks, num_kv_heads, block_size, head_dim)
    k_cache = torch.full(shape, float("nan"), dtype=torch.bfloat16)
    v_cache = torch.full(shape, float("nan"), dtype=torch.bfloat16)
    perm = torch.randperm(num_blocks, generator=g)
    max_blocks = max([_blocks_needed(L, block_size) for L in lens_k] + [1])
    table, used = _assign_tables(lens_k, perm, 0, block_size, max_blocks)
    if used > num_blocks:
        raise ValueError("block pool too small")
    slots = torch.empty(Tk, dtype=torch.int64)
    base = 0
    for i, L in enumerate(lens_k):
        p = torch.arange(L, dtype=torch.int64)
        slots[base:base + L] = table[i, p // block_size].to(torch.int64) * block_size + p % block_size
        base += L
    return ChunkedPrefillInputs(q=q, key=key, value=value, slot_mapping=slots, cu_seqlens_q=cu,
                                seq_lens_k=torch.tensor(list(lens_k), dtype=torch.int32),
                                block_tables=table, k_cache=k_cache, v_cache=v_cache,
                                scale=1.0 / math.sqrt(head_dim), name=name)


def e4m3_prefill_cache(inp):
    """An E4M3 cache for a prefill batch (PrefillInputs or ChunkedPrefillInputs): K and
    V pools of the batch's shape filled with the NaN code 0x7F (so a read of a row no
    sequence owns poisons the result) and per-kv-head scales amax / 448 over the
    tokens the batch writes (K and V separately). Returns (k_cache, v_cache,
    k_scale, v_scale); the codes themselves come from the cache write."""
    shape = tuple(inp.k_cache.shape)
    k_cache = torch.full(shape, 0x7F, dtype=torch.uint8)
    v_cache = torch.full(shape, 0x7F, dtype=torch.uint8)
    scale = lambda x: (x.float().abs().amax(dim=(0, 2)).clamp_min(1e-12) / 448.0).float()
    return k_cache, v_cache, scale(inp.key), scale(inp.value)


def _pool_for(lens: Sequence[int], base: int, rotations: int, bs: int = BLOCK_SIZE) -> int:
    """Smallest pool (a multiple of 1024 blocks, at least ``base``) that holds
    ``rotations + 1`` disjoint copies of the tables for ``lens``."""
    need = sum(_blocks_needed(L, bs) for L in lens) * (rotations + 1)
    return max(base, -(-need // 1024) * 1024)


def _uniform_lens(n: int, lo: int, hi: int, seed: int) -> List[int]:
    g = _gen(seed)
    return torch.randint(lo, hi + 1, (n,), generator=g).tolist()


# ----------------------------------------------------------------- presets
# Seed 0 plus a per-workload offset.

def tiny_decode(seed: int = 0) -> DecodeInputs:
    """batch 2, 4 query / 2 kv heads, head_dim 64, contexts {37, 50}, a pool of
    16 blocks assigned by a seeded permutation."""
    return make_decode([37, 50], 4, 2, 64, 16, seed + 1, name="tiny decode B2 Hq4 Hkv2 D64")


def llama3_8b_decode(seed: int = 0, rotations: int = 0) -> DecodeInputs:
    """batch 64, 32 query / 8 kv heads, head_dim 128, contexts uniform on
    [256, 1024], physical blocks shuffled from an 8192-block pool."""
    lens = _uniform_lens(64, 256, 1024, seed + 2)
    return make_decode(lens, 32, 8, 128, 8192, seed + 2, rotations=rotations,
                       name="Llama-3-8B decode B64 Hq32 Hkv8 D128 ctx U[256,1024]")


def llama70b_decode(seed: int = 0, cache_dtype: str = "bf16", rotations: int = 0) -> DecodeInputs:
    """batch 32, 64 query / 8 kv heads, head_dim 128, contexts uniform on
    [1024, 4096], shuffled blocks; bf16 or E4M3 cache with per-kv-head scales."""
    lens = _uniform_lens(32, 1024, 4096, seed + 3)
    nb = _pool_for(lens, 8192, rotations)
    return make_decode(lens, 64, 8, 128, nb, seed + 3, cache_dtype=cache_dtype,
                       rotations=rotations,
                       name=f"70B decode B32 Hq64 Hkv8 D128 ctx U[1024,4096] {cache_dtype}")


def varlen_prefill(seed: int = 0) -> PrefillInputs:
    """16 sequences, lengths uniform on [128, 2048], 32 query / 8 kv heads,
    head_dim 128, written into a shuffled 2048-block pool via slot_mapping."""
    lens = _uniform_lens(16, 128, 2048, seed + 4)
    return make_prefill(lens, 32, 8, 128, 2048, seed + 4,
                        name="varlen causal prefill 16 seqs L U[128,2048] Hq32 Hkv8 D128")


def chunked_prefill(seed: int = 0) -> ChunkedPrefillInputs:
    """Prefill over a cached prefix: 16 sequences with a cached prefix uniform on
    [512, 3584] tokens and a new chunk uniform on [128, 512], 32 query / 8 kv heads,
    head_dim 128, a shuffled 4096-block pool."""
    prefix = _uniform_lens(16, 512, 3584, seed + 6)
    chunk = _uniform_lens(16, 128, 512, seed + 7)
    lens_k = [a + b for a, b in zip(prefix, chunk)]
    return make_chunked_prefill(lens_k, chunk, 32, 8, 128, 4096, seed + 6,
                                name="chunked prefill 16 seqs prefix U[512,3584] + chunk "
                                     "U[128,512] Hq32 Hkv8 D128")


def speculative_verify(seed: int = 0, draft: int = 5) -> ChunkedPrefillInputs:
    """Speculative verification: batch 64, contexts uniform on [256, 1024] (the last
    `draft` tokens are the drafts being checked), 32 query / 8 kv heads, head_dim 128."""
    lens_k = _uniform_lens(64, 256, 1024, seed + 8)
    return make_chunked_prefill(lens_k, [draft] * 64, 32, 8, 128, 8192, seed + 8,
                                name=f"speculative verification B64 ctx U[256,1024] "
                                     f"{draft} tokens/seq Hq32 Hkv8 D128")


def prefix_sharing_decode(seed: int = 0, rotations: int = 0) -> DecodeInputs:
    """batch 16, context 8192, 32 query / 8 kv heads, head_dim 128; each group of
    4 sequences shares the physical blocks of its first 4096 tokens."""
    nb = max(8192, 5120 * (rotations + 1))
    return make_decode([8192] * 16, 32, 8, 128, nb, seed + 5, prefix_group=4,
                       prefix_tokens=4096, rotations=rotations,
                       name="prefix-sharing decode B16 ctx8192 Hq32 Hkv8 D128 groups of 4")


def kv_read_bytes(inp: DecodeInputs, unique: bool = False) -> int:
    """Algorithmic KV bytes one decode pass reads: every cached token of every
    kv-head, K and V, once. unique=True counts shared physical blocks once."""
    elem = 1 if inp.cache_dtype == "e4m3" else 2
    row = inp.num_kv_heads * inp.head_dim * elem * 2
    if not unique:
        return int(inp.context_lens.to(torch.int64).sum().item()) * row
    seen = {}
    bs = inp.block_size
    for b, L in enumerate(inp.context_lens.tolist()):
        for j in range(_blocks_needed(L, bs)):
            pbn = int(inp.block_tables[b, j])
            rows = min(bs, L - j * bs)
            seen[pbn] = max(seen.get(pbn, 0), rows)
    return sum(seen.values()) * row


def chunked_flops(inp: "ChunkedPrefillInputs") -> int:
    """Useful FLOPs of a prefill over a cached prefix: chunk position p attends to
    Lk - Lq + p + 1 keys (QK^T and PV, 2 flops per multiply-add each)."""
    Hq, D = inp.q.shape[1], inp.q.shape[2]
    total = 0
    for Lq, Lk in zip(inp.lens_q, inp.seq_lens_k.tolist()):
        pairs = Lq * (Lk - Lq) + Lq * (Lq + 1) // 2
        total += 4 * Hq * D * pairs
    return total


def chunked_kv_bytes(inp: "ChunkedPrefillInputs") -> int:
    """K and V bytes of every cached key of every sequence, read once per kv-head."""
    Hkv, D = inp.key.shape[1], inp.key.shape[2]
    return int(inp.seq_lens_k.sum()) * Hkv * D * 2 * 2


def causal_flops(seq_lens: Sequence[int], num_q_heads: int, head_dim: int) -> int:
    """Useful FLOPs of causal prefill: 2 matmuls x 2 flop per multiply-add over the
    unmasked (query, key) pairs, L(L+1)/2 per sequence and query head."""
    return int(sum(4 * num_q_heads * head_dim * L * (L + 1) // 2 for L in seq_lens))
