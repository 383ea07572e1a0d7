"""Seeded synthetic inputs for the paged-KV hot path.

This module is shared by the oracle tests, the GPU parity tests, ``bench.py``
and ``__graft_entry__.smoke``.  It holds no attention or store arithmetic: it
only plays the part of the engine's runner, turning per-sequence block tables
into the tensors the attention layer receives (slot mappings, -1 padded block
tables, context lengths and cumulative sequence lengths), and it fills the
paged pool with random values.

Runner steps restated here (from "nano-vLLM Part 2: Block Tables, KV Cache, and
the Path to the GPU"):

* position -> slot: ``block_table[p // bs] * bs + p % bs`` (section 2.2);
* the prefill slot loop over the scheduled range ``[start, end)``, first-page
  offset and last-page end (section 2.2, ``prepare_prefill``);
* the decode slot of the last token (section 3.1, ``prepare_decode``);
* padding block tables with -1 (section 3.2, ``prepare_block_tables``);
* ``cu_seqlens_q`` / ``cu_seqlens_k`` as cumulative query and context
  lengths (section 4.1).

Workload recipe (all values drawn from one ``torch.Generator`` seeded with the
workload's index): q, new k/v and every cached token are N(0, 1) cast to the
workload dtype; unused pool rows hold the NaN sentinel 0x7FC1 so that a stray
read poisons the result; physical block ids are ``randperm(pool)[:need]``
assigned in logical order.  An fp8 pool (``make_decode_fp8``) holds the E4M3
codes of N(0, 1) values over per-tensor scales 4/448 (K) and 3/448 (V), made
by torch's float8_e4m3fn cast, and the NaN code 0x7F in unused rows.
"""

from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch

SENTINEL_BITS = 0x7FC1  # a quiet NaN in both bf16 and fp16


# ---------------------------------------------------------------------------
# Runner-side index preparation (pinned by the pages' worked examples)
# ---------------------------------------------------------------------------

def slot_of(block_table, block_size: int, position: int) -> int:
    """Flattened cache slot of logical ``position`` (page 1, section 2.2)."""
    page = block_table[position // block_size]
    return page * block_size + position % block_size


def slots_for_range(block_table, block_size: int, start: int, end: int) -> list[int]:
    """Slots of the scheduled token range ``[start, end)``.

    Walks the pages the range touches; the first page starts at
    ``start % bs`` and the last page stops at ``end`` (page 1, section 2.2 and
    page 2, "Prepare Prefill").
    """
    out: list[int] = []
    if end <= start:
        return out
    first = start // block_size
    last = (end + block_size - 1) // block_size
    for i in range(first, last):
        base = block_table[i] * block_size
        lo = base + (start % block_size if i == first else 0)
        hi = base + (end - i * block_size if i == last - 1 else block_size)
        out.extend(range(lo, hi))
    return out


def decode_slot(block_table, block_size: int, seq_len: int) -> int:
    """Slot of the last token of a length-``seq_len`` sequence (page 1, section 3.1)."""
    return block_table[-1] * block_size + (seq_len - 1) % block_size


def pad_block_tables(tables, width: int | None = None) -> torch.Tensor:
    """Batch per-sequence block tables into an int32 matrix padded with -1 (page 1, section 3.2)."""
    width = max((len(t) for t in tables), default=0) if width is None else width
    out = torch.full((len(tables), max(width, 1)), -1, dtype=torch.int32)
    for i, t in enumerate(tables):
        if len(t):
            out[i, : len(t)] = torch.tensor(t, dtype=torch.int32)
    return out


def cu_seqlens(lengths) -> torch.Tensor:
    """Cumulative lengths ``[0, l0, l0+l1, ...]`` as int32 (page 1, section 4.1)."""
    out = [0]
    for n in lengths:
        out.append(out[-1] + int(n))
    return torch.tensor(out, dtype=torch.int32)


def num_pages(tokens: int, block_size: int) -> int:
    return (tokens + block_size - 1) // block_size


# ---------------------------------------------------------------------------
# Pool construction
# ---------------------------------------------------------------------------

@dataclass
class SeqSpec:
    """One sequence of a step: ``cached`` tokens already in the pool, ``new``
    tokens computed this step (stored via slot_mapping).  Sequences with the
    same ``share_group`` share the physical blocks of their first
    ``share_tokens`` tokens (a common prefix; must be whole pages)."""

    cached: int
    new: int
    share_group: int = -1
    share_tokens: int = 0


@dataclass
class Pool:
    dtype: torch.dtype
    num_blocks: int
    block_size: int
    num_kv_heads: int
    head_dim: int
    k_cache: torch.Tensor  # [N, bs, H_kv, D], pre-store contents
    v_cache: torch.Tensor
    tables: list  # per-sequence physical block ids, logical order
    specs: list


def _sentinel_pool(n, bs, hkv, d, dtype) -> torch.Tensor:
    t = torch.full((n, bs, hkv, d), SENTINEL_BITS, dtype=torch.int16)
    return t.view(dtype)


def build_pool(specs: list[SeqSpec], *, block_size: int, num_kv_heads: int, head_dim: int,
               dtype: torch.dtype, gen: torch.Generator, num_blocks: int | None = None,
               pool_factor: float = 1.25) -> Pool:
    """Assign physical blocks to every sequence and fill the cached tokens.

    Block ids come from one seeded ``randperm`` over the pool, taken in
    logical order; shared prefix pages are allocated once per group.
    """
    bs = block_size
    need = 0
    group_pages: dict[int, int] = {}
    for s in specs:
        total = num_pages(s.cached + s.new, bs)
        if s.share_group >= 0:
            assert s.share_tokens % bs == 0 and s.share_tokens <= s.cached
            sp = s.share_tokens // bs
            if s.share_group not in group_pages:
                group_pages[s.share_group] = sp
                need += sp
            need += total - sp
        else:
            need += total
    if num_blocks is None:
        num_blocks = max(1, math.ceil(pool_factor * need))
    assert num_blocks >= need, (num_blocks, need)
    perm = torch.randperm(num_blocks, generator=gen)[:need].tolist()
    cursor = 0
    group_ids: dict[int, list[int]] = {}
    tables = []
    for s in specs:
        total = num_pages(s.cached + s.new, bs)
        t: list[int] = []
        if s.share_group >= 0:
            sp = s.share_tokens // bs
            if s.share_group not in group_ids:
                group_ids[s.share_group] = perm[cursor: cursor + sp]
                cursor += sp
            t.extend(group_ids[s.share_group])
        while len(t) < total:
            t.append(perm[cursor])
            cursor += 1
        tables.append(t)

    k_cache = _sentinel_pool(num_blocks, bs, num_kv_heads, head_dim, dtype)
    v_cache = _sentinel_pool(num_blocks, bs, num_kv_heads, head_dim, dtype)
    rows = []
    for s, t in zip(specs, tables):
        if s.cached == 0:
            continue
        pos = torch.arange(s.cached)
        tt = torch.tensor(t, dtype=torch.int64)
        rows.append(tt[pos // bs] * bs + pos % bs)
    if rows:
        rows = torch.unique(torch.cat(rows))  # shared prefix rows filled once
        n = rows.numel()
        kf = k_cache.view(num_blocks * bs, num_kv_heads, head_dim)
        vf = v_cache.view(num_blocks * bs, num_kv_heads, head_dim)
        kf[rows] = torch.randn(n, num_kv_heads, head_dim, generator=gen).to(dtype)
        vf[rows] = torch.randn(n, num_kv_heads, head_dim, generator=gen).to(dtype)
    return Pool(dtype, num_blocks, bs, num_kv_heads, head_dim, k_cache, v_cache, tables, specs)


# ---------------------------------------------------------------------------
# Step inputs
# ---------------------------------------------------------------------------

@dataclass
class DecodeStep:
    """One decode step: store one token per sequence, then attend over the
    sequence's whole context (which includes that token, page 1, section 3.1)."""

    pool: Pool
    num_q_heads: int
    q: torch.Tensor            # [B, H_q, D]
    k_new: torch.Tensor        # [B, H_kv, D]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor  # int32 [B]
    block_tables: torch.Tensor  # int32 [B, max_blocks], -1 padded
    context_lens: torch.Tensor  # int32 [B]
    scale: float

    @property
    def batch(self) -> int:
        return self.q.shape[0]

    def kv_bytes(self) -> int:
        """Algorithmic K+V bytes the attention reads: sum(ctx) * 2 * H_kv * D * elem
        (the per-token cache size of page 2, Step 5)."""
        p = self.pool
        return int(self.context_lens.sum()) * 2 * p.num_kv_heads * p.head_dim * self.q.element_size()

    def unique_kv_bytes(self) -> int:
        """K+V bytes counting each physical row once (shared prefixes read once)."""
        p = self.pool
        rows = set()
        for t, L in zip(p.tables, self.context_lens.tolist()):
            for j in range(num_pages(L, p.block_size)):
                n = min(p.block_size, L - j * p.block_size)
                rows.add((t[j], n))
        per_page: dict[int, int] = {}
        for page, n in rows:
            per_page[page] = max(per_page.get(page, 0), n)
        return sum(per_page.values()) * 2 * p.num_kv_heads * p.head_dim * self.q.element_size()


@dataclass
class PrefillStep:
    """Chunked prefill: each sequence has ``cached`` tokens in the pool and a
    chunk of new query tokens that attend causally over prefix + chunk."""

    pool: Pool
    num_q_heads: int
    q: torch.Tensor            # [Tq, H_q, D]
    k_new: torch.Tensor        # [Tq, H_kv, D]
    v_new: torch.Tensor
    slot_mapping: torch.Tensor  # int32 [Tq]
    cu_seqlens_q: torch.Tensor  # int32 [S+1]
    cu_seqlens_k: torch.Tensor  # int32 [S+1]
    block_tables: torch.Tensor | None
    max_seqlen_q: int
    max_seqlen_k: int
    scale: float

    def flops(self) -> int:
        """Causal QK^T + PV flops, masked work excluded: per q head and query
        row r of a sequence with prefix P, 4*D*(P + r + 1)."""
        H, D = self.num_q_heads, self.q.shape[2]
        tot = 0
        cq, ck = self.cu_seqlens_q.tolist(), self.cu_seqlens_k.tolist()
        for i in range(len(cq) - 1):
            lq, lk = cq[i + 1] - cq[i], ck[i + 1] - ck[i]
            p = lk - lq
            tot += lq * p + lq * (lq + 1) // 2
        return 4 * D * H * tot


def _decode_from_pool(pool: Pool, ctx: list[int], num_q_heads: int, gen, scale=None) -> DecodeStep:
    B, hkv, d, dt = len(ctx), pool.num_kv_heads, pool.head_dim, pool.dtype
    q = torch.randn(B, num_q_heads, d, generator=gen).to(dt)
    k_new = torch.randn(B, hkv, d, generator=gen).to(dt)
    v_new = torch.randn(B, hkv, d, generator=gen).to(dt)
    slots = [decode_slot(t, pool.block_size, L) if L > 0 else -1 for t, L in zip(pool.tables, ctx)]
    width = max(num_pages(L, pool.block_size) for L in ctx) if ctx else 1
    return DecodeStep(pool, num_q_heads, q, k_new, v_new,
                      torch.tensor(slots, dtype=torch.int32),
                      pad_block_tables(pool.tables, max(width, 1)),
                      torch.tensor(ctx, dtype=torch.int32),
                      scale if scale is not None else 1.0 / math.sqrt(d))


def make_decode_shared(seqs: list[tuple[int, int, int]], *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                       block_size: int, dtype: torch.dtype, seed: int, num_blocks: int | None = None) -> DecodeStep:
    """Decode step over sequences given as (context length, share group or -1, shared tokens):
    the members of a share group point at the same physical pages for their first shared
    tokens (whole pages, below every member's context length); -1 shares nothing."""
    gen = torch.Generator().manual_seed(seed)
    specs = []
    for L, grp, share in seqs:
        if L == 0:
            specs.append(SeqSpec(0, 0))
        else:
            specs.append(SeqSpec(L - 1, 1, grp, share if grp >= 0 else 0))
    pool = build_pool(specs, block_size=block_size, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      dtype=dtype, gen=gen, num_blocks=num_blocks)
    return _decode_from_pool(pool, [L for L, _, _ in seqs], num_q_heads, gen)


def next_decode_step(st: DecodeStep, seed: int) -> DecodeStep:
    """The decode step after ``st`` over the same pool and block tables: each sequence
    gains one token while its last allocated page has room (else keeps its length),
    with new random q and new K/V rows stored at the slot of its new last position."""
    p = st.pool
    gen = torch.Generator().manual_seed(seed)
    ctx = [L + 1 if 0 < L < len(t) * p.block_size else L for t, L in zip(p.tables, st.context_lens.tolist())]
    B, hkv, d = len(ctx), p.num_kv_heads, p.head_dim
    q = torch.randn(B, st.num_q_heads, d, generator=gen).to(st.q.dtype)
    k_new = torch.randn(B, hkv, d, generator=gen).to(st.q.dtype)
    v_new = torch.randn(B, hkv, d, generator=gen).to(st.q.dtype)
    slots = [decode_slot(t, p.block_size, L) if L > 0 else -1 for t, L in zip(p.tables, ctx)]
    return DecodeStep(p, st.num_q_heads, q, k_new, v_new, torch.tensor(slots, dtype=torch.int32),
                      st.block_tables.clone(), torch.tensor(ctx, dtype=torch.int32), st.scale)


def make_decode(ctx: list[int], *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                block_size: int, dtype: torch.dtype, seed: int, num_blocks: int | None = None,
                share_groups: int = 0, share_tokens: int = 0, scale=None) -> DecodeStep:
    """Decode step over sequences of the given context lengths (each length
    includes the token stored this step).  With ``share_groups = g > 0``,
    consecutive runs of ``g`` sequences share their first ``share_tokens``
    tokens' pages."""
    gen = torch.Generator().manual_seed(seed)
    specs = []
    for i, L in enumerate(ctx):
        if L == 0:
            specs.append(SeqSpec(0, 0))
        elif share_groups:
            specs.append(SeqSpec(L - 1, 1, i // share_groups, share_tokens))
        else:
            specs.append(SeqSpec(L - 1, 1))
    pool = build_pool(specs, block_size=block_size, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      dtype=dtype, gen=gen, num_blocks=num_blocks)
    return _decode_from_pool(pool, ctx, num_q_heads, gen, scale)


def make_prefill(prefix: list[int], chunk: list[int], *, num_q_heads: int, num_kv_heads: int,
                 head_dim: int, block_size: int, dtype: torch.dtype, seed: int,
                 num_blocks: int | None = None, extra_specs: list[SeqSpec] | None = None,
                 gen: torch.Generator | None = None, scale=None):
    """Chunked-prefill step: sequence i has ``prefix[i]`` cached tokens and
    ``chunk[i]`` new ones.  ``extra_specs`` adds sequences (e.g. decode rows of
    a mixed step) to the same pool; their tables follow the prefill ones."""
    gen = gen or torch.Generator().manual_seed(seed)
    specs = [SeqSpec(p, c) for p, c in zip(prefix, chunk)] + list(extra_specs or [])
    pool = build_pool(specs, block_size=block_size, num_kv_heads=num_kv_heads, head_dim=head_dim,
                      dtype=dtype, gen=gen, num_blocks=num_blocks)
    S = len(prefix)
    tq = sum(chunk)
    q = torch.randn(tq, num_q_heads, head_dim, generator=gen).to(dtype)
    k_new = torch.randn(tq, num_kv_heads, head_dim, generator=gen).to(dtype)
    v_new = torch.randn(tq, num_kv_heads, head_dim, generator=gen).to(dtype)
    slots = []
    for i in range(S):
        slots.extend(slots_for_range(pool.tables[i], block_size, prefix[i], prefix[i] + chunk[i]))
    width = max(num_pages(p + c, block_size) for p, c in zip(prefix, chunk))
    step = PrefillStep(pool, num_q_heads, q, k_new, v_new,
                       torch.tensor(slots, dtype=torch.int32),
                       cu_seqlens(chunk), cu_seqlens([p + c for p, c in zip(prefix, chunk)]),
                       pad_block_tables(pool.tables[:S], width),
                       max(chunk), max(p + c for p, c in zip(prefix, chunk)),
                       scale if scale is not None else 1.0 / math.sqrt(head_dim))
    return step, gen


# ---------------------------------------------------------------------------
# The named workloads
# ---------------------------------------------------------------------------

@dataclass
class MixedStep:
    """Store of every new token, chunked prefill of some sequences and decode
    of the others, all over one pool."""

    prefill: PrefillStep
    decode: DecodeStep
    slot_mapping: torch.Tensor   # prefill tokens then decode tokens
    k_new: torch.Tensor
    v_new: torch.Tensor


def tiny_decode(seed: int = 1) -> DecodeStep:
    """4 sequences, context {1, 17, 100, 255}, H_q 4, H_kv 2, D 64, fp16,
    block_size 16, 64-block pool."""
    return make_decode([1, 17, 100, 255], num_q_heads=4, num_kv_heads=2, head_dim=64,
                       block_size=16, dtype=torch.float16, seed=seed, num_blocks=64)


def qwen3_0p6b_decode(seed: int = 2, batch: int = 64) -> DecodeStep:
    """Qwen3-0.6B-like layer: batch 64, H_q 16, H_kv 8, D 128, bf16,
    block_size 256, context uniform in [128, 4096], pool 1.25x need."""
    gen = torch.Generator().manual_seed(seed)
    ctx = torch.randint(128, 4097, (batch,), generator=gen).tolist()
    return make_decode(ctx, num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=256,
                       dtype=torch.bfloat16, seed=seed + 1000)


def qwen3_8b_shared_decode(seed: int = 3, batch: int = 256) -> DecodeStep:
    """Qwen3-8B-like GQA: batch 256, H_q 32, H_kv 8, D 128, bf16, block_size 16,
    context uniform in [513, 2048]; groups of 8 share a 512-token prefix."""
    gen = torch.Generator().manual_seed(seed)
    ctx = torch.randint(513, 2049, (batch,), generator=gen).tolist()
    return make_decode(ctx, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                       dtype=torch.bfloat16, seed=seed + 1000, share_groups=8, share_tokens=512)


def long_context_decode(seed: int = 4, batch: int = 4, ctx: int = 32768) -> DecodeStep:
    """Split-K stress: batch 4 x 32768 context, H_q 32, H_kv 8, D 128, bf16,
    block_size 256, 600-block pool."""
    pool = max(600, math.ceil(1.1 * batch * num_pages(ctx, 256)))
    return make_decode([ctx] * batch, num_q_heads=32, num_kv_heads=8, head_dim=128,
                       block_size=256, dtype=torch.bfloat16, seed=seed, num_blocks=pool)


def mixed_chunked_prefill(seed: int = 5, n_prefill: int = 8, chunk: int = 512, n_decode: int = 120,
                          max_prefix: int = 3584) -> MixedStep:
    """8 prefill sequences (512-token chunk over a cached prefix uniform in
    [0, 3584]) plus 120 decode sequences (context uniform in [256, 4096]);
    H_q 32, H_kv 8, D 128, bf16, block_size 256."""
    gen = torch.Generator().manual_seed(seed)
    prefix = torch.randint(0, max_prefix + 1, (n_prefill,), generator=gen).tolist()
    dctx = torch.randint(256, 4097, (n_decode,), generator=gen).tolist()
    extra = [SeqSpec(L - 1, 1) for L in dctx]
    pf, gen = make_prefill(prefix, [chunk] * n_prefill, num_q_heads=32, num_kv_heads=8,
                           head_dim=128, block_size=256, dtype=torch.bfloat16, seed=seed,
                           extra_specs=extra, gen=gen)
    pool = pf.pool
    dec = _decode_from_pool(Pool(pool.dtype, pool.num_blocks, pool.block_size, pool.num_kv_heads,
                                 pool.head_dim, pool.k_cache, pool.v_cache,
                                 pool.tables[n_prefill:], pool.specs[n_prefill:]),
                            dctx, 32, gen)
    return MixedStep(pf, dec, torch.cat([pf.slot_mapping, dec.slot_mapping]),
                     torch.cat([pf.k_new, dec.k_new]), torch.cat([pf.v_new, dec.v_new]))


def store_stress(seed: int = 6, tokens: int = 16384, num_kv_heads: int = 8, head_dim: int = 128,
                 block_size: int = 256, dtype=torch.bfloat16):
    """16384 new tokens (the engine's max batched tokens) stored at distinct
    random slots of a 1.25x pool."""
    gen = torch.Generator().manual_seed(seed)
    nb = math.ceil(1.25 * num_pages(tokens, block_size))
    slots = torch.randperm(nb * block_size, generator=gen)[:tokens].to(torch.int32)
    k = torch.randn(tokens, num_kv_heads, head_dim, generator=gen).to(dtype)
    v = torch.randn(tokens, num_kv_heads, head_dim, generator=gen).to(dtype)
    kc = _sentinel_pool(nb, block_size, num_kv_heads, head_dim, dtype)
    vc = _sentinel_pool(nb, block_size, num_kv_heads, head_dim, dtype)
    return k, v, kc, vc, slots


# ---------------------------------------------------------------------------
# FP8 (E4M3) pools
# ---------------------------------------------------------------------------

FP8_SENTINEL = 0x7F  # an E4M3 NaN code: unused fp8 pool rows
FP8_K_SCALE = 4.0 / 448.0  # per-tensor scales: N(0, 1) values up to 4 (K) and 3 (V) sigma use
FP8_V_SCALE = 3.0 / 448.0  # the whole code range


def random_e4m3_codes(n_rows: int, row: int, scale: float, gen: torch.Generator) -> torch.Tensor:
    """uint8 E4M3 codes of N(0, 1) values divided by ``scale`` (torch's float8_e4m3fn
    cast after clamping to +-448): synthetic contents of an fp8 pool."""
    x = (torch.randn(n_rows, row, generator=gen) / scale).clamp(-448.0, 448.0)
    return x.to(torch.float8_e4m3fn).view(torch.uint8)


@dataclass
class Fp8DecodeStep:
    """A decode step over an E4M3 pool: ``step`` gives q, the new 16-bit k/v rows
    (quantised by the store), slot mapping, tables and lengths; the pools hold codes,
    K = code * k_scale and V = code * v_scale."""

    step: DecodeStep
    k_cache: torch.Tensor  # uint8 [N, bs, H_kv, D], pre-store contents
    v_cache: torch.Tensor
    k_scale: float
    v_scale: float

    def kv_bytes(self) -> int:
        return self.step.kv_bytes() // self.step.q.element_size()

    def unique_kv_bytes(self) -> int:
        return self.step.unique_kv_bytes() // self.step.q.element_size()


def make_decode_fp8(ctx: list[int], *, num_q_heads: int, num_kv_heads: int, head_dim: int, block_size: int,
                    dtype: torch.dtype, seed: int, num_blocks: int | None = None, share_groups: int = 0,
                    share_tokens: int = 0, k_scale: float = FP8_K_SCALE, v_scale: float = FP8_V_SCALE
                    ) -> Fp8DecodeStep:
    """``make_decode``'s step with the pool's cached rows as random E4M3 codes and the
    unused rows as the NaN code."""
    st = make_decode(ctx, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads, head_dim=head_dim,
                     block_size=block_size, dtype=dtype, seed=seed, num_blocks=num_blocks,
                     share_groups=share_groups, share_tokens=share_tokens)
    p = st.pool
    row = num_kv_heads * head_dim
    filled = (p.k_cache.view(torch.int16).view(-1, row) != SENTINEL_BITS).any(dim=1).nonzero().flatten()
    gen = torch.Generator().manual_seed(seed + 7919)
    kc = torch.full((p.num_blocks * block_size, row), FP8_SENTINEL, dtype=torch.uint8)
    vc = torch.full((p.num_blocks * block_size, row), FP8_SENTINEL, dtype=torch.uint8)
    kc[filled] = random_e4m3_codes(filled.numel(), row, k_scale, gen)
    vc[filled] = random_e4m3_codes(filled.numel(), row, v_scale, gen)
    # the 16-bit pool is no longer needed: keep only its geometry and tables
    st.pool = Pool(p.dtype, p.num_blocks, p.block_size, p.num_kv_heads, p.head_dim, torch.empty(0, dtype=dtype),
                   torch.empty(0, dtype=dtype), p.tables, p.specs)
    shape = (p.num_blocks, block_size, num_kv_heads, head_dim)
    return Fp8DecodeStep(st, kc.view(shape), vc.view(shape), k_scale, v_scale)


def qwen3_0p6b_decode_fp8(seed: int = 2, batch: int = 64) -> Fp8DecodeStep:
    """``qwen3_0p6b_decode``'s shapes and lengths over an E4M3 pool."""
    gen = torch.Generator().manual_seed(seed)
    ctx = torch.randint(128, 4097, (batch,), generator=gen).tolist()
    return make_decode_fp8(ctx, num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=256,
                           dtype=torch.bfloat16, seed=seed + 1000)


WORKLOADS = {
    "tiny_decode": tiny_decode,
    "qwen3_0p6b_decode": qwen3_0p6b_decode,
    "qwen3_8b_shared_decode": qwen3_8b_shared_decode,
    "long_context_decode": long_context_decode,
    "mixed_chunked_prefill": mixed_chunked_prefill,
    "qwen3_0p6b_decode_fp8": qwen3_0p6b_decode_fp8,
}
