"""Pins the CPU oracle to things other than itself.

Each ``pin_*`` function takes an oracle library handle and raises on a
mismatch; ``test_oracle_mutants.py`` re-runs them on deliberately broken
copies of the oracle to show that every planted mistake fails at least one.

What pins what:
* store      -- torch ``index_put`` on the flattened cache (library routine);
                rejection of out-of-range slots.
* addressing -- dense, contiguous K/V scattered into a fragmented pool with
                the pinned slot formula; attention must match library attention
                (``scaled_dot_product_attention`` in float64) on the dense data;
                bit-identical output under any relabelling of physical blocks
                and with shared prefix pages versus private copies.
* softmax    -- identical key rows give the mean of V (closed form); one key
                gives v0 exactly; two and three keys match brute force in
                double; an empty context gives zeros.
* prefill    -- no prefix: library causal attention; with a prefix: the last
                Lq rows of library causal attention over the whole contiguous
                sequence (bottom-right alignment); Lq = 1 equals decode.
* dtype      -- fp16/bf16 decoding matches numpy/torch on all 65536 words.
* fp8 cache  -- E4M3 decoding equals torch's float8_e4m3fn on all 256 codes;
                encoding equals torch's rounding (nearest, ties to even) on
                random values and on every midpoint, and saturates at +-448;
                the quantizing store equals torch's conversion of x / scale;
                fp8 decode with power-of-two scales is bit-identical to the
                16-bit decode on the dequantized cache, and matches library
                attention on the dequantized values for any scales.
* sample     -- unit noise gives the first argmax of the logits (closed form);
                scores match a float64 evaluation of the pages' formula except
                at near-ties; scaling logits and temperature by a power of two
                changes nothing; -inf logits never win, T <= 1e-10 gives -1;
                with Exp(1) noise the frequencies follow softmax(z / T)
                (chi-square, the exponential-race theorem of the pages).
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from tests import inputs


# --------------------------------------------------------------- helpers

def _dense_to_pool(dense_k, dense_v, tables, bs, num_blocks, dtype):
    """Scatter per-sequence dense [L, H_kv, D] K/V into a sentinel pool using
    the page formula (pinned by the golden examples)."""
    hkv, d = dense_k[0].shape[1:]
    kc = torch.full((num_blocks, bs, hkv, d), inputs.SENTINEL_BITS, dtype=torch.int16).view(dtype)
    vc = kc.clone()
    kf, vf = kc.view(-1, hkv, d), vc.view(-1, hkv, d)
    for K, V, t in zip(dense_k, dense_v, tables):
        for j in range(K.shape[0]):
            s = inputs.slot_of(t, bs, j)
            kf[s] = K[j]
            vf[s] = V[j]
    return kc, vc


def _lib_attention(q, K, V, scale, causal=False):
    """Library attention in float64: q [H_q, Lq, D], K/V [H_kv, L, D] with
    GQA groups expanded (q head h reads kv head h // G)."""
    g = q.shape[0] // K.shape[0]
    K = K.repeat_interleave(g, dim=0)
    V = V.repeat_interleave(g, dim=0)
    return F.scaled_dot_product_attention(q.double(), K.double(), V.double(), is_causal=causal, scale=scale)


def _random_case(gen, B, hq, hkv, d, bs, ctx, dtype, pool_extra=3):
    need = sum(inputs.num_pages(L, bs) for L in ctx)
    nb = need + pool_extra
    perm = torch.randperm(nb, generator=gen).tolist()
    tables, c = [], 0
    for L in ctx:
        n = inputs.num_pages(L, bs)
        tables.append(perm[c:c + n])
        c += n
    dk = [torch.randn(L, hkv, d, generator=gen).to(dtype) for L in ctx]
    dv = [torch.randn(L, hkv, d, generator=gen).to(dtype) for L in ctx]
    q = torch.randn(B, hq, d, generator=gen).to(dtype)
    return q, dk, dv, tables, nb


# ------------------------------------------------------------------ pins

def pin_store_matches_index_put(lib):
    gen = torch.Generator().manual_seed(11)
    for dtype in (torch.float16, torch.bfloat16):
        T, hkv, d, N, bs = 13, 2, 16, 6, 4
        big = torch.randn(T, 3 * hkv, d, generator=gen).to(dtype)   # k, v as views of a wider row
        k, v = big[:, :hkv], big[:, hkv:2 * hkv]
        slots = torch.randperm(N * bs, generator=gen)[:T].to(torch.int32)
        slots[[2, 7]] = -1
        kc = torch.full((N, bs, hkv, d), inputs.SENTINEL_BITS, dtype=torch.int16).view(dtype)
        vc = kc.clone()
        ek, ev = kc.clone(), vc.clone()
        keep = slots >= 0
        ek.view(N * bs, hkv, d)[slots[keep].long()] = k[keep]
        ev.view(N * bs, hkv, d)[slots[keep].long()] = v[keep]
        oracle.store_kv(k, v, kc, vc, slots, lib=lib)
        assert torch.equal(kc.view(torch.int16), ek.view(torch.int16))
        assert torch.equal(vc.view(torch.int16), ev.view(torch.int16))


def pin_store_rejects_bad_slot(lib):
    k = torch.zeros(2, 1, 8, dtype=torch.bfloat16)
    kc = torch.zeros(2, 4, 1, 8, dtype=torch.bfloat16)
    for bad in (8, -2):
        with pytest.raises(oracle.OracleError):
            oracle.store_kv(k, k, kc.clone(), kc.clone(), torch.tensor([0, bad], dtype=torch.int32), lib=lib)


def pin_decode_vs_library(lib):
    gen = torch.Generator().manual_seed(12)
    for dtype, scale in ((torch.bfloat16, None), (torch.float16, 0.3)):
        B, hq, hkv, d, bs = 5, 8, 2, 32, 4
        ctx = [1, 6, 9, 16, 23]
        q, dk, dv, tables, nb = _random_case(gen, B, hq, hkv, d, bs, ctx, dtype)
        kc, vc = _dense_to_pool(dk, dv, tables, bs, nb, dtype)
        sc = scale if scale is not None else 1.0 / math.sqrt(d)
        out = oracle.decode(q, kc, vc, inputs.pad_block_tables(tables), torch.tensor(ctx, dtype=torch.int32),
                            sc, lib=lib)
        for b in range(B):
            ref = _lib_attention(q[b].float().unsqueeze(1), dk[b].float().transpose(0, 1),
                                 dv[b].float().transpose(0, 1), sc)[:, 0]
            torch.testing.assert_close(out[b].double(), ref, rtol=0, atol=2e-6)


def pin_decode_permutation_invariance(lib):
    st = inputs.make_decode([5, 19, 33, 1], num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=4,
                            dtype=torch.bfloat16, seed=13)
    p = st.pool
    oracle.store_kv(st.k_new, st.v_new, p.k_cache, p.v_cache, st.slot_mapping, lib=lib)
    a = oracle.decode(st.q, p.k_cache, p.v_cache, st.block_tables, st.context_lens, st.scale, lib=lib)
    perm = torch.randperm(p.num_blocks, generator=torch.Generator().manual_seed(5))
    kc2, vc2 = torch.empty_like(p.k_cache), torch.empty_like(p.v_cache)
    kc2[perm] = p.k_cache
    vc2[perm] = p.v_cache
    bt2 = st.block_tables.clone()
    valid = bt2 >= 0
    bt2[valid] = perm[bt2[valid].long()].to(torch.int32)
    b = oracle.decode(st.q, kc2, vc2, bt2, st.context_lens, st.scale, lib=lib)
    assert torch.equal(a, b)
    assert not torch.isnan(a).any()


def pin_decode_sharing(lib):
    st = inputs.make_decode([40, 37, 50, 33], num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=8,
                            dtype=torch.float16, seed=14, share_groups=4, share_tokens=32)
    p = st.pool
    oracle.store_kv(st.k_new, st.v_new, p.k_cache, p.v_cache, st.slot_mapping, lib=lib)
    a = oracle.decode(st.q, p.k_cache, p.v_cache, st.block_tables, st.context_lens, st.scale, lib=lib)
    # give every sequence private copies of the shared pages
    shared = p.tables[0][:4]
    extra = len(shared) * 3
    kc = torch.cat([p.k_cache, p.k_cache[:extra].clone()])
    vc = torch.cat([p.v_cache, p.v_cache[:extra].clone()])
    bt = st.block_tables.clone()
    nxt = p.num_blocks
    for i in range(1, 4):
        for j, blk in enumerate(shared):
            kc[nxt] = p.k_cache[blk]
            vc[nxt] = p.v_cache[blk]
            bt[i, j] = nxt
            nxt += 1
    b = oracle.decode(st.q, kc, vc, bt, st.context_lens, st.scale, lib=lib)
    assert torch.equal(a, b)


def pin_identical_keys_give_mean_of_v(lib):
    gen = torch.Generator().manual_seed(15)
    L, hkv, d, bs = 37, 1, 16, 8
    krow = torch.randn(1, hkv, d, generator=gen).to(torch.bfloat16)
    dk = [krow.expand(L, hkv, d).clone()]
    dv = [torch.randn(L, hkv, d, generator=gen).to(torch.bfloat16)]
    tables = [[3, 0, 4, 1, 2]]
    kc, vc = _dense_to_pool(dk, dv, tables, bs, 6, torch.bfloat16)
    q = torch.randn(1, 2, d, generator=gen).to(torch.bfloat16)
    out = oracle.decode(q, kc, vc, inputs.pad_block_tables(tables), torch.tensor([L], dtype=torch.int32),
                        0.25, lib=lib)
    mean = dv[0].double().mean(dim=0)[0]
    for h in range(2):
        torch.testing.assert_close(out[0, h].double(), mean, rtol=1e-6, atol=1e-6)


def pin_one_key_gives_v0(lib):
    gen = torch.Generator().manual_seed(16)
    for dtype in (torch.float16, torch.bfloat16):
        dk = [torch.randn(1, 2, 16, generator=gen).to(dtype)]
        dv = [torch.randn(1, 2, 16, generator=gen).to(dtype)]
        kc, vc = _dense_to_pool(dk, dv, [[2]], 4, 3, dtype)
        q = torch.randn(1, 4, 16, generator=gen).to(dtype)
        out = oracle.decode(q, kc, vc, torch.tensor([[2]], dtype=torch.int32), torch.tensor([1], dtype=torch.int32),
                            0.25, lib=lib)
        for h in range(4):
            assert torch.equal(out[0, h], dv[0][0, h // 2].float())


def pin_two_three_keys_brute_force(lib):
    gen = torch.Generator().manual_seed(17)
    d, scale = 8, 0.7
    for L in (2, 3):
        dk = [torch.randn(L, 1, d, generator=gen).to(torch.bfloat16)]
        dv = [torch.randn(L, 1, d, generator=gen).to(torch.bfloat16)]
        kc, vc = _dense_to_pool(dk, dv, [[1, 0]], 2, 2, torch.bfloat16)
        q = torch.randn(1, 1, d, generator=gen).to(torch.bfloat16)
        out = oracle.decode(q, kc, vc, torch.tensor([[1, 0]], dtype=torch.int32), torch.tensor([L], dtype=torch.int32),
                            scale, lib=lib)
        qq = [float(x) for x in q[0, 0]]
        kk = [[float(x) for x in dk[0][j, 0]] for j in range(L)]
        vv = [[float(x) for x in dv[0][j, 0]] for j in range(L)]
        w = [math.exp(scale * sum(a * b for a, b in zip(qq, kk[j]))) for j in range(L)]
        z = sum(w)
        ref = [sum(w[j] * vv[j][e] for j in range(L)) / z for e in range(d)]
        assert max(abs(float(out[0, 0, e]) - ref[e]) for e in range(d)) < 1e-6


def pin_empty_context_gives_zeros(lib):
    q = torch.ones(2, 2, 8, dtype=torch.float16)
    kc = torch.ones(2, 4, 1, 8, dtype=torch.float16)
    out = oracle.decode(q, kc, kc, torch.tensor([[-1], [0]], dtype=torch.int32), torch.tensor([0, 3], dtype=torch.int32),
                        1.0, lib=lib)
    assert torch.equal(out[0], torch.zeros(2, 8))
    assert torch.equal(out[1], torch.ones(2, 8))


def pin_bad_block_rejected(lib):
    q = torch.ones(1, 2, 8, dtype=torch.float16)
    kc = torch.ones(2, 4, 1, 8, dtype=torch.float16)
    for bt in ([[0, -1]], [[0, 2]]):
        with pytest.raises(oracle.OracleError):
            oracle.decode(q, kc, kc, torch.tensor(bt, dtype=torch.int32), torch.tensor([6], dtype=torch.int32),
                          1.0, lib=lib)


def _prefill_case(gen, prefix, chunk, hq, hkv, d, bs, dtype):
    """Dense contiguous K/V per sequence (prefix + chunk); the prefix part is
    scattered into a pool, the chunk part is the packed new k/v."""
    lk = [p + c for p, c in zip(prefix, chunk)]
    need = sum(inputs.num_pages(L, bs) for L in lk)
    nb = need + 2
    perm = torch.randperm(nb, generator=gen).tolist()
    tables, c = [], 0
    for L in lk:
        n = inputs.num_pages(L, bs)
        tables.append(perm[c:c + n])
        c += n
    dk = [torch.randn(L, hkv, d, generator=gen).to(dtype) for L in lk]
    dv = [torch.randn(L, hkv, d, generator=gen).to(dtype) for L in lk]
    kc, vc = _dense_to_pool([k[:p] for k, p in zip(dk, prefix)], [v[:p] for v, p in zip(dv, prefix)],
                            tables, bs, nb, dtype)
    q = torch.randn(sum(chunk), hq, d, generator=gen).to(dtype)
    kn = torch.cat([k[p:] for k, p in zip(dk, prefix)])
    vn = torch.cat([v[p:] for v, p in zip(dv, prefix)])
    return q, kn, vn, kc, vc, tables, dk, dv


def pin_prefill_vs_library(lib):
    gen = torch.Generator().manual_seed(18)
    hq, hkv, d, bs = 4, 2, 16, 4
    for prefix, chunk in (([0, 0], [7, 3]), ([5, 0, 9], [4, 6, 1])):
        q, kn, vn, kc, vc, tables, dk, dv = _prefill_case(gen, prefix, chunk, hq, hkv, d, bs, torch.bfloat16)
        bt = inputs.pad_block_tables(tables) if any(prefix) else None
        cq = inputs.cu_seqlens(chunk)
        ck = inputs.cu_seqlens([p + c for p, c in zip(prefix, chunk)])
        scale = 0.2
        out = oracle.prefill_paged(q, kn, vn, kc, vc, cq, ck, bt, scale, lib=lib)
        for i, (p, c) in enumerate(zip(prefix, chunk)):
            # full causal attention over the contiguous sequence, last c rows
            L = p + c
            qfull = torch.zeros(hq, L, d, dtype=torch.float64)
            qfull[:, p:] = q[cq[i]:cq[i + 1]].double().transpose(0, 1)
            ref = _lib_attention(qfull, dk[i].double().transpose(0, 1), dv[i].double().transpose(0, 1), scale,
                                 causal=True)[:, p:]
            torch.testing.assert_close(out[cq[i]:cq[i + 1]].double().transpose(0, 1), ref, rtol=0, atol=2e-6)


def pin_prefill_single_query_equals_decode(lib):
    gen = torch.Generator().manual_seed(19)
    hq, hkv, d, bs = 4, 2, 16, 4
    prefix, chunk = [10, 3], [1, 1]
    q, kn, vn, kc, vc, tables, dk, dv = _prefill_case(gen, prefix, chunk, hq, hkv, d, bs, torch.float16)
    bt = inputs.pad_block_tables(tables)
    out = oracle.prefill_paged(q, kn, vn, kc, vc, inputs.cu_seqlens(chunk),
                               inputs.cu_seqlens([p + 1 for p in prefix]), bt, 0.25, lib=lib)
    slots = torch.tensor([inputs.slot_of(t, bs, p) for t, p in zip(tables, prefix)], dtype=torch.int32)
    oracle.store_kv(kn, vn, kc, vc, slots, lib=lib)
    dec = oracle.decode(q, kc, vc, bt, torch.tensor([p + 1 for p in prefix], dtype=torch.int32), 0.25, lib=lib)
    torch.testing.assert_close(out, dec, rtol=0, atol=1e-6)


def pin_half_decoding(lib):
    words = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    f16 = words.view(np.float16).astype(np.float32)
    bf = torch.from_numpy(words.astype(np.int16)).view(torch.bfloat16).float().numpy()
    got16 = np.array([lib.oracle_half_to_float(int(w), oracle.F16) for w in words], dtype=np.float32)
    gotbf = np.array([lib.oracle_half_to_float(int(w), oracle.BF16) for w in words], dtype=np.float32)
    for got, ref in ((got16, f16), (gotbf, bf)):
        nan = np.isnan(ref)
        assert np.array_equal(np.isnan(got), nan)
        assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def _sample_rows(seed, B, V, dtype=torch.float32):
    g = torch.Generator().manual_seed(seed)
    logits = (3 * torch.randn(B, V, generator=g)).to(dtype)
    temps = 0.3 + 1.5 * torch.rand(B, generator=g)
    noise = torch.empty(B, V).exponential_(1, generator=g)
    return logits, temps, noise


def pin_sample_unit_noise_is_first_argmax(lib):
    logits, temps, _ = _sample_rows(1, 40, 97)
    logits[3, [5, 60]] = 50.0                     # a tie: the first index wins
    for dt in (torch.float32, torch.bfloat16, torch.float16):
        lg = logits.to(dt)
        got = oracle.sample(lg, temps, torch.ones(40, 97), lib=lib)
        ref = torch.tensor([int(np.argmax(row.float().numpy())) for row in lg], dtype=torch.int32)
        assert torch.equal(got, ref), dt
    assert int(oracle.sample(logits, temps, torch.ones(40, 97), lib=lib)[3]) == 5


def pin_sample_matches_float64_formula(lib):
    logits, temps, noise = _sample_rows(2, 300, 50)
    got = oracle.sample(logits, temps, noise, lib=lib)
    a = logits.double() / temps.double()[:, None]
    p = torch.softmax(a, dim=-1)
    score = p / noise.double().clamp_min(1e-10)
    ref = score.argmax(dim=-1)
    for b in torch.nonzero(got != ref.to(torch.int32)).flatten().tolist():
        s1, s2 = float(score[b, got[b]]), float(score[b, ref[b]])
        assert abs(s1 - s2) <= 1e-5 * s2, (b, s1, s2)  # only a near-tie may differ


def pin_sample_power_of_two_scaling(lib):
    logits, temps, noise = _sample_rows(3, 200, 64)
    a = oracle.sample(logits, temps, noise, lib=lib)
    b = oracle.sample(logits * 8, temps * 8, noise, lib=lib)
    assert torch.equal(a, b)


def pin_sample_masked_and_invalid(lib):
    logits, temps, noise = _sample_rows(4, 30, 40)
    logits[:, ::2] = float("-inf")
    temps[7] = 0.0
    got = oracle.sample(logits, temps, noise, lib=lib)
    assert int(got[7]) == -1
    ok = torch.arange(30) != 7
    assert bool((got[ok] % 2 == 1).all())


def pin_sample_frequencies_follow_softmax(lib):
    V, N, T = 6, 120000, 0.8
    z = torch.tensor([0.0, 1.0, 2.0, 4.0, -1.0, 3.0])
    g = torch.Generator().manual_seed(5)
    noise = torch.empty(N, V).exponential_(1, generator=g)
    got = oracle.sample(z.repeat(N, 1), torch.full((N,), T), noise, lib=lib)
    counts = torch.bincount(got.long(), minlength=V).double()
    expect = torch.softmax(z.double() / T, dim=0) * N
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 33.4, chi2  # 5 degrees of freedom: p < 1e-5 beyond this


def pin_e4m3_decoding(lib):
    codes = torch.arange(256, dtype=torch.uint8)
    ref = codes.view(torch.float8_e4m3fn).float()
    got = torch.tensor([lib.oracle_e4m3_to_float(int(c)) for c in codes])
    nan = torch.isnan(ref)
    assert torch.equal(torch.isnan(got), nan) and torch.equal(got[~nan], ref[~nan])


def pin_e4m3_encoding(lib):
    vals = torch.arange(127, dtype=torch.uint8).view(torch.float8_e4m3fn).float()
    mids = (vals[:-1] + vals[1:]) / 2                    # exact ties: nearest-even decides
    g = torch.Generator().manual_seed(6)
    rnd = (torch.randn(4000, generator=g) * 60).clamp(-448, 448)
    for x in (mids, -mids, rnd, torch.tensor([0.0, -0.0, 1e-9, -1e-9])):
        ref = x.to(torch.float8_e4m3fn).view(torch.uint8)
        got = torch.tensor([lib.oracle_float_to_e4m3(float(v)) for v in x], dtype=torch.uint8)
        assert torch.equal(got, ref)
    assert lib.oracle_float_to_e4m3(1000.0) == 0x7E and lib.oracle_float_to_e4m3(-5e5) == 0xFE  # +-448
    assert lib.oracle_float_to_e4m3(float("nan")) == 0x7F


def _fp8_step(seed, bs=16, hkv=2, hq=8, d=64, ctx=(40, 1, 130), dtype=torch.bfloat16):
    st = inputs.make_decode(list(ctx), num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, dtype=dtype,
                            seed=seed)
    g = torch.Generator().manual_seed(seed)
    kc = torch.randint(0, 255, st.pool.k_cache.shape, generator=g, dtype=torch.uint8)
    vc = torch.randint(0, 255, st.pool.v_cache.shape, generator=g, dtype=torch.uint8)
    kc[kc == 0x7F] = 0
    vc[vc == 0x7F] = 0
    kc[kc == 0xFF] = 0
    vc[vc == 0xFF] = 0
    return st, kc, vc


def pin_store_fp8_matches_torch(lib):
    st, kc, vc = _fp8_step(61)
    ks, vs = 0.37, 1.9
    k0, v0 = kc.clone(), vc.clone()
    oracle.store_kv_fp8(st.k_new, st.v_new, kc, vc, st.slot_mapping, ks, vs, lib=lib)
    rk, rv = k0.view(-1, k0.shape[2], k0.shape[3]), v0.view(-1, v0.shape[2], v0.shape[3])
    rows = st.slot_mapping.long()
    keep = rows >= 0
    rk[rows[keep]] = (st.k_new.float()[keep] / ks).to(torch.float8_e4m3fn).view(torch.uint8)
    rv[rows[keep]] = (st.v_new.float()[keep] / vs).to(torch.float8_e4m3fn).view(torch.uint8)
    assert torch.equal(kc, k0) and torch.equal(vc, v0)


def pin_decode_fp8_power_of_two_scales_equals_16bit_decode(lib):
    st, kc, vc = _fp8_step(62)
    ks, vs = 0.25, 4.0
    deq_k = (kc.view(torch.float8_e4m3fn).float() * ks).to(torch.bfloat16)
    deq_v = (vc.view(torch.float8_e4m3fn).float() * vs).to(torch.bfloat16)
    a = oracle.decode_fp8(st.q, kc, vc, st.block_tables, st.context_lens, st.scale, ks, vs, lib=lib)
    b = oracle.decode(st.q, deq_k, deq_v, st.block_tables, st.context_lens, st.scale, lib=lib)
    assert torch.equal(a, b)


def pin_decode_fp8_vs_library(lib):
    st, kc, vc = _fp8_step(63, ctx=(77, 300, 5))
    ks, vs = 0.0731, 2.33
    got = oracle.decode_fp8(st.q, kc, vc, st.block_tables, st.context_lens, st.scale, ks, vs, lib=lib)
    deq_k = kc.view(torch.float8_e4m3fn).double() * ks
    deq_v = vc.view(torch.float8_e4m3fn).double() * vs
    p = st.pool
    for b in range(st.batch):
        n = int(st.context_lens[b])
        rows = [inputs.slot_of(p.tables[b], p.block_size, j) for j in range(n)]
        K = deq_k.view(-1, p.num_kv_heads, p.head_dim)[rows]
        V = deq_v.view(-1, p.num_kv_heads, p.head_dim)[rows]
        group = st.q.shape[1] // p.num_kv_heads
        for h in range(st.q.shape[1]):
            s = (st.q[b, h].double() @ K[:, h // group].T) * st.scale
            ref = torch.softmax(s, dim=0) @ V[:, h // group]
            assert float((got[b, h].double() - ref).abs().max()) < 1e-4 * max(1.0, float(ref.abs().max()))


PINS = [pin_store_matches_index_put, pin_store_rejects_bad_slot, pin_decode_vs_library,
        pin_decode_permutation_invariance, pin_decode_sharing, pin_identical_keys_give_mean_of_v,
        pin_one_key_gives_v0, pin_two_three_keys_brute_force, pin_empty_context_gives_zeros,
        pin_bad_block_rejected, pin_prefill_vs_library, pin_prefill_single_query_equals_decode,
        pin_half_decoding, pin_sample_unit_noise_is_first_argmax, pin_sample_matches_float64_formula,
        pin_sample_power_of_two_scaling, pin_sample_masked_and_invalid, pin_sample_frequencies_follow_softmax,
        pin_e4m3_decoding, pin_e4m3_encoding, pin_store_fp8_matches_torch,
        pin_decode_fp8_power_of_two_scales_equals_16bit_decode, pin_decode_fp8_vs_library]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin, oracle_lib):
    pin(oracle_lib)
