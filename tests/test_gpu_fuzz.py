"""Seeded random cases of the attention calls against the oracle.

The fixed-shape tests pin the configurations the pages and the benchmark name;
these draw shapes, block sizes, length mixes and launch options at random
(from fixed seeds, so a failure reproduces) to reach combinations no fixed
case lists: prefill with random GQA groups, head dims, prefixes, chunk sizes
(empty and one-row chunks included) and persistent-grid caps; decode with random
split-K partitions, ring depths, and shared-prefix groups derived from the
tables.  Each case is small enough for the oracle to finish in a fraction of a
second.
"""

import random

import pytest
import torch

import oracle
from paged_kv_cache_bs_gb300.block_manager import prefix_groups
from tests import inputs
from tests.gpu_cases import TOL, check_decode, max_err

pytestmark = pytest.mark.gpu

HEADS = [(4, 4), (8, 4), (8, 2), (8, 1), (16, 4), (32, 8)]


@pytest.mark.parametrize("seed", range(40))
def test_prefill_random_cases(pa, seed):
    rnd = random.Random(1000 + seed)
    hq, hkv = rnd.choice(HEADS)
    d = rnd.choice([64, 128])
    bs = rnd.choice([8, 16, 64, 256, 1024])
    dtype = rnd.choice([torch.float16, torch.bfloat16])
    n = rnd.randint(1, 7)
    prefix = [rnd.choice([0, rnd.randint(1, 40), rnd.randint(100, 1500)]) for _ in range(n)]
    chunk = [rnd.choice([0, 1, rnd.randint(2, 127), 128, rnd.randint(129, 400)]) for _ in range(n)]
    if sum(chunk) == 0:
        chunk[0] = 5
    max_ctas = rnd.choice([0, 0, 1, 2, 5, 24])
    st, _ = inputs.make_prefill(prefix, chunk, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs,
                                dtype=dtype, seed=2000 + seed)
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.store_kv(st.k_new.cuda(), st.v_new.cuda(), kc, vc, st.slot_mapping.cuda())
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = pa.prefill_paged(st.q.cuda(), None, None, kc, vc, st.cu_seqlens_q.cuda(), st.cu_seqlens_k.cuda(),
                           st.max_seqlen_q, st.max_seqlen_k, st.block_tables.cuda(), st.scale, err_flag=flag,
                           max_ctas=max_ctas)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    okc, ovc = p.k_cache.clone(), p.v_cache.clone()
    oracle.store_kv(st.k_new, st.v_new, okc, ovc, st.slot_mapping)
    ref = oracle.prefill_paged(st.q, st.k_new, st.v_new, okc, ovc, st.cu_seqlens_q, st.cu_seqlens_k,
                               st.block_tables, st.scale)
    err = max_err(out, ref)
    assert err <= TOL[dtype], (f"heads {hq}/{hkv} D {d} bs {bs} {dtype} prefix {prefix} chunk {chunk} "
                               f"max_ctas {max_ctas}: max|err| {err}")


@pytest.mark.parametrize("seed", range(40))
def test_decode_random_cases(pa, seed):
    rnd = random.Random(3000 + seed)
    hq, hkv = rnd.choice(HEADS)
    d = rnd.choice([64, 128])
    bs = rnd.choice([8, 16, 32, 128, 256])
    dtype = rnd.choice([torch.float16, torch.bfloat16])
    b = rnd.randint(1, 40)
    ctx = [rnd.choice([0, 1, rnd.randint(2, 200), rnd.randint(200, 3000)]) for _ in range(b)]
    options = None
    if rnd.random() < 0.5:
        options = pa.DecodeOptions(partition=rnd.choice([0, 64, 128, 448, 1024]), stages=rnd.choice([0, 2, 3]))
    st = inputs.make_decode(ctx, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, dtype=dtype,
                            seed=4000 + seed)
    check_decode(pa, st, options=options)


@pytest.mark.parametrize("seed", range(16))
def test_decode_random_shared_prefixes(pa, seed):
    # runs of sequences sharing a prefix of whole pages, grouped from the tables as an engine would
    rnd = random.Random(5000 + seed)
    hq, hkv = rnd.choice([(8, 2), (16, 4), (32, 8), (8, 8)])
    bs = rnd.choice([16, 32, 64])
    share = bs * rnd.randint(1, 12)
    g = rnd.randint(2, 9)
    b = g * rnd.randint(1, 5)
    ctx = [share + rnd.randint(1, 900) for _ in range(b)]
    st = inputs.make_decode(ctx, num_q_heads=hq, num_kv_heads=hkv, head_dim=128, block_size=bs,
                            dtype=torch.bfloat16, seed=6000 + seed, share_groups=g, share_tokens=share)
    groups = prefix_groups(st.block_tables, st.context_lens, bs)
    assert groups.num_groups >= 1
    opt = pa.DecodeOptions(groups=groups.to("cuda"), partition=rnd.choice([0, 0, 256, 512]))
    check_decode(pa, st, options=opt)


@pytest.mark.parametrize("seed", range(12))
def test_store_decode_random_operands_in_place(pa, seed):
    # random shapes, dtypes, block sizes and split plans: q and the new rows read through the operands
    # array (page-locked or device, the call's own arguments zero-filled decoys) give the output and
    # pool of the direct call bit for bit
    rnd = random.Random(7000 + seed)
    hq, hkv = rnd.choice(HEADS)
    d = rnd.choice([64, 128])
    bs = rnd.choice([8, 16, 64, 256])
    dtype = rnd.choice([torch.float16, torch.bfloat16])
    b = rnd.randint(1, 33)
    ctx = [rnd.randint(1, 2500) for _ in range(b)]
    st = inputs.make_decode(ctx, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, block_size=bs, dtype=dtype,
                            seed=8000 + seed)
    options = pa.DecodeOptions(partition=rnd.choice([0, 64, 256, 1024]))
    where = rnd.choice(["pinned", "device"])
    real = {n: (t.pin_memory() if where == "pinned" else t.cuda()) for n, t in
            dict(k=st.k_new, v=st.v_new, q=st.q).items()}
    decoy = {n: torch.zeros_like(t, device="cuda") for n, t in real.items()}
    sm, bt, cl = st.slot_mapping.cuda(), st.block_tables.cuda(), st.context_lens.cuda()
    kc_a, vc_a = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    ref = pa.store_decode(real["k"], real["v"], sm, real["q"], kc_a, vc_a, bt, cl, st.scale, options=options)
    ops = torch.tensor([real["q"].data_ptr(), real["k"].data_ptr(), real["v"].data_ptr()],
                       dtype=torch.int64).pin_memory()
    kc_b, vc_b = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = pa.store_decode(decoy["k"], decoy["v"], sm, decoy["q"], kc_b, vc_b, bt, cl, st.scale, err_flag=flag,
                          options=pa.DecodeOptions(partition=options.partition, operands=ops.data_ptr()))
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"seed {seed}: output differs"
    assert torch.equal(kc_b.view(torch.int16), kc_a.view(torch.int16)), f"seed {seed}: k pool differs"
    assert torch.equal(vc_b.view(torch.int16), vc_a.view(torch.int16)), f"seed {seed}: v pool differs"
