"""GPU parity of pa_decode (after pa_store_kv) against the oracle.

Full-size workloads run through the same call ``bench.py`` times; the oracle
computes every sequence (it finishes in seconds at these sizes).  Edge cases:
empty and one-token contexts, contexts on and off tile/partition/page
boundaries, block sizes 8..1024, GQA groups 1..8, both dtypes and head dims,
relabelled physical blocks, bad metadata (flagged, never faulting)."""

import os

import pytest
import torch

import oracle
from tests import inputs
from tests.gpu_cases import TOL, assert_bit_equal, check_decode, max_err, run_decode_gpu

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name", ["tiny_decode", "qwen3_0p6b_decode", "qwen3_8b_shared_decode",
                                  "long_context_decode"])
def test_decode_workloads_full(pa, name):
    st = inputs.WORKLOADS[name]()
    err = check_decode(pa, st)
    print(f"{name}: max|err| = {err:.3e}")


def test_decode_mixed_step_decode_rows(pa):
    m = inputs.mixed_chunked_prefill()
    st = m.decode
    check_decode(pa, st)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (8, 1)])
def test_decode_shapes(pa, dtype, head_dim, hq, hkv):
    # contexts around tile (64), page (16) and partition boundaries, incl. empty rows
    ctx = [0, 1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 500, 1023, 1024, 1025, 3000]
    st = inputs.make_decode(ctx, num_q_heads=hq, num_kv_heads=hkv, head_dim=head_dim, block_size=16,
                            dtype=dtype, seed=31 + hq + hkv + head_dim)
    check_decode(pa, st)


@pytest.mark.parametrize("bs", [8, 32, 64, 128, 512, 1024])
def test_decode_block_sizes(pa, bs):
    ctx = [1, bs - 1, bs, bs + 1, 3 * bs + 5, 2100]
    st = inputs.make_decode(ctx, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=bs,
                            dtype=torch.bfloat16, seed=40 + bs)
    check_decode(pa, st)


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("hq,hkv,head_dim,bs", [(32, 8, 128, 16), (8, 1, 64, 256), (4, 4, 128, 8)])
def test_decode_context_of_one_returns_its_value_row(pa, dtype, hq, hkv, head_dim, bs):
    # A context of one token (the one this step stores) has weight 1: the output is that token's value
    # row for every query head of its group, bit for bit, through pa_decode and the fused store + decode
    # (the row maximum, the exponent and the sum must agree exactly).
    ctx = [1, 1, 37, 1, 300, 1]
    st = inputs.make_decode(ctx, num_q_heads=hq, num_kv_heads=hkv, head_dim=head_dim, block_size=bs,
                            dtype=dtype, seed=52 + hq + bs)
    out, _, _ = run_decode_gpu(pa, st)
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    fused = pa.store_decode(st.k_new.cuda(), st.v_new.cuda(), st.slot_mapping.cuda(), st.q.cuda(), kc, vc,
                            st.block_tables.cuda(), st.context_lens.cuda(), st.scale)
    torch.cuda.synchronize()
    for b, L in enumerate(ctx):
        if L == 1:
            expect = st.v_new[b].repeat_interleave(hq // hkv, dim=0)
            assert_bit_equal(out[b], expect, f"sequence {b}")
            assert_bit_equal(fused[b], expect, f"sequence {b}, fused")


def test_decode_empty_context_rows_are_zero(pa):
    st = inputs.make_decode([0, 5, 0, 70], num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                            dtype=torch.float16, seed=50)
    out, _, _ = run_decode_gpu(pa, st)
    assert not out[0].any() and not out[2].any()
    check_decode(pa, st)


def test_decode_block_relabelling_is_bit_identical(pa):
    st = inputs.make_decode([300, 1000, 77, 4096], num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=16,
                            dtype=torch.bfloat16, seed=51)
    a, _, _ = run_decode_gpu(pa, st)
    p = st.pool
    perm = torch.randperm(p.num_blocks, generator=torch.Generator().manual_seed(9))
    kc2, vc2 = torch.empty_like(p.k_cache), torch.empty_like(p.v_cache)
    kc2[perm], vc2[perm] = p.k_cache, p.v_cache
    bt2 = st.block_tables.clone()
    bt2[bt2 >= 0] = perm[bt2[bt2 >= 0].long()].to(torch.int32)
    slots2 = (perm[(st.slot_mapping // p.block_size).long()] * p.block_size
              + st.slot_mapping % p.block_size).to(torch.int32)
    kc, vc = kc2.cuda(), vc2.cuda()
    pa.store_kv(st.k_new.cuda(), st.v_new.cuda(), kc, vc, slots2.cuda())
    b = pa.decode(st.q.cuda(), kc, vc, bt2.cuda(), st.context_lens.cuda(), st.scale)
    torch.cuda.synchronize()
    assert_bit_equal(a, b, "decode output under block relabelling")


def test_decode_shared_prefix_equals_private_copies(pa):
    st = inputs.make_decode([600, 700, 900, 513], num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                            dtype=torch.bfloat16, seed=52, share_groups=4, share_tokens=512)
    a, kc, vc = run_decode_gpu(pa, st)
    shared = st.pool.tables[0][:32]
    n0 = st.pool.num_blocks
    kc2 = torch.cat([kc, kc[shared].repeat(3, 1, 1, 1)])
    vc2 = torch.cat([vc, vc[shared].repeat(3, 1, 1, 1)])
    bt = st.block_tables.clone()
    for i in range(1, 4):
        bt[i, :32] = torch.arange(n0 + (i - 1) * 32, n0 + i * 32, dtype=torch.int32)
    b = pa.decode(st.q.cuda(), kc2.contiguous(), vc2.contiguous(), bt.cuda(), st.context_lens.cuda(), st.scale)
    torch.cuda.synchronize()
    assert_bit_equal(a, b, "shared prefix vs private copies")


@pytest.mark.parametrize("part,stages", [(64, 3), (128, 2), (512, 0), (4096, 3)])
def test_decode_partition_size_does_not_change_result(pa, part, stages):
    # the split-K plan overridden through pa_decode_ex's options: the same attention
    st = inputs.make_decode([1, 700, 2049, 5000], num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=256,
                            dtype=torch.bfloat16, seed=53)
    check_decode(pa, st, options=pa.DecodeOptions(partition=part, stages=stages))


def test_decode_identical_keys_mean_of_v(pa):
    st = inputs.make_decode([777], num_q_heads=4, num_kv_heads=1, head_dim=128, block_size=16,
                            dtype=torch.bfloat16, seed=54)
    p = st.pool
    kf = p.k_cache.view(-1, 1, 128)
    rows = [inputs.slot_of(p.tables[0], 16, j) for j in range(777)]
    k0 = kf[rows[0]].clone()
    kf[rows] = k0
    st.k_new[:] = k0
    out, _, vc = run_decode_gpu(pa, st)
    mean = vc.view(-1, 1, 128)[torch.tensor(rows).cuda()].double().mean(0)[0]
    for h in range(4):
        assert float((out[0, h].double() - mean).abs().max()) < 2e-3


def test_decode_strided_q(pa):
    st = inputs.make_decode([100, 2000], num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=256,
                            dtype=torch.bfloat16, seed=55)
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.store_kv(st.k_new.cuda(), st.v_new.cuda(), kc, vc, st.slot_mapping.cuda())
    qkv = torch.zeros(2, 32, 128, dtype=torch.bfloat16, device="cuda")
    qkv[:, :16] = st.q.cuda()
    out = pa.decode(qkv[:, :16], kc, vc, st.block_tables.cuda(), st.context_lens.cuda(), st.scale)
    okc, ovc = p.k_cache.clone(), p.v_cache.clone()
    oracle.store_kv(st.k_new, st.v_new, okc, ovc, st.slot_mapping)
    ref = oracle.decode(st.q, okc, ovc, st.block_tables, st.context_lens, st.scale)
    assert max_err(out, ref) <= TOL[torch.bfloat16]


def test_decode_bad_metadata_is_flagged_not_fatal(pa):
    st = inputs.make_decode([40, 40, 40], num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                            dtype=torch.float16, seed=56)
    bt = st.block_tables.clone()
    bt[0, 1] = -1                       # hole inside the context
    bt[1, 2] = st.pool.num_blocks + 5   # id past the pool
    ctx = st.context_lens.clone()
    ctx[2] = 10_000                     # longer than the table allows
    kc, vc = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.decode(st.q.cuda(), kc, vc, bt.cuda(), ctx.cuda(), st.scale, err_flag=flag)
    torch.cuda.synchronize()
    f = int(flag.item())
    assert f & pa.FLAG_BAD_BLOCK and f & pa.FLAG_BAD_LENGTH
    # the device is still healthy
    check_decode(pa, inputs.tiny_decode())


@pytest.mark.parametrize("fused", [False, True])
def test_store_and_decode_replay_from_a_cuda_graph(pa, fused):
    # A decode step captured once and replayed on new inputs of the same shapes, as an
    # engine replays its decode graph every step ("nano-vLLM Part 2", section 4.2): padding
    # rows (context 0, slot -1) included.
    ctx = [700, 0, 33, 2048, 1, 129, 0, 512]
    steps = [inputs.make_decode(ctx, num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                                dtype=torch.bfloat16, seed=seed) for seed in (71, 72, 73)]
    for st in steps[1:]:
        assert st.pool.k_cache.shape == steps[0].pool.k_cache.shape
        assert st.block_tables.shape == steps[0].block_tables.shape
    st0 = steps[0]
    kc, vc = st0.pool.k_cache.cuda(), st0.pool.v_cache.cuda()
    q, kn, vn = st0.q.cuda(), st0.k_new.cuda(), st0.v_new.cuda()
    sm, bt, cl = st0.slot_mapping.cuda(), st0.block_tables.cuda(), st0.context_lens.cuda()
    ws = pa.alloc_decode_workspace(q, kc, bt)
    out = torch.empty_like(q)

    def step():
        if fused:
            pa.store_decode(kn, vn, sm, q, kc, vc, bt, cl, st0.scale, out=out, workspace=ws)
        else:
            pa.store_kv(kn, vn, kc, vc, sm)
            pa.decode(q, kc, vc, bt, cl, st0.scale, out=out, workspace=ws)

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        step()                                   # first call on the device: set-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for st in steps:
        for dst, src in ((kc, st.pool.k_cache), (vc, st.pool.v_cache), (q, st.q), (kn, st.k_new), (vn, st.v_new),
                         (sm, st.slot_mapping), (bt, st.block_tables), (cl, st.context_lens)):
            dst.copy_(src)
        out.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        okc, ovc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
        oracle.store_kv(st.k_new, st.v_new, okc, ovc, st.slot_mapping)
        assert_bit_equal(kc, okc, "k_cache after a replayed store")
        ref = oracle.decode(st.q, okc, ovc, st.block_tables, st.context_lens, st.scale)
        assert max_err(out, ref) <= TOL[torch.bfloat16]
