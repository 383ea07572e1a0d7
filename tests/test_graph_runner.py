"""The bucketed CUDA-graph decode runner ("nano-vLLM Part 2", section 4.2): bucket sizes on
the CPU; on the GPU, a replayed step equals the eager fused call on the same inputs (output
and pool bit-identical), for batch sizes that fill a bucket and ones that need padding rows,
over 16-bit and E4M3 pools, with the kernels reading the step's operands from pinned host
memory (zero copy) and with copies to and from device buffers."""

import pytest
import torch

import oracle
from tests import inputs
from tests.gpu_cases import TOL, max_err


def test_graph_batch_sizes():
    from paged_kv_cache_bs_gb300.graphs import graph_batch_sizes
    assert graph_batch_sizes(1) == [1]
    assert graph_batch_sizes(8) == [1, 2, 4, 8]
    assert graph_batch_sizes(64) == [1, 2, 4, 8, 16, 32, 48, 64]
    assert graph_batch_sizes(100) == [1, 2, 4, 8, 16, 32, 48, 64, 80, 96, 100]
    assert graph_batch_sizes(512)[-1] == 512 and len(graph_batch_sizes(512)) == 4 + 32
    with pytest.raises(ValueError):
        graph_batch_sizes(0)


def _eager(pa, st, kc, vc, fs=None):
    d = {k: t.cuda() for k, t in dict(k=st.k_new, v=st.v_new, sm=st.slot_mapping, q=st.q, bt=st.block_tables,
                                      cl=st.context_lens).items()}
    if fs is None:
        out = pa.store_decode(d["k"], d["v"], d["sm"], d["q"], kc, vc, d["bt"], d["cl"], st.scale)
    else:
        out = pa.store_decode_fp8(d["k"], d["v"], d["sm"], d["q"], kc, vc, d["bt"], d["cl"], st.scale, fs.k_scale,
                                  fs.v_scale)
    torch.cuda.synchronize()
    return out.cpu()


@pytest.mark.gpu
@pytest.mark.parametrize("zero_copy", [True, False])
@pytest.mark.parametrize("fp8", [False, True])
def test_runner_equals_eager_step(pa, fp8, zero_copy):
    from paged_kv_cache_bs_gb300.graphs import DecodeGraphRunner
    ctx_all = torch.randint(1, 3000, (40,), generator=torch.Generator().manual_seed(170)).tolist()
    kw = dict(num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=16, dtype=torch.bfloat16, seed=171)
    fs = inputs.make_decode_fp8(ctx_all, **kw) if fp8 else None
    st = fs.step if fp8 else inputs.make_decode(ctx_all, **kw)
    pool_k, pool_v = (fs.k_cache, fs.v_cache) if fp8 else (st.pool.k_cache, st.pool.v_cache)
    width = st.block_tables.shape[1]
    kc, vc = pool_k.cuda(), pool_v.cuda()
    runner = DecodeGraphRunner(kc, vc, 16, 40, width, st.scale, torch.bfloat16,
                               k_scale=fs.k_scale if fp8 else None, v_scale=fs.v_scale if fp8 else None,
                               zero_copy=zero_copy)
    for batch in (1, 3, 16, 17, 40):  # exact buckets and padded ones
        b = runner.bucket(batch)
        # the eager call on the bucket's padded inputs (slot -1, context 0 past `batch`): the split-K
        # plan depends on the batch size, so the graph of bucket b matches the eager call of size b
        pad = lambda t, v: torch.cat([t[:batch], torch.full((b - batch,) + tuple(t.shape[1:]), v, dtype=t.dtype)])  # noqa: E731
        sub = type(st)(st.pool, st.num_q_heads, pad(st.q, 0), pad(st.k_new, 0), pad(st.v_new, 0),
                       pad(st.slot_mapping, -1), pad(st.block_tables, -1), pad(st.context_lens, 0), st.scale)
        kc2, vc2 = pool_k.cuda(), pool_v.cuda()
        ref = _eager(pa, sub, kc2, vc2, fs)[:batch]
        kc.copy_(pool_k.cuda())
        vc.copy_(pool_v.cuda())
        sl = slice(0, batch)
        got = runner.step(st.q[sl], st.k_new[sl], st.v_new[sl], st.slot_mapping[sl], st.context_lens[sl],
                          st.block_tables[sl])
        assert got.shape == ref.shape
        assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"batch {batch}: output differs"
        if zero_copy:
            # the caller's page-locked tensors, read in place by the graph's first kernel (the step is
            # stored again: the same rows into the same slots)
            pinned = [t[sl].contiguous().pin_memory() for t in (st.q, st.k_new, st.v_new, st.slot_mapping,
                                                               st.context_lens, st.block_tables)]
            got = runner.step(*pinned).clone()
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"batch {batch}: pinned inputs"
        bits = (lambda t: t.cpu().view(torch.uint8))  # noqa: E731  (NaN sentinels compare by bits)
        assert torch.equal(bits(kc), bits(kc2)) and torch.equal(bits(vc), bits(vc2)), f"batch {batch}: pool differs"
    # and the replayed step against the oracle on the real rows
    okc, ovc = pool_k.clone(), pool_v.clone()
    if fp8:
        oracle.store_kv_fp8(st.k_new, st.v_new, okc, ovc, st.slot_mapping, fs.k_scale, fs.v_scale)
        ref = oracle.decode_fp8(st.q, okc, ovc, st.block_tables, st.context_lens, st.scale, fs.k_scale, fs.v_scale)
    else:
        oracle.store_kv(st.k_new, st.v_new, okc, ovc, st.slot_mapping)
        ref = oracle.decode(st.q, okc, ovc, st.block_tables, st.context_lens, st.scale)
    assert max_err(got, ref) <= TOL[st.q.dtype]


@pytest.mark.gpu
@pytest.mark.parametrize("zero_copy", [True, False])
def test_runner_with_shared_prefix_groups(pa, zero_copy):
    # a runner captured for shared-prefix groups: steps with their groups (fewer than the capacity,
    # and none at all) replayed from the staging, each against the oracle
    from paged_kv_cache_bs_gb300.block_manager import prefix_groups
    from paged_kv_cache_bs_gb300.graphs import DecodeGraphRunner
    seqs = [(600 + 37 * i, i // 6, 512) for i in range(18)] + [(90 + i, -1, 0) for i in range(5)]
    st = inputs.make_decode_shared(seqs, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                                   dtype=torch.bfloat16, seed=181)
    kc, vc = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    runner = DecodeGraphRunner(kc, vc, 32, 24, st.block_tables.shape[1], st.scale, torch.bfloat16,
                               zero_copy=zero_copy, group_caps=(4, 8, 1024))
    okc, ovc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
    steps = [st, inputs.next_decode_step(st, seed=182)]
    for i, s in enumerate(steps * 3):
        # the groups passed in, none (plain decode), or derived by the runner from the staged tables
        g = prefix_groups(s.block_tables, s.context_lens, 16) if i < 2 else None
        if g is not None:
            assert g.num_groups == 3
        got = runner.step(s.q, s.k_new, s.v_new, s.slot_mapping, s.context_lens, s.block_tables, groups=g,
                          share_prefixes=i >= 4)
        if i >= 4:
            assert int(runner.host_inputs(s.q.shape[0])["group_offsets"][3]) == 18
        oracle.store_kv(s.k_new, s.v_new, okc, ovc, s.slot_mapping)
        ref = oracle.decode(s.q, okc, ovc, s.block_tables, s.context_lens, s.scale)
        assert max_err(got, ref) <= TOL[torch.bfloat16], f"step {i}"
    with pytest.raises(ValueError):
        big = prefix_groups(st.block_tables, st.context_lens, 16)
        runner.set_inputs(st.q, st.k_new, st.v_new, st.slot_mapping, st.context_lens, st.block_tables,
                          groups=pa.PrefixGroups(big.group_offsets, big.group_seqs, big.prefix_lens, 9, 512))


@pytest.mark.gpu
def test_runner_with_tables_narrower_than_its_width(pa):
    # the runner is captured for wider tables than the steps pass: the staged rows are padded with
    # -1 past the step's columns (no stale entry from an earlier, wider step is ever in reach), and
    # steps of several batch sizes alternate with the derived shared-prefix groups
    from paged_kv_cache_bs_gb300.graphs import DecodeGraphRunner
    seqs = [(300 + 41 * i, i // 4, 256) for i in range(12)] + [(40 + i, -1, 0) for i in range(4)]
    st = inputs.make_decode_shared(seqs, num_q_heads=16, num_kv_heads=4, head_dim=128, block_size=16,
                                   dtype=torch.bfloat16, seed=191)
    width = st.block_tables.shape[1]
    kc, vc = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    runner = DecodeGraphRunner(kc, vc, 16, 16, width + 7, st.scale, torch.bfloat16, group_caps=(4, 8, 512))
    okc, ovc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
    # a first step with garbage in the extra columns of the staging
    runner.host_inputs(16)["block_tables"].fill_(12345)
    for i, s in enumerate([st, inputs.next_decode_step(st, seed=192)]):
        for share in (True, False):
            got = runner.step(s.q, s.k_new, s.v_new, s.slot_mapping, s.context_lens, s.block_tables,
                              share_prefixes=share).clone()
            staged = runner.host_inputs(16)["block_tables"]
            assert (staged[:, width:] == -1).all()
            if share:
                oracle.store_kv(s.k_new, s.v_new, okc, ovc, s.slot_mapping)
            ref = oracle.decode(s.q, okc, ovc, s.block_tables, s.context_lens, s.scale)
            assert max_err(got, ref) <= TOL[torch.bfloat16], f"step {i} share {share}"


@pytest.mark.gpu
def test_runner_full_shared_prefix_workload_in_place_bit_equal(pa):
    # the full Qwen3-8B-like shared-prefix step as a caller runs it: page-locked inputs read in
    # place through the operands array, groups derived by the native staging call, two alternating
    # steps; each output and the pool bit-identical to the eager fused call with the same groups
    from paged_kv_cache_bs_gb300.block_manager import prefix_groups
    from paged_kv_cache_bs_gb300.graphs import DecodeGraphRunner
    st = inputs.qwen3_8b_shared_decode()
    steps = [st, inputs.next_decode_step(st, seed=4242)]
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    runner = DecodeGraphRunner(kc, vc, st.num_q_heads, st.batch, st.block_tables.shape[1], st.scale,
                               torch.bfloat16, group_caps=(st.batch // 2, 8, 512))
    kc_e, vc_e = p.k_cache.cuda(), p.v_cache.cuda()
    for i, s in enumerate(steps):
        pinned = [t.contiguous().pin_memory() for t in (s.q, s.k_new, s.v_new, s.slot_mapping, s.context_lens,
                                                         s.block_tables)]
        got = runner.step(*pinned, share_prefixes=True).clone()
        g = prefix_groups(s.block_tables, s.context_lens, p.block_size).to("cuda")
        ref = pa.store_decode(s.k_new.cuda(), s.v_new.cuda(), s.slot_mapping.cuda(), s.q.cuda(), kc_e, vc_e,
                              s.block_tables.cuda(), s.context_lens.cuda(), s.scale,
                              options=pa.DecodeOptions(groups=g))
        torch.cuda.synchronize()
        assert runner._use_inplace[st.batch], "page-locked inputs take the in-place graph"
        assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16)), f"step {i}: output differs"
    assert torch.equal(kc.cpu().view(torch.int16), kc_e.cpu().view(torch.int16)), "k pool differs"
    assert torch.equal(vc.cpu().view(torch.int16), vc_e.cpu().view(torch.int16)), "v pool differs"


@pytest.mark.gpu
def test_runner_full_fp8_workload_in_place_bit_equal(pa):
    # the Qwen3-0.6B-like step over its E4M3 pool as a caller runs it: page-locked inputs read in place
    # through pa_store_decode_fp8_ex's operands, two alternating steps; output and codes bit-identical to
    # the eager fused call
    from paged_kv_cache_bs_gb300.graphs import DecodeGraphRunner
    fs = inputs.qwen3_0p6b_decode_fp8()
    st = fs.step
    steps = [st, inputs.next_decode_step(st, seed=4243)]
    kc, vc = fs.k_cache.cuda(), fs.v_cache.cuda()
    runner = DecodeGraphRunner(kc, vc, st.num_q_heads, st.batch, st.block_tables.shape[1], st.scale,
                               torch.bfloat16, k_scale=fs.k_scale, v_scale=fs.v_scale)
    kc_e, vc_e = fs.k_cache.cuda(), fs.v_cache.cuda()
    for i, s in enumerate(steps):
        pinned = [t.contiguous().pin_memory() for t in (s.q, s.k_new, s.v_new, s.slot_mapping, s.context_lens,
                                                         s.block_tables)]
        got = runner.step(*pinned).clone()
        ref = pa.store_decode_fp8(s.k_new.cuda(), s.v_new.cuda(), s.slot_mapping.cuda(), s.q.cuda(), kc_e, vc_e,
                                  s.block_tables.cuda(), s.context_lens.cuda(), s.scale, fs.k_scale, fs.v_scale)
        torch.cuda.synchronize()
        assert runner._use_inplace[runner.bucket(st.batch)], "page-locked inputs take the in-place graph"
        assert torch.equal(got.view(torch.int16), ref.cpu().view(torch.int16)), f"step {i}: output differs"
    assert torch.equal(kc.cpu(), kc_e.cpu()) and torch.equal(vc.cpu(), vc_e.cpu()), "E4M3 pool differs"
