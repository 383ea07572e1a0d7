"""GPU parity of pa_store_decode (the decode step's store fused into decode)
against the oracle, and against pa_store_kv followed by pa_decode."""

import pytest
import torch

import oracle
from tests import inputs
from tests.gpu_cases import TOL, assert_bit_equal, max_err

pytestmark = pytest.mark.gpu


def run_fused(pa, st, err_flag=None, slots=None):
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    sm = (st.slot_mapping if slots is None else slots).cuda()
    out = pa.store_decode(st.k_new.cuda(), st.v_new.cuda(), sm, st.q.cuda(), kc, vc, st.block_tables.cuda(),
                          st.context_lens.cuda(), st.scale, err_flag=err_flag)
    torch.cuda.synchronize()
    return out, kc, vc


def check_fused(pa, st):
    out, kc, vc = run_fused(pa, st)
    okc, ovc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
    oracle.store_kv(st.k_new, st.v_new, okc, ovc, st.slot_mapping)
    assert_bit_equal(kc, okc, "k_cache after the fused store")
    assert_bit_equal(vc, ovc, "v_cache after the fused store")
    ref = oracle.decode(st.q, okc, ovc, st.block_tables, st.context_lens, st.scale)
    err = max_err(out, ref)
    assert err <= TOL[st.q.dtype], f"max |err| {err}"
    return out


@pytest.mark.parametrize("name", ["tiny_decode", "qwen3_0p6b_decode", "qwen3_8b_shared_decode",
                                  "long_context_decode"])
def test_store_decode_workloads_full(pa, name):
    check_fused(pa, inputs.WORKLOADS[name]())


def test_store_decode_equals_separate_calls(pa):
    st = inputs.qwen3_0p6b_decode()
    fused = check_fused(pa, st)
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.store_kv(st.k_new.cuda(), st.v_new.cuda(), kc, vc, st.slot_mapping.cuda())
    sep = pa.decode(st.q.cuda(), kc, vc, st.block_tables.cuda(), st.context_lens.cuda(), st.scale)
    torch.cuda.synchronize()
    assert_bit_equal(fused, sep, "fused vs separate store + decode")


@pytest.mark.parametrize("bs", [8, 16, 64, 256, 1024])
@pytest.mark.parametrize("dtype,head_dim", [(torch.bfloat16, 128), (torch.float16, 64)])
def test_store_decode_block_sizes(pa, bs, dtype, head_dim):
    # contexts on and off tile, page and partition boundaries, and padding rows
    ctx = [1, 0, 63, 64, 65, bs, bs + 1, 2049, 0, 5000]
    st = inputs.make_decode(ctx, num_q_heads=16, num_kv_heads=4, head_dim=head_dim, block_size=bs, dtype=dtype,
                            seed=100 + bs + head_dim)
    out = check_fused(pa, st)
    assert not out[1].any() and not out[8].any()


def test_store_decode_flags_a_slot_that_is_not_the_last_position(pa):
    st = inputs.make_decode([40, 300, 0, 77], num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                            dtype=torch.bfloat16, seed=110)
    slots = st.slot_mapping.clone()
    good = int(slots[1])
    slots[1] = good - 1          # a slot of the same sequence, but not position L-1
    slots[2] = 5                 # a new row for a sequence with no context
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    out, kc, vc = run_fused(pa, st, err_flag=flag, slots=slots)
    assert int(flag.item()) & pa.FLAG_BAD_SLOT
    # the flagged rows were not written; the others were
    okc = st.pool.k_cache.clone()
    ovc = st.pool.v_cache.clone()
    keep = st.slot_mapping.clone()
    keep[1] = -1
    keep[2] = -1
    oracle.store_kv(st.k_new, st.v_new, okc, ovc, keep)
    assert_bit_equal(kc, okc, "k_cache with the flagged rows skipped")
    ref = oracle.decode(st.q[[0, 3]], okc, ovc, st.block_tables[[0, 3]], st.context_lens[[0, 3]], st.scale)
    assert max_err(out[[0, 3]], ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("fp8", [False, True])
def test_store_decode_with_pinned_host_operands(pa, fp8):
    """The per-step operands (q, the new rows, slot mapping, tables, lengths, out) in pinned host
    memory, read and written by the kernels directly: output and pool bit-identical to the call
    on device copies of the same operands.  Pageable host memory is refused."""
    ctx = torch.randint(1, 5000, (37,), generator=torch.Generator().manual_seed(181)).tolist()
    kw = dict(num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=256, dtype=torch.bfloat16, seed=182)
    fs = inputs.make_decode_fp8(ctx, **kw) if fp8 else None
    st = fs.step if fp8 else inputs.make_decode(ctx, **kw)
    pool_k, pool_v = (fs.k_cache, fs.v_cache) if fp8 else (st.pool.k_cache, st.pool.v_cache)
    ops = dict(k=st.k_new, v=st.v_new, sm=st.slot_mapping, q=st.q, bt=st.block_tables, cl=st.context_lens)

    def call(d, kc, vc, out):
        if fp8:
            return pa.store_decode_fp8(d["k"], d["v"], d["sm"], d["q"], kc, vc, d["bt"], d["cl"], st.scale,
                                       fs.k_scale, fs.v_scale, out=out)
        return pa.store_decode(d["k"], d["v"], d["sm"], d["q"], kc, vc, d["bt"], d["cl"], st.scale, out=out)

    kc_d, vc_d = pool_k.cuda(), pool_v.cuda()
    ref = call({n: t.cuda() for n, t in ops.items()}, kc_d, vc_d, None)
    kc_h, vc_h = pool_k.cuda(), pool_v.cuda()
    out_h = torch.full(tuple(st.q.shape), float("nan"), dtype=st.q.dtype).pin_memory()
    call({n: t.pin_memory() for n, t in ops.items()}, kc_h, vc_h, out_h)
    torch.cuda.synchronize()
    assert_bit_equal(out_h, ref.cpu(), "output written to pinned host memory")
    bits = (lambda t: t.cpu().view(torch.uint8))  # noqa: E731
    assert torch.equal(bits(kc_h), bits(kc_d)) and torch.equal(bits(vc_h), bits(vc_d)), "pool differs"
    with pytest.raises(ValueError):
        call(dict(ops), kc_h, vc_h, None)  # pageable host tensors


@pytest.mark.parametrize("where", ["device", "pinned"])
@pytest.mark.parametrize("grouped", [False, True])
def test_store_decode_operands_read_at_run_time(pa, where, grouped):
    """pa_decode_options.operands: the kernels take q and the new K/V rows from an array of three
    addresses read when they run.  The call's own q / k / v point at a zero-filled decoy: output and
    pool are bit-identical to the call that passes the real tensors, with and without shared-prefix
    groups, for operands in device or page-locked host memory."""
    from paged_kv_cache_bs_gb300.block_manager import prefix_groups
    seqs = [(500 + 29 * i, i // 5, 256) for i in range(15)] + [(70 + 3 * i, -1, 0) for i in range(6)]
    st = inputs.make_decode_shared(seqs, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                                   dtype=torch.bfloat16, seed=211)
    groups = prefix_groups(st.block_tables, st.context_lens, 16).to("cuda") if grouped else None
    real = dict(k=st.k_new, v=st.v_new, q=st.q)
    real = {n: (t.cuda() if where == "device" else t.pin_memory()) for n, t in real.items()}
    decoy = {n: torch.zeros_like(t, device="cuda") for n, t in real.items()}
    sm, bt, cl = st.slot_mapping.cuda(), st.block_tables.cuda(), st.context_lens.cuda()
    kc_a, vc_a = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    ref = pa.store_decode(real["k"], real["v"], sm, real["q"], kc_a, vc_a, bt, cl, st.scale,
                          options=pa.DecodeOptions(groups=groups) if grouped else None)
    ops = torch.tensor([real["q"].data_ptr(), real["k"].data_ptr(), real["v"].data_ptr()],
                       dtype=torch.int64).pin_memory()
    kc_b, vc_b = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = pa.store_decode(decoy["k"], decoy["v"], sm, decoy["q"], kc_b, vc_b, bt, cl, st.scale, err_flag=flag,
                          options=pa.DecodeOptions(groups=groups, operands=ops.data_ptr()))
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    assert_bit_equal(got, ref, "output through the operands array")
    bits = (lambda t: t.cpu().view(torch.uint8))  # noqa: E731
    assert torch.equal(bits(kc_b), bits(kc_a)) and torch.equal(bits(vc_b), bits(vc_a)), "pool differs"
    # an unaligned address is flagged before any access through it (no load is issued from it)
    ops[0] = real["q"].data_ptr() + 2
    kc_c, vc_c = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    pa.store_decode(decoy["k"], decoy["v"], sm, decoy["q"], kc_c, vc_c, bt, cl, st.scale, err_flag=flag,
                    options=pa.DecodeOptions(groups=groups, operands=ops.data_ptr()))
    torch.cuda.synchronize()
    assert int(flag.item()) & pa.FLAG_BAD_VALUE


def test_store_decode_fp8_operands_read_at_run_time(pa):
    """pa_store_decode_fp8_ex with operands only: output and E4M3 pool bit-identical to the direct
    call, the operands in page-locked host memory and the call's own q / k / v a zero-filled decoy."""
    ctx = torch.randint(1, 3000, (29,), generator=torch.Generator().manual_seed(221)).tolist()
    fs = inputs.make_decode_fp8(ctx, num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=256,
                                dtype=torch.bfloat16, seed=222)
    st = fs.step
    real = {n: t.pin_memory() for n, t in dict(k=st.k_new, v=st.v_new, q=st.q).items()}
    decoy = {n: torch.zeros_like(t, device="cuda") for n, t in real.items()}
    sm, bt, cl = st.slot_mapping.cuda(), st.block_tables.cuda(), st.context_lens.cuda()
    kc_a, vc_a = fs.k_cache.cuda(), fs.v_cache.cuda()
    ref = pa.store_decode_fp8(real["k"], real["v"], sm, real["q"], kc_a, vc_a, bt, cl, st.scale, fs.k_scale,
                              fs.v_scale)
    ops = torch.tensor([real["q"].data_ptr(), real["k"].data_ptr(), real["v"].data_ptr()],
                       dtype=torch.int64).pin_memory()
    kc_b, vc_b = fs.k_cache.cuda(), fs.v_cache.cuda()
    got = pa.store_decode_fp8(decoy["k"], decoy["v"], sm, decoy["q"], kc_b, vc_b, bt, cl, st.scale, fs.k_scale,
                              fs.v_scale, operands=ops.data_ptr())
    torch.cuda.synchronize()
    assert_bit_equal(got, ref, "output through the operands array")
    assert torch.equal(kc_b.cpu(), kc_a.cpu()) and torch.equal(vc_b.cpu(), vc_a.cpu()), "pool differs"
