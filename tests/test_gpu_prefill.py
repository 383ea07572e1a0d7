"""GPU parity of pa_prefill_paged (after pa_store_kv) against the oracle.

Small cases run whole; the mixed chunked-prefill workload (8 x 512-token
chunks over prefixes up to 3584 tokens) runs at full size through the call
bench.py times and is compared whole, every row of every sequence, against
the oracle's OpenMP build (bit-identical to the single-threaded build; the
step is ~137 GFLOP).
"""

import pytest
import torch

import oracle
from tests import inputs
from tests.gpu_cases import TOL, assert_bit_equal, max_err

pytestmark = pytest.mark.gpu


def run_prefill_gpu(pa, st, use_table=True, err_flag=None):
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    kn, vn = st.k_new.cuda(), st.v_new.cuda()
    pa.store_kv(kn, vn, kc, vc, st.slot_mapping.cuda(), err_flag=err_flag)
    bt = st.block_tables.cuda() if use_table else None
    out = pa.prefill_paged(st.q.cuda(), kn, vn, kc, vc, st.cu_seqlens_q.cuda(), st.cu_seqlens_k.cuda(),
                           st.max_seqlen_q, st.max_seqlen_k, bt, st.scale, err_flag=err_flag)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_after_store(st):
    okc, ovc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
    oracle.store_kv(st.k_new, st.v_new, okc, ovc, st.slot_mapping)
    return okc, ovc


def check_prefill_full(pa, st, use_table=True):
    out, kc, vc = run_prefill_gpu(pa, st, use_table)
    okc, ovc = oracle_after_store(st)
    assert_bit_equal(kc, okc, "k_cache after store")
    ref = oracle.prefill_paged(st.q, st.k_new, st.v_new, okc, ovc, st.cu_seqlens_q, st.cu_seqlens_k,
                               st.block_tables if use_table else None, st.scale)
    err = max_err(out, ref)
    assert err <= TOL[st.q.dtype], f"max |err| {err}"
    return err


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
@pytest.mark.parametrize("head_dim", [128, 64])
@pytest.mark.parametrize("bs", [16, 256])
def test_prefill_over_prefix_small(pa, dtype, head_dim, bs):
    # prefixes on and off tile boundaries, chunks from 1 row to several 128-row tiles
    prefix = [0, 5, 128, 300, 1000, 77]
    chunk = [7, 128, 200, 1, 129, 300]
    st, _ = inputs.make_prefill(prefix, chunk, num_q_heads=8, num_kv_heads=2, head_dim=head_dim, block_size=bs,
                                dtype=dtype, seed=70 + bs + head_dim)
    err = check_prefill_full(pa, st)
    print(f"prefill {dtype} D{head_dim} bs{bs}: max|err| {err:.2e}")


@pytest.mark.parametrize("hq,hkv", [(4, 4), (8, 1), (32, 8)])
@pytest.mark.parametrize("bs", [8, 64, 1024])
def test_prefill_group_sizes_and_block_sizes(pa, hq, hkv, bs):
    st, _ = inputs.make_prefill([33, 0, 640], [100, 64, 257], num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                                block_size=bs, dtype=torch.bfloat16, seed=80 + hq + bs)
    check_prefill_full(pa, st)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_prefill_without_block_table(pa, dtype):
    # fresh prompts: no cached prefix, keys are the packed k/v rows
    st, _ = inputs.make_prefill([0, 0, 0], [11, 300, 129], num_q_heads=8, num_kv_heads=4, head_dim=128,
                                block_size=16, dtype=dtype, seed=90)
    check_prefill_full(pa, st, use_table=False)


def test_prefill_table_and_packed_agree_without_prefix(pa):
    st, _ = inputs.make_prefill([0, 0], [200, 77], num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                dtype=torch.bfloat16, seed=91)
    a, _, _ = run_prefill_gpu(pa, st, use_table=True)
    b, _, _ = run_prefill_gpu(pa, st, use_table=False)
    assert_bit_equal(a, b, "paged vs packed keys")


def test_prefill_single_query_matches_decode(pa):
    st, _ = inputs.make_prefill([500, 31, 4000], [1, 1, 1], num_q_heads=32, num_kv_heads=8, head_dim=128,
                                block_size=256, dtype=torch.bfloat16, seed=92)
    out, kc, vc = run_prefill_gpu(pa, st)
    ctx = (st.cu_seqlens_k[1:] - st.cu_seqlens_k[:-1]).to(torch.int32)
    dec = pa.decode(st.q.cuda(), kc, vc, st.block_tables.cuda(), ctx.cuda(), st.scale)
    torch.cuda.synchronize()
    assert max_err(out, dec.cpu().float()) <= TOL[torch.bfloat16]


def test_prefill_mixed_workload_every_row(pa):
    # the full mixed chunked-prefill workload, every output row of every sequence against the
    # oracle (its OpenMP build, bit-identical to the single-threaded one, keeps this to seconds)
    m = inputs.mixed_chunked_prefill()
    st = m.prefill
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.store_kv(m.k_new.cuda(), m.v_new.cuda(), kc, vc, m.slot_mapping.cuda())
    out = pa.prefill_paged(st.q.cuda(), st.k_new.cuda(), st.v_new.cuda(), kc, vc, st.cu_seqlens_q.cuda(),
                           st.cu_seqlens_k.cuda(), st.max_seqlen_q, st.max_seqlen_k, st.block_tables.cuda(),
                           st.scale)
    torch.cuda.synchronize()
    okc, ovc = p.k_cache.clone(), p.v_cache.clone()
    oracle.store_kv(m.k_new, m.v_new, okc, ovc, m.slot_mapping)
    assert_bit_equal(kc, okc, "k_cache after the mixed store")
    assert_bit_equal(vc, ovc, "v_cache after the mixed store")
    ref = oracle.prefill_paged(st.q, st.k_new, st.v_new, okc, ovc, st.cu_seqlens_q, st.cu_seqlens_k,
                               st.block_tables, st.scale, lib=oracle.load_omp())
    out = out.cpu()
    cq = st.cu_seqlens_q.tolist()
    errs = [max_err(out[cq[i]:cq[i + 1]], ref[cq[i]:cq[i + 1]]) for i in range(len(cq) - 1)]
    assert max(errs) <= TOL[torch.bfloat16], f"max |err| per sequence {errs}"
    prefixes = (st.cu_seqlens_k[1:] - st.cu_seqlens_k[:-1] - (st.cu_seqlens_q[1:] - st.cu_seqlens_q[:-1])).tolist()
    print(f"mixed workload prefill, all {cq[-1]} rows (prefixes {prefixes}): max|err| {max(errs):.2e}")


@pytest.mark.parametrize("hq,hkv,bs", [(32, 8, 8), (8, 1, 256), (4, 4, 16)])
def test_prefill_row_seeing_one_key_returns_its_value_row(pa, hq, hkv, bs):
    # The first query row of a fresh prompt sees one key, its own: weight 1, so the output is that
    # token's value row for every head of the group, bit for bit (the row maximum, the exponent and
    # the sum must agree exactly; any column of the 128-key tile leaking into the maximum shows).
    chunk = [1, 64, 128, 129, 300, 7]
    st, _ = inputs.make_prefill([0] * len(chunk), chunk, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                                block_size=bs, dtype=torch.bfloat16, seed=96 + bs)
    out, _, _ = run_prefill_gpu(pa, st)
    out = out.cpu()
    for r in st.cu_seqlens_q[:-1].tolist():
        expect = st.v_new[r].repeat_interleave(hq // hkv, dim=0)
        assert_bit_equal(out[r], expect, f"row {r}")


@pytest.mark.parametrize("max_ctas", [1, 3, 16])
def test_prefill_few_ctas_many_items_each(pa, max_ctas):
    # the persistent grid capped at a few CTAs: each works through many items, so the K/V stream
    # runs across item boundaries (short and long items, chunks of 1 row to several tiles, an empty
    # chunk, block sizes below the tile); results equal the oracle and, bit for bit, the full grid
    prefix = [0, 5, 300, 1000, 77, 2000, 0]
    chunk = [7, 200, 1, 129, 300, 0, 260]
    st, _ = inputs.make_prefill(prefix, chunk, num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=64,
                                dtype=torch.bfloat16, seed=94 + max_ctas)
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.store_kv(st.k_new.cuda(), st.v_new.cuda(), kc, vc, st.slot_mapping.cuda())
    args = (st.q.cuda(), None, None, kc, vc, st.cu_seqlens_q.cuda(), st.cu_seqlens_k.cuda(), st.max_seqlen_q,
            st.max_seqlen_k, st.block_tables.cuda(), st.scale)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    few = pa.prefill_paged(*args, err_flag=flag, max_ctas=max_ctas)
    full = pa.prefill_paged(*args)
    torch.cuda.synchronize()
    assert int(flag.item()) == 0
    assert_bit_equal(few, full, f"max_ctas {max_ctas} vs the full grid")
    okc, ovc = oracle_after_store(st)
    ref = oracle.prefill_paged(st.q, st.k_new, st.v_new, okc, ovc, st.cu_seqlens_q, st.cu_seqlens_k,
                               st.block_tables, st.scale)
    assert max_err(few, ref) <= TOL[torch.bfloat16]


@pytest.mark.parametrize("dtype,head_dim,hq,hkv", [(torch.float16, 64, 4, 4), (torch.bfloat16, 128, 8, 1)])
def test_prefill_one_cta_without_gqa_pairs_and_packed_keys(pa, dtype, head_dim, hq, hkv):
    # one CTA for every item: heads one per item without GQA (hq == hkv), two per item with it;
    # keys from the packed rows (no block table)
    st, _ = inputs.make_prefill([0, 0, 0], [11, 300, 129], num_q_heads=hq, num_kv_heads=hkv, head_dim=head_dim,
                                block_size=16, dtype=dtype, seed=95 + hq)
    out = pa.prefill_paged(st.q.cuda(), st.k_new.cuda(), st.v_new.cuda(), st.pool.k_cache.cuda(),
                           st.pool.v_cache.cuda(), st.cu_seqlens_q.cuda(), st.cu_seqlens_k.cuda(), st.max_seqlen_q,
                           st.max_seqlen_k, None, st.scale, max_ctas=1)
    torch.cuda.synchronize()
    ref = oracle.prefill_paged(st.q, st.k_new, st.v_new, st.pool.k_cache, st.pool.v_cache, st.cu_seqlens_q,
                               st.cu_seqlens_k, None, st.scale)
    assert max_err(out, ref) <= TOL[dtype]


def test_prefill_mixed_workload_capped_grid_bit_equal(pa):
    # the full mixed workload on 40 CTAs (about 13 items each) equals the default grid bit for bit
    m = inputs.mixed_chunked_prefill()
    st = m.prefill
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.store_kv(m.k_new.cuda(), m.v_new.cuda(), kc, vc, m.slot_mapping.cuda())
    args = (st.q.cuda(), None, None, kc, vc, st.cu_seqlens_q.cuda(), st.cu_seqlens_k.cuda(), st.max_seqlen_q,
            st.max_seqlen_k, st.block_tables.cuda(), st.scale)
    a = pa.prefill_paged(*args, max_ctas=40)
    b = pa.prefill_paged(*args)
    torch.cuda.synchronize()
    assert_bit_equal(a, b, "40 CTAs vs the full grid")


def test_prefill_output_in_pinned_host_memory(pa):
    # out page-locked on the host, written by the epilogue's plain stores over the CPU-GPU link: the
    # same bits as a device out; host inputs (read by TMA) and a pageable out are refused up front
    st, _ = inputs.make_prefill([0, 300, 1200], [300, 129, 200], num_q_heads=8, num_kv_heads=2, head_dim=128,
                                block_size=64, dtype=torch.bfloat16, seed=241)
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.store_kv(st.k_new.cuda(), st.v_new.cuda(), kc, vc, st.slot_mapping.cuda())
    args = (st.q.cuda(), None, None, kc, vc, st.cu_seqlens_q.cuda(), st.cu_seqlens_k.cuda(), st.max_seqlen_q,
            st.max_seqlen_k, st.block_tables.cuda(), st.scale)
    ref = pa.prefill_paged(*args)
    out = torch.full(tuple(st.q.shape), float("nan"), dtype=st.q.dtype).pin_memory()
    pa.prefill_paged(*args, out=out)
    torch.cuda.synchronize()
    assert_bit_equal(out, ref.cpu(), "prefill output in pinned memory")
    with pytest.raises(ValueError):
        pa.prefill_paged(*args, out=torch.empty(tuple(st.q.shape), dtype=st.q.dtype))
    with pytest.raises(ValueError):
        pa.prefill_paged(st.q.pin_memory(), *args[1:])


def test_decode_refuses_host_operands(pa):
    st = inputs.make_decode([40, 90], num_q_heads=4, num_kv_heads=2, head_dim=128, block_size=16,
                            dtype=torch.bfloat16, seed=242)
    kc, vc = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    with pytest.raises(ValueError):
        pa.decode(st.q, kc, vc, st.block_tables.cuda(), st.context_lens.cuda(), st.scale)


def test_prefill_bad_metadata_is_flagged_not_fatal(pa):
    st, _ = inputs.make_prefill([40, 40], [30, 30], num_q_heads=4, num_kv_heads=2, head_dim=128, block_size=16,
                                dtype=torch.bfloat16, seed=93)
    bt = st.block_tables.clone()
    bt[0, 1] = -1
    bt[1, 2] = st.pool.num_blocks + 3
    kc, vc = st.pool.k_cache.cuda(), st.pool.v_cache.cuda()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.prefill_paged(st.q.cuda(), None, None, kc, vc, st.cu_seqlens_q.cuda(), st.cu_seqlens_k.cuda(),
                     st.max_seqlen_q, st.max_seqlen_k, bt.cuda(), st.scale, err_flag=flag)
    ck = st.cu_seqlens_k.clone()
    ck[2] = ck[1] + 10                      # context shorter than the query chunk
    pa.prefill_paged(st.q.cuda(), None, None, kc, vc, st.cu_seqlens_q.cuda(), ck.cuda(),
                     st.max_seqlen_q, st.max_seqlen_k, st.block_tables.cuda(), st.scale, err_flag=flag)
    torch.cuda.synchronize()
    f = int(flag.item())
    assert f & pa.FLAG_BAD_BLOCK and f & pa.FLAG_BAD_LENGTH and not f & pa.FLAG_TIMEOUT
    check_prefill_full(pa, st)
