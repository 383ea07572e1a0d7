"""GPU parity of pa_mixed_step (store + chunked prefill + decode of one step), with the prefill
and the decode on two disjoint SM partitions (pa_sm_split) and without: bit-identical to the
three separate calls, and within tolerance of the oracle."""

import pytest
import torch

import oracle
from tests import inputs
from tests.gpu_cases import TOL, assert_bit_equal, max_err

pytestmark = pytest.mark.gpu


def _device(m):
    pf, st = m.prefill, m.decode
    d = dict(k=m.k_new, v=m.v_new, sm=m.slot_mapping, pq=pf.q, cuq=pf.cu_seqlens_q, cuk=pf.cu_seqlens_k,
             pbt=pf.block_tables, dq=st.q, dbt=st.block_tables, cl=st.context_lens)
    return {n: t.cuda() for n, t in d.items()}


def _separate(pa, m):
    pf, st = m.prefill, m.decode
    d = _device(m)
    kc, vc = pf.pool.k_cache.cuda(), pf.pool.v_cache.cuda()
    pa.store_kv(d["k"], d["v"], kc, vc, d["sm"])
    pout = pa.prefill_paged(d["pq"], None, None, kc, vc, d["cuq"], d["cuk"], pf.max_seqlen_q, pf.max_seqlen_k,
                            d["pbt"], pf.scale)
    dout = pa.decode(d["dq"], kc, vc, d["dbt"], d["cl"], st.scale)
    torch.cuda.synchronize()
    return pout, dout, kc, vc


def _mixed(pa, m, split):
    pf, st = m.prefill, m.decode
    d = _device(m)
    kc, vc = pf.pool.k_cache.cuda(), pf.pool.v_cache.cuda()
    pout, dout = pa.mixed_step(d["k"], d["v"], d["sm"], d["pq"], d["cuq"], d["cuk"], pf.max_seqlen_q,
                               pf.max_seqlen_k, d["pbt"], d["dq"], d["dbt"], d["cl"], kc, vc, pf.scale, split=split)
    torch.cuda.synchronize()
    return pout, dout, kc, vc


@pytest.fixture(scope="module")
def split(pa):
    s = pa.SmSplit(96)
    yield s
    s.close()


@pytest.mark.parametrize("use_split", [True, False])
def test_mixed_step_equals_separate_calls(pa, split, use_split):
    m = inputs.mixed_chunked_prefill()
    ref = _separate(pa, m)
    got = _mixed(pa, m, split if use_split else None)
    for name, a, b in zip(("prefill out", "decode out", "k_cache", "v_cache"), got, ref):
        assert_bit_equal(a, b, f"mixed step vs separate calls: {name}")


@pytest.mark.parametrize("use_split", [True, False])
def test_mixed_step_small_against_oracle(pa, split, use_split):
    m = inputs.mixed_chunked_prefill(seed=41, n_prefill=3, chunk=96, n_decode=7, max_prefix=700)
    pf, st = m.prefill, m.decode
    pout, dout, kc, vc = _mixed(pa, m, split if use_split else None)
    okc, ovc = pf.pool.k_cache.clone(), pf.pool.v_cache.clone()
    oracle.store_kv(m.k_new, m.v_new, okc, ovc, m.slot_mapping)
    assert_bit_equal(kc, okc, "k_cache after the mixed step's store")
    assert_bit_equal(vc, ovc, "v_cache after the mixed step's store")
    pref = oracle.prefill_paged(pf.q, pf.k_new, pf.v_new, okc, ovc, pf.cu_seqlens_q, pf.cu_seqlens_k,
                                pf.block_tables, pf.scale)
    dref = oracle.decode(st.q, okc, ovc, st.block_tables, st.context_lens, st.scale)
    assert max_err(pout, pref) <= TOL[pf.q.dtype]
    assert max_err(dout, dref) <= TOL[st.q.dtype]


def test_sm_split_sizes(pa, split):
    assert split.sms[0] == 96 and split.sms[0] + split.sms[1] == torch.cuda.get_device_properties(0).multi_processor_count
    for bad in (0, 12, 4, split.sms[0] + split.sms[1]):
        with pytest.raises(pa.PagedAttentionError):
            pa.SmSplit(bad)


def test_mixed_step_with_one_side_empty(pa, split):
    """A step with no decode sequences (store + prefill) or no prefill sequences (store + decode):
    the split is not used and the results equal the separate calls."""
    m = inputs.mixed_chunked_prefill(seed=43, n_prefill=2, chunk=64, n_decode=5, max_prefix=400)
    pf, st = m.prefill, m.decode
    n_pf = int(pf.cu_seqlens_q[-1])  # the prefill tokens come first in the step's store
    pout, dout, kc, vc = _separate(pa, m)
    d = _device(m)
    # no decode sequences: store only the prefill tokens, then the prefill
    kc1, vc1 = pf.pool.k_cache.cuda(), pf.pool.v_cache.cuda()
    empty_q = d["dq"][:0]
    p1, d1 = pa.mixed_step(d["k"][:n_pf], d["v"][:n_pf], d["sm"][:n_pf].contiguous(), d["pq"], d["cuq"], d["cuk"],
                           pf.max_seqlen_q, pf.max_seqlen_k, d["pbt"], empty_q, d["dbt"][:0], d["cl"][:0], kc1, vc1,
                           pf.scale, split=split)
    torch.cuda.synchronize()
    assert d1.shape[0] == 0
    assert_bit_equal(p1, pout, "prefill out without decode sequences")
    # no prefill sequences: store only the decode tokens, then the decode
    kc2, vc2 = pf.pool.k_cache.cuda(), pf.pool.v_cache.cuda()
    cu0 = torch.zeros(1, dtype=torch.int32, device="cuda")
    p2, d2 = pa.mixed_step(d["k"][n_pf:], d["v"][n_pf:], d["sm"][n_pf:].contiguous(), d["pq"][:0], cu0, cu0, 0, 0,
                           d["pbt"][:0], d["dq"], d["dbt"], d["cl"], kc2, vc2, st.scale, split=split)
    torch.cuda.synchronize()
    assert p2.shape[0] == 0
    assert_bit_equal(d2, dout, "decode out without prefill sequences")


@pytest.mark.parametrize("use_split", [True, False])
def test_mixed_step_outputs_in_pinned_host_memory(pa, split, use_split):
    # both outputs page-locked on the host, written by the kernels over the CPU-GPU link: the same
    # bits as device outputs; a pageable host output is refused before any launch
    m = inputs.mixed_chunked_prefill()
    pf, st = m.prefill, m.decode
    ref = _mixed(pa, m, split if use_split else None)
    d = _device(m)
    kc, vc = pf.pool.k_cache.cuda(), pf.pool.v_cache.cuda()
    pout = torch.full(tuple(pf.q.shape), float("nan"), dtype=pf.q.dtype).pin_memory()
    dout = torch.full(tuple(st.q.shape), float("nan"), dtype=st.q.dtype).pin_memory()
    pa.mixed_step(d["k"], d["v"], d["sm"], d["pq"], d["cuq"], d["cuk"], pf.max_seqlen_q, pf.max_seqlen_k, d["pbt"],
                  d["dq"], d["dbt"], d["cl"], kc, vc, pf.scale, prefill_out=pout, decode_out=dout,
                  split=split if use_split else None)
    torch.cuda.synchronize()
    assert_bit_equal(pout, ref[0].cpu(), "prefill output in pinned memory")
    assert_bit_equal(dout, ref[1].cpu(), "decode output in pinned memory")
    with pytest.raises(ValueError):
        pa.mixed_step(d["k"], d["v"], d["sm"], d["pq"], d["cuq"], d["cuk"], pf.max_seqlen_q, pf.max_seqlen_k,
                      d["pbt"], d["dq"], d["dbt"], d["cl"], kc, vc, pf.scale,
                      prefill_out=torch.empty(tuple(pf.q.shape), dtype=pf.q.dtype), split=None)
    with pytest.raises(ValueError):  # the prefill's q is read by TMA: device memory only
        pa.mixed_step(d["k"], d["v"], d["sm"], pf.q.pin_memory(), d["cuq"], d["cuk"], pf.max_seqlen_q,
                      pf.max_seqlen_k, d["pbt"], d["dq"], d["dbt"], d["cl"], kc, vc, pf.scale, split=None)
