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
