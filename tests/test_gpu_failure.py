"""Failure detection on the GPU without a fault: a bounded wait that nothing satisfies gives up,
reports PA_FLAG_TIMEOUT through the caller's flag, and the context stays usable (a decode right
after it matches the oracle)."""

import pytest
import torch

import oracle
from tests import inputs
from tests.gpu_cases import TOL, max_err

pytestmark = pytest.mark.gpu


def test_bounded_wait_times_out_with_a_status(pa):
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.selftest_wait_timeout(err, max_cycles=2_000_000)  # about a millisecond
    torch.cuda.synchronize()
    assert int(err.item()) & pa.FLAG_TIMEOUT
    # the context is intact: a decode after the timeout is right
    st = inputs.tiny_decode()
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.store_kv(st.k_new.cuda(), st.v_new.cuda(), kc, vc, st.slot_mapping.cuda())
    out = pa.decode(st.q.cuda(), kc, vc, st.block_tables.cuda(), st.context_lens.cuda(), st.scale)
    torch.cuda.synchronize()
    okc, ovc = p.k_cache.clone(), p.v_cache.clone()
    oracle.store_kv(st.k_new, st.v_new, okc, ovc, st.slot_mapping)
    ref = oracle.decode(st.q, okc, ovc, st.block_tables, st.context_lens, st.scale)
    assert max_err(out, ref) <= TOL[st.q.dtype]
