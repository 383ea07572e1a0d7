"""The oracle built with -fopenmp (the benchmark's all-core CPU baseline) gives
the same bits as the usual single-threaded build: the threads only divide
independent rows (gathered positions, (query row, head) attention rows), each
row's arithmetic and its order unchanged."""

import os

import pytest
import torch

import oracle
from tests import inputs


@pytest.fixture(scope="module")
def omp():
    os.environ.setdefault("OMP_NUM_THREADS", "4")
    return oracle.load_omp()


def _store(st):
    kc, vc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
    oracle.store_kv(st.k_new, st.v_new, kc, vc, st.slot_mapping)
    return kc, vc


def test_openmp_decode_is_bit_identical(omp):
    st = inputs.make_decode([1, 17, 300, 2049, 0, 513], num_q_heads=32, num_kv_heads=8, head_dim=128,
                            block_size=16, dtype=torch.bfloat16, seed=81)
    kc, vc = _store(st)
    a = oracle.decode(st.q, kc, vc, st.block_tables, st.context_lens, st.scale)
    b = oracle.decode(st.q, kc, vc, st.block_tables, st.context_lens, st.scale, lib=omp)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_openmp_prefill_is_bit_identical(omp):
    st, _ = inputs.make_prefill([0, 300, 1000], [40, 64, 7], num_q_heads=8, num_kv_heads=2, head_dim=64,
                                block_size=16, dtype=torch.float16, seed=82)
    kc, vc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
    oracle.store_kv(st.k_new, st.v_new, kc, vc, st.slot_mapping)
    args = (st.q, st.k_new, st.v_new, kc, vc, st.cu_seqlens_q, st.cu_seqlens_k, st.block_tables, st.scale)
    a = oracle.prefill_paged(*args)
    b = oracle.prefill_paged(*args, lib=omp)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_openmp_decode_fp8_is_bit_identical(omp):
    fs = inputs.make_decode_fp8([5, 700, 64], num_q_heads=16, num_kv_heads=8, head_dim=128, block_size=64,
                                dtype=torch.bfloat16, seed=83)
    st = fs.step
    args = (st.q, fs.k_cache, fs.v_cache, st.block_tables, st.context_lens, st.scale, fs.k_scale, fs.v_scale)
    a = oracle.decode_fp8(*args)
    b = oracle.decode_fp8(*args, lib=omp)
    assert torch.equal(a.view(torch.int32), b.view(torch.int32))


def test_openmp_rejects_what_the_serial_build_rejects(omp):
    st = inputs.make_decode([40, 40], num_q_heads=4, num_kv_heads=2, head_dim=64, block_size=16,
                            dtype=torch.float16, seed=84)
    bt = st.block_tables.clone()
    bt[1, 1] = -1
    for lib in (None, omp):
        with pytest.raises(oracle.OracleError):
            oracle.decode(st.q, st.pool.k_cache, st.pool.v_cache, bt, st.context_lens, st.scale, lib=lib)
