"""Helpers shared by the GPU parity tests: run a step through the CUDA path
and through the oracle on the same seeded inputs, and compare."""

from __future__ import annotations

import torch

import oracle

# Attention tolerances (max |err| for N(0,1) inputs, fp32 accumulation).
TOL = {torch.float16: 2e-3, torch.bfloat16: 1.5e-2}


def bits(t: torch.Tensor) -> torch.Tensor:
    """Raw 16-bit words (so NaN sentinels compare equal)."""
    return t.contiguous().view(torch.int16)


def assert_bit_equal(a: torch.Tensor, b: torch.Tensor, what: str):
    a, b = bits(a.cpu()), bits(b.cpu())
    if not torch.equal(a, b):
        bad = (a != b).nonzero()
        raise AssertionError(f"{what}: {bad.shape[0]} words differ, first at {bad[0].tolist()}")


def max_err(gpu_out: torch.Tensor, ref: torch.Tensor) -> float:
    g = gpu_out.cpu().float()
    assert not torch.isnan(g).any(), "NaN in GPU output"
    assert not torch.isnan(ref).any(), "NaN in oracle output"
    return float((g - ref).abs().max()) if g.numel() else 0.0


def run_decode_gpu(pa, st, dev="cuda", err_flag=None, options=None):
    """Store the step's new tokens and run decode on the GPU (with ``options``: through
    pa_decode_ex).  Returns (out, k_cache, v_cache) on the device."""
    p = st.pool
    kc, vc = p.k_cache.to(dev), p.v_cache.to(dev)
    pa.store_kv(st.k_new.to(dev), st.v_new.to(dev), kc, vc, st.slot_mapping.to(dev), err_flag=err_flag)
    out = pa.decode(st.q.to(dev), kc, vc, st.block_tables.to(dev), st.context_lens.to(dev), st.scale,
                    err_flag=err_flag, options=options)
    torch.cuda.synchronize()
    return out, kc, vc


def oracle_store(st_pool_k, st_pool_v, k_new, v_new, slots):
    kc, vc = st_pool_k.clone(), st_pool_v.clone()
    oracle.store_kv(k_new, v_new, kc, vc, slots)
    return kc, vc


def check_decode(pa, st, rows=None, options=None):
    """Full parity of one decode step: caches bit-exact after the store,
    attention within tolerance on all (or the sampled) sequences."""
    out, kc, vc = run_decode_gpu(pa, st, options=options)
    okc, ovc = oracle_store(st.pool.k_cache, st.pool.v_cache, st.k_new, st.v_new, st.slot_mapping)
    assert_bit_equal(kc, okc, "k_cache after store")
    assert_bit_equal(vc, ovc, "v_cache after store")
    if rows is None:
        ref = oracle.decode(st.q, okc, ovc, st.block_tables, st.context_lens, st.scale)
        got = out
    else:
        idx = torch.tensor(rows)
        ref = oracle.decode(st.q[idx], okc, ovc, st.block_tables[idx], st.context_lens[idx], st.scale)
        got = out[idx.to(out.device)]
    err = max_err(got, ref)
    assert err <= TOL[st.q.dtype], f"max |err| {err} > {TOL[st.q.dtype]}"
    return err
