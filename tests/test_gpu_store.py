"""GPU parity of pa_store_kv: the pool after the store is bit-identical to the
oracle's, on every workload's slot mapping and on the edge cases."""

import pytest
import torch

import oracle
from tests import inputs
from tests.gpu_cases import assert_bit_equal

pytestmark = pytest.mark.gpu


def _store_both(pa, k, v, kc, vc, slots, err_flag=None):
    dkc, dvc = kc.cuda(), vc.cuda()
    pa.store_kv(k.cuda() if not k.is_cuda else k, v.cuda() if not v.is_cuda else v, dkc, dvc, slots.cuda(),
                err_flag=err_flag)
    torch.cuda.synchronize()
    okc, ovc = kc.clone(), vc.clone()
    kk = k.cpu() if k.is_cuda else k
    vv = v.cpu() if v.is_cuda else v
    keep = slots >= 0 if err_flag is None else (slots >= 0) & (slots < kc.shape[0] * kc.shape[1])
    oracle.store_kv(kk, vv, okc, ovc, torch.where(keep, slots, torch.full_like(slots, -1)))
    return dkc, dvc, okc, ovc


@pytest.mark.parametrize("name", ["tiny_decode", "qwen3_0p6b_decode", "qwen3_8b_shared_decode",
                                  "long_context_decode"])
def test_store_decode_workloads(pa, name):
    st = inputs.WORKLOADS[name]()
    p = st.pool
    dkc, dvc, okc, ovc = _store_both(pa, st.k_new, st.v_new, p.k_cache, p.v_cache, st.slot_mapping)
    assert_bit_equal(dkc, okc, "k_cache")
    assert_bit_equal(dvc, ovc, "v_cache")


def test_store_mixed_step(pa):
    m = inputs.mixed_chunked_prefill()
    p = m.prefill.pool
    assert m.slot_mapping.numel() == 8 * 512 + 120
    dkc, dvc, okc, ovc = _store_both(pa, m.k_new, m.v_new, p.k_cache, p.v_cache, m.slot_mapping)
    assert_bit_equal(dkc, okc, "k_cache")
    assert_bit_equal(dvc, ovc, "v_cache")


def test_store_stress_16384_tokens(pa):
    k, v, kc, vc, slots = inputs.store_stress()
    dkc, dvc, okc, ovc = _store_both(pa, k, v, kc, vc, slots)
    assert_bit_equal(dkc, okc, "k_cache")
    assert_bit_equal(dvc, ovc, "v_cache")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
def test_store_strided_views_and_padding(pa, dtype):
    # k and v as views into a fused [T, (H_q + 2 H_kv), D] projection; some pad rows (-1)
    g = torch.Generator().manual_seed(21)
    T, hq, hkv, d, N, bs = 37, 8, 2, 64, 12, 16
    qkv = torch.randn(T, hq + 2 * hkv, d, generator=g).to(dtype).cuda()
    k, v = qkv[:, hq:hq + hkv], qkv[:, hq + hkv:]
    slots = torch.randperm(N * bs, generator=g)[:T].to(torch.int32)
    slots[::5] = -1
    kc = torch.full((N, bs, hkv, d), inputs.SENTINEL_BITS, dtype=torch.int16).view(dtype)
    vc = kc.clone()
    dkc, dvc, okc, ovc = _store_both(pa, k, v, kc, vc, slots)
    assert_bit_equal(dkc, okc, "k_cache")
    assert_bit_equal(dvc, ovc, "v_cache")


def test_store_unaligned_rows_take_the_narrow_path(pa):
    g = torch.Generator().manual_seed(22)
    T, hkv, d, N, bs = 9, 2, 64, 4, 8
    base = torch.randn(T * hkv * d + 1, generator=g).to(torch.bfloat16).cuda()
    k = base[1:].view(T, hkv, d)          # 2-byte aligned only
    v = base[:-1].view(T, hkv, d)
    slots = torch.randperm(N * bs, generator=g)[:T].to(torch.int32)
    kc = torch.zeros(N, bs, hkv, d, dtype=torch.bfloat16)
    dkc, dvc, okc, ovc = _store_both(pa, k, v, kc, kc.clone(), slots)
    assert_bit_equal(dkc, okc, "k_cache")
    assert_bit_equal(dvc, ovc, "v_cache")


def test_store_empty_and_all_padding(pa):
    kc = torch.zeros(2, 8, 1, 64, dtype=torch.float16, device="cuda")
    k = torch.ones(3, 1, 64, dtype=torch.float16, device="cuda")
    pa.store_kv(k[:0], k[:0], kc, kc.clone(), torch.empty(0, dtype=torch.int32, device="cuda"))
    pa.store_kv(k, k, kc, kc.clone(), torch.full((3,), -1, dtype=torch.int32, device="cuda"))
    torch.cuda.synchronize()
    assert not kc.any()


def test_store_out_of_range_slot_is_flagged_and_skipped(pa):
    g = torch.Generator().manual_seed(23)
    T, hkv, d, N, bs = 6, 2, 64, 4, 8
    k = torch.randn(T, hkv, d, generator=g).to(torch.float16)
    v = torch.randn(T, hkv, d, generator=g).to(torch.float16)
    slots = torch.tensor([0, 5, N * bs, 7, -3, 31], dtype=torch.int32)
    kc = torch.zeros(N, bs, hkv, d, dtype=torch.float16)
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    dkc, dvc, okc, ovc = _store_both(pa, k, v, kc, kc.clone(), slots, err_flag=flag)
    assert int(flag.item()) & pa.FLAG_BAD_SLOT
    assert_bit_equal(dkc, okc, "k_cache (valid rows written, bad ones skipped)")
    assert_bit_equal(dvc, ovc, "v_cache")


def test_store_from_pinned_host_rows(pa):
    """The new rows and slots in pinned host memory, read by the kernel directly: the pool equals the
    oracle's bit for bit; pageable host memory is refused."""
    k, v, kc, vc, slots = inputs.store_stress(tokens=2048)
    dkc, dvc = kc.cuda(), vc.cuda()
    pa.store_kv(k.pin_memory(), v.pin_memory(), dkc, dvc, slots.pin_memory())
    torch.cuda.synchronize()
    okc, ovc = kc.clone(), vc.clone()
    oracle.store_kv(k, v, okc, ovc, slots)
    assert_bit_equal(dkc, okc, "k_cache after a store from pinned host rows")
    assert_bit_equal(dvc, ovc, "v_cache after a store from pinned host rows")
    with pytest.raises(ValueError):
        pa.store_kv(k, v, dkc, dvc, slots)
