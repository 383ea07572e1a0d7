"""GPU parity of the E4M3 pool: pa_store_kv_fp8 (codes bit-exact against the
oracle's nearest-code search) and pa_decode_fp8 (within the attention
tolerance of the oracle's dequantise-then-attend).

Cases: the Qwen3-0.6B-like decode workload over an fp8 pool (every sequence
checked), GQA groups 1..8, block sizes 8..1024, empty and one-token contexts,
contexts on and off tile/page/partition boundaries, both query dtypes, every
rounding tie of the E4M3 grid, saturation, subnormals, NaN, and bad metadata
(flagged, never faulting)."""

import pytest
import torch

import oracle
from tests import inputs
from tests.gpu_cases import TOL, max_err

pytestmark = pytest.mark.gpu


def _e4m3_values() -> torch.Tensor:
    """Value of every non-negative finite E4M3 code (0x00 .. 0x7E), by the oracle."""
    lib = oracle.load()
    return torch.tensor([lib.oracle_e4m3_to_float(c) for c in range(0x7F)], dtype=torch.float64)


def _store_both(pa, k, v, kc, vc, slots, k_scale, v_scale):
    gk, gv = kc.cuda(), vc.cuda()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.store_kv_fp8(k.cuda(), v.cuda(), gk, gv, slots.cuda(), k_scale, v_scale, err_flag=flag)
    torch.cuda.synchronize()
    ok, ov = kc.clone(), vc.clone()
    oracle.store_kv_fp8(k, v, ok, ov, slots, k_scale, v_scale)
    return gk.cpu(), gv.cpu(), ok, ov, int(flag.item())


def _run_fp8_step(pa, fs, err_flag=None):
    s = fs.step
    kc, vc = fs.k_cache.cuda(), fs.v_cache.cuda()
    pa.store_kv_fp8(s.k_new.cuda(), s.v_new.cuda(), kc, vc, s.slot_mapping.cuda(), fs.k_scale, fs.v_scale,
                    err_flag=err_flag)
    out = pa.decode_fp8(s.q.cuda(), kc, vc, s.block_tables.cuda(), s.context_lens.cuda(), s.scale, fs.k_scale,
                        fs.v_scale, err_flag=err_flag)
    torch.cuda.synchronize()
    return out, kc, vc


def _check_fp8_step(pa, fs, rows=None):
    s = fs.step
    out, kc, vc = _run_fp8_step(pa, fs)
    okc, ovc = fs.k_cache.clone(), fs.v_cache.clone()
    oracle.store_kv_fp8(s.k_new, s.v_new, okc, ovc, s.slot_mapping, fs.k_scale, fs.v_scale)
    assert torch.equal(kc.cpu(), okc), "k codes after the store"
    assert torch.equal(vc.cpu(), ovc), "v codes after the store"
    idx = torch.arange(s.batch) if rows is None else torch.tensor(rows)
    ref = oracle.decode_fp8(s.q[idx], okc, ovc, s.block_tables[idx], s.context_lens[idx], s.scale, fs.k_scale,
                            fs.v_scale)
    err = max_err(out[idx.cuda()], ref)
    assert err <= TOL[s.q.dtype], f"max |err| {err} > {TOL[s.q.dtype]}"
    return err


# ---- the quantising store


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_store_fp8_random_rows_bit_exact(pa, dtype):
    gen = torch.Generator().manual_seed(71)
    T, hkv, d, bs = 3000, 8, 128, 16
    nb = (T * 5 // 4 + bs - 1) // bs
    slots = torch.randperm(nb * bs, generator=gen)[:T].to(torch.int32)
    slots[::97] = -1  # padding rows are skipped
    k = (torch.randn(T, hkv, d, generator=gen) * 3).to(dtype)
    v = (torch.randn(T, hkv, d, generator=gen) * 3).to(dtype)
    kc = torch.full((nb, bs, hkv, d), inputs.FP8_SENTINEL, dtype=torch.uint8)
    vc = kc.clone()
    gk, gv, ok, ov, flag = _store_both(pa, k, v, kc, vc, slots, inputs.FP8_K_SCALE, inputs.FP8_V_SCALE)
    assert flag == 0
    assert torch.equal(gk, ok) and torch.equal(gv, ov)


@pytest.mark.parametrize("dtype", [torch.bfloat16, torch.float16])
def test_store_fp8_ties_saturation_subnormals(pa, dtype):
    """Scale 1: every midpoint between neighbouring E4M3 values that the input dtype
    holds exactly (ties go to the even code), values just either side of them,
    saturation above 448 (and infinities), zeros of both signs and subnormals."""
    vals = _e4m3_values()
    mids = ((vals[:-1] + vals[1:]) / 2).to(dtype)  # 5 significant bits: exact in fp16 and bf16
    bits = mids.view(torch.int16)
    above, below = (bits + 1).view(dtype), (bits - 1).view(dtype)  # the dtype's neighbours of each tie
    extra = torch.tensor([448.0, 464.0, 480.0, 500.0, 1e4, float("inf"), 0.0, -0.0, 2.0 ** -10, 2.0 ** -11,
                          3 * 2.0 ** -11], dtype=torch.float64)
    ex16 = extra.to(dtype)
    ex16 = ex16[ex16.double() == extra]  # only values the input dtype holds exactly
    x16 = torch.cat([vals.to(dtype), mids, above, below, ex16])
    x16 = torch.cat([x16, -x16])
    n = x16.numel()
    row = 128
    T = (n + row - 1) // row
    k = torch.zeros(T * row, dtype=dtype)
    k[:n] = x16
    k = k.view(T, 1, row)
    v = k.flip(0).contiguous()
    slots = torch.arange(T, dtype=torch.int32)
    kc = torch.zeros(T, 1, 1, row, dtype=torch.uint8)
    gk, gv, ok, ov, flag = _store_both(pa, k, v, kc, kc.clone(), slots, 1.0, 1.0)
    assert flag == 0
    assert torch.equal(gk, ok) and torch.equal(gv, ov)


def test_store_fp8_nan_stays_nan(pa):
    k = torch.full((2, 1, 128), float("nan"), dtype=torch.bfloat16)
    slots = torch.tensor([0, 1], dtype=torch.int32)
    kc = torch.zeros(2, 1, 1, 128, dtype=torch.uint8)
    gk, gv, ok, ov, _ = _store_both(pa, k, k.clone(), kc, kc.clone(), slots, 0.5, 0.5)
    for t in (gk, gv, ok, ov):
        assert bool(((t & 0x7F) == 0x7F).all()), "a NaN input must give a NaN code"


def test_store_fp8_bad_slot_is_flagged(pa):
    gen = torch.Generator().manual_seed(72)
    k = torch.randn(4, 2, 128, generator=gen).to(torch.bfloat16)
    kc = torch.zeros(4, 8, 2, 128, dtype=torch.uint8)
    slots = torch.tensor([0, 5, 32, -7], dtype=torch.int32)  # 32 = pool rows, -7 invalid
    gk, gv = kc.cuda(), kc.clone().cuda()
    f = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.store_kv_fp8(k.cuda(), k.cuda(), gk, gv, slots.cuda(), 1.0, 1.0, err_flag=f)
    torch.cuda.synchronize()
    assert int(f.item()) & pa.FLAG_BAD_SLOT
    ok = kc.clone()
    oracle.store_kv_fp8(k[:2], k[:2], ok, ok.clone(), slots[:2], 1.0, 1.0)
    assert torch.equal(gk.cpu(), ok), "valid rows are stored, invalid ones skipped"


# ---- decode over the fp8 pool


def test_decode_fp8_qwen3_0p6b_full(pa):
    fs = inputs.qwen3_0p6b_decode_fp8()
    err = _check_fp8_step(pa, fs)
    print(f"qwen3_0p6b_decode_fp8: max|err| = {err:.3e}")


@pytest.mark.parametrize("dtype", [torch.float16, torch.bfloat16])
@pytest.mark.parametrize("hq,hkv", [(8, 8), (8, 4), (8, 2), (8, 1), (32, 8)])
def test_decode_fp8_shapes(pa, dtype, hq, hkv):
    ctx = [0, 1, 2, 15, 16, 17, 63, 64, 65, 127, 128, 129, 500, 1023, 1024, 1025, 3000]
    fs = inputs.make_decode_fp8(ctx, num_q_heads=hq, num_kv_heads=hkv, head_dim=128, block_size=16, dtype=dtype,
                                seed=131 + hq + hkv)
    _check_fp8_step(pa, fs)


@pytest.mark.parametrize("bs", [8, 32, 64, 128, 512, 1024])
def test_decode_fp8_block_sizes(pa, bs):
    ctx = [1, bs - 1, bs, bs + 1, 3 * bs + 5, 2100]
    fs = inputs.make_decode_fp8(ctx, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=bs,
                                dtype=torch.bfloat16, seed=140 + bs)
    _check_fp8_step(pa, fs)


def test_decode_fp8_long_context_split(pa):
    fs = inputs.make_decode_fp8([32768, 20000], num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=256,
                                dtype=torch.bfloat16, seed=150)
    _check_fp8_step(pa, fs)


def test_decode_fp8_shared_prefix(pa):
    ctx = torch.randint(513, 2049, (32,), generator=torch.Generator().manual_seed(151)).tolist()
    fs = inputs.make_decode_fp8(ctx, num_q_heads=32, num_kv_heads=8, head_dim=128, block_size=16,
                                dtype=torch.bfloat16, seed=152, share_groups=8, share_tokens=512)
    _check_fp8_step(pa, fs)


def test_decode_fp8_scales_apply(pa):
    """Doubling k_scale with codes fixed doubles the scores: same as halving the
    softmax temperature through `scale`; doubling v_scale doubles the output."""
    fs = inputs.make_decode_fp8([300, 77], num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                dtype=torch.float16, seed=153)
    s = fs.step
    kc, vc = fs.k_cache.cuda(), fs.v_cache.cuda()
    pa.store_kv_fp8(s.k_new.cuda(), s.v_new.cuda(), kc, vc, s.slot_mapping.cuda(), fs.k_scale, fs.v_scale)
    args = (s.q.cuda(), kc, vc, s.block_tables.cuda(), s.context_lens.cuda())
    a = pa.decode_fp8(*args, s.scale, 2 * fs.k_scale, fs.v_scale)
    b = pa.decode_fp8(*args, 2 * s.scale, fs.k_scale, fs.v_scale)
    c = pa.decode_fp8(*args, s.scale, fs.k_scale, fs.v_scale)
    e = pa.decode_fp8(*args, s.scale, fs.k_scale, 2 * fs.v_scale)
    torch.cuda.synchronize()
    assert torch.equal(a, b)
    assert torch.equal(e.float(), (2 * c.float()).to(e.dtype).float())


def test_decode_fp8_bad_block_is_flagged(pa):
    fs = inputs.make_decode_fp8([40, 100], num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                dtype=torch.bfloat16, seed=154)
    s = fs.step
    bt = s.block_tables.clone()
    bt[1, 2] = fs.k_cache.shape[0] + 5
    kc, vc = fs.k_cache.cuda(), fs.v_cache.cuda()
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    pa.decode_fp8(s.q.cuda(), kc, vc, bt.cuda(), s.context_lens.cuda(), s.scale, fs.k_scale, fs.v_scale,
                  err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) & pa.FLAG_BAD_BLOCK


def test_decode_fp8_accepts_float8_tensors(pa):
    fs = inputs.make_decode_fp8([90, 33], num_q_heads=8, num_kv_heads=8, head_dim=128, block_size=16,
                                dtype=torch.bfloat16, seed=155)
    s = fs.step
    out_u8, kc, vc = _run_fp8_step(pa, fs)
    out_f8 = pa.decode_fp8(s.q.cuda(), kc.view(torch.float8_e4m3fn), vc.view(torch.float8_e4m3fn),
                           s.block_tables.cuda(), s.context_lens.cuda(), s.scale, fs.k_scale, fs.v_scale)
    torch.cuda.synchronize()
    assert torch.equal(out_u8, out_f8)


# ---- the fused step (pa_store_decode_fp8)


def _fused_fp8(pa, fs, err_flag=None):
    s = fs.step
    kc, vc = fs.k_cache.cuda(), fs.v_cache.cuda()
    out = pa.store_decode_fp8(s.k_new.cuda(), s.v_new.cuda(), s.slot_mapping.cuda(), s.q.cuda(), kc, vc,
                              s.block_tables.cuda(), s.context_lens.cuda(), s.scale, fs.k_scale, fs.v_scale,
                              err_flag=err_flag)
    torch.cuda.synchronize()
    return out, kc, vc


@pytest.mark.parametrize("name", ["qwen3_0p6b", "shapes_bs16", "bs8_long"])
def test_store_decode_fp8_equals_store_then_decode(pa, name):
    if name == "qwen3_0p6b":
        fs = inputs.qwen3_0p6b_decode_fp8()
    elif name == "shapes_bs16":
        fs = inputs.make_decode_fp8([0, 1, 2, 15, 16, 17, 63, 64, 65, 500, 1025, 3000], num_q_heads=32,
                                    num_kv_heads=8, head_dim=128, block_size=16, dtype=torch.float16, seed=160)
    else:
        fs = inputs.make_decode_fp8([8, 9, 4000, 777], num_q_heads=8, num_kv_heads=1, head_dim=128, block_size=8,
                                    dtype=torch.bfloat16, seed=161)
    s = fs.step
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    fused, kc, vc = _fused_fp8(pa, fs, err_flag=flag)
    assert int(flag.item()) == 0
    two, kc2, vc2 = _run_fp8_step(pa, fs)
    assert torch.equal(kc, kc2) and torch.equal(vc, vc2), "pools differ between fused and two-call steps"
    assert torch.equal(fused.view(torch.int16), two.view(torch.int16)), "outputs differ"
    okc, ovc = fs.k_cache.clone(), fs.v_cache.clone()
    oracle.store_kv_fp8(s.k_new, s.v_new, okc, ovc, s.slot_mapping, fs.k_scale, fs.v_scale)
    assert torch.equal(kc.cpu(), okc)
    ref = oracle.decode_fp8(s.q, okc, ovc, s.block_tables, s.context_lens, s.scale, fs.k_scale, fs.v_scale)
    assert max_err(fused, ref) <= TOL[s.q.dtype]


def test_store_decode_fp8_wrong_slot_is_flagged_and_not_stored(pa):
    fs = inputs.make_decode_fp8([40, 100, 7], num_q_heads=8, num_kv_heads=2, head_dim=128, block_size=16,
                                dtype=torch.bfloat16, seed=162)
    s = fs.step
    bad = s.slot_mapping.clone()
    bad[1] = bad[1] - 1  # the slot of position L-2: not this step's token
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    kc, vc = fs.k_cache.cuda(), fs.v_cache.cuda()
    pa.store_decode_fp8(s.k_new.cuda(), s.v_new.cuda(), bad.cuda(), s.q.cuda(), kc, vc, s.block_tables.cuda(),
                        s.context_lens.cuda(), s.scale, fs.k_scale, fs.v_scale, err_flag=flag)
    torch.cuda.synchronize()
    assert int(flag.item()) & pa.FLAG_BAD_SLOT
    row = lambda c, slot: c.view(-1, c.shape[2] * c.shape[3])[slot]  # noqa: E731
    assert torch.equal(row(kc.cpu(), int(bad[1])), row(fs.k_cache, int(bad[1]))), "the wrong slot was written"


def test_store_decode_fp8_graph_replay(pa):
    """The fused fp8 step captured in a CUDA graph and replayed gives the eager result."""
    fs = inputs.make_decode_fp8([300, 1000, 77, 4096], num_q_heads=16, num_kv_heads=8, head_dim=128,
                                block_size=256, dtype=torch.bfloat16, seed=163)
    s = fs.step
    d = {k: t.cuda() for k, t in dict(k=s.k_new, v=s.v_new, sm=s.slot_mapping, q=s.q, bt=s.block_tables,
                                      cl=s.context_lens).items()}
    kc, vc = fs.k_cache.cuda(), fs.v_cache.cuda()
    out = torch.empty_like(d["q"])
    nbytes = pa.decode_fp8_workspace_bytes(4, 16, 8, 128, s.block_tables.shape[1], 256)
    ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")

    def step():
        pa.store_decode_fp8(d["k"], d["v"], d["sm"], d["q"], kc, vc, d["bt"], d["cl"], s.scale, fs.k_scale,
                            fs.v_scale, out=out, workspace=ws)
    st = torch.cuda.Stream()
    st.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(st):
        step()
    torch.cuda.current_stream().wait_stream(st)
    torch.cuda.synchronize()
    eager = out.clone()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        step()
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), eager.view(torch.int16))
