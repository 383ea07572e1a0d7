"""GPU parity of pa_sample (temperature sampling by the exponential race)
against the oracle with the same Exp(1) noise, and statistical checks of the
in-kernel noise (Philox4x32-10): frequencies follow softmax(z / T)."""

import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu


def rows(seed, B, V, dtype):
    g = torch.Generator().manual_seed(seed)
    logits = (3 * torch.randn(B, V, generator=g)).to(dtype)
    temps = 0.3 + 1.5 * torch.rand(B, generator=g)
    noise = torch.empty(B, V).exponential_(1, generator=g)
    return logits, temps, noise


def assert_same_or_near_tie(got, ref, logits, temps, noise):
    a = logits.double() / temps.double()[:, None]
    score = torch.softmax(a, dim=-1) / noise.double().clamp_min(1e-10)
    bad = torch.nonzero(got != ref).flatten().tolist()
    for b in bad:
        s1, s2 = float(score[b, got[b]]), float(score[b, ref[b]])
        assert abs(s1 - s2) <= 1e-5 * max(s1, s2), (b, int(got[b]), int(ref[b]), s1, s2)
    assert len(bad) <= max(1, got.numel() // 100)


@pytest.mark.parametrize("dtype", [torch.float32, torch.bfloat16, torch.float16])
@pytest.mark.parametrize("V", [1000, 1003, 151936])
def test_sample_with_given_noise_matches_oracle(pa, dtype, V):
    logits, temps, noise = rows(10 + V, 37, V, dtype)
    got = pa.sample(logits.cuda(), temps.cuda(), noise.cuda()).cpu()
    ref = oracle.sample(logits, temps, noise)
    assert_same_or_near_tie(got, ref, logits.float(), temps, noise)


def test_sample_strided_rows_and_masked_logits(pa):
    logits, temps, noise = rows(20, 16, 500, torch.bfloat16)
    logits[:, 1::2] = float("-inf")
    wide = torch.zeros(16, 512, dtype=torch.bfloat16)
    wide[:, :500] = logits
    got = pa.sample(wide.cuda()[:, :500], temps.cuda(), noise.cuda()).cpu()
    assert bool((got % 2 == 0).all())
    assert torch.equal(got, oracle.sample(logits, temps, noise))


def test_sample_invalid_temperature_is_flagged(pa):
    logits, temps, noise = rows(21, 8, 300, torch.float32)
    temps[2] = 0.0
    temps[5] = 1e-12
    flag = torch.zeros(1, dtype=torch.int32, device="cuda")
    got = pa.sample(logits.cuda(), temps.cuda(), noise.cuda(), err_flag=flag).cpu()
    assert int(got[2]) == -1 and int(got[5]) == -1 and int(flag.item()) & pa.FLAG_BAD_VALUE
    ok = [0, 1, 3, 4, 6, 7]
    assert torch.equal(got[ok], oracle.sample(logits, temps, noise)[ok])


def test_in_kernel_noise_is_deterministic_and_fresh_per_offset(pa):
    logits, temps, _ = rows(22, 64, 4096, torch.bfloat16)
    lg, tp = logits.cuda(), temps.cuda()
    a = pa.sample(lg, tp, seed=1234, offset=7).cpu()
    b = pa.sample(lg, tp, seed=1234, offset=7).cpu()
    c = pa.sample(lg, tp, seed=1234, offset=8).cpu()
    d = pa.sample(lg, tp, seed=99, offset=7).cpu()
    assert torch.equal(a, b)
    assert (a != c).sum() > 16 and (a != d).sum() > 16


@pytest.mark.parametrize("T", [0.5, 1.0, 2.0])
def test_in_kernel_noise_frequencies_follow_softmax(pa, T):
    V, N = 6, 60000
    z = torch.tensor([0.0, 1.0, 2.0, 4.0, -1.0, 3.0])
    got = pa.sample(z.repeat(N, 1).cuda(), torch.full((N,), T).cuda(), seed=2026, offset=int(T * 10)).cpu()
    counts = torch.bincount(got.long(), minlength=V).double()
    expect = torch.softmax(z.double() / T, dim=0) * N
    chi2 = float(((counts - expect) ** 2 / expect).sum())
    assert chi2 < 33.4, (chi2, counts.tolist(), expect.tolist())


def test_sample_from_pinned_host_operands(pa):
    """Logits, temperatures and noise in pinned host memory and the tokens written there by the
    kernel directly: the same tokens as with device operands (given noise and in-kernel noise)."""
    logits, temps, noise = rows(77, 16, 151936, torch.bfloat16)
    dev = torch.device("cuda", 0)
    pl, pt, pn = logits.pin_memory(), temps.pin_memory(), noise.pin_memory()
    for use_noise in (True, False):
        ref = pa.sample(logits.cuda(), temps.cuda(), noise.cuda() if use_noise else None, seed=5, offset=3).cpu()
        out = torch.full((16,), -7, dtype=torch.int32).pin_memory()
        pa.sample(pl, pt, pn if use_noise else None, seed=5, offset=3, out=out, device=dev)
        torch.cuda.synchronize()
        assert torch.equal(out, ref)
    with pytest.raises(ValueError):
        pa.sample(logits, temps, device=dev)
