"""Engine-style steps on the GPU driven by the native page directory: the
block tables and slot mappings come from BlockManager (prefix sharing, page
growth at block boundaries), the K/V rows of a token are a fixed function of
(token, position) as for a real model, and every step's attention output is
checked against the oracle run on a plain contiguous copy of each sequence's
logical context."""

import pytest
import torch

import oracle
from tests.gpu_cases import TOL, max_err

pytestmark = pytest.mark.gpu

BS, HQ, HKV, D, NBLK, MAXB, VOCAB, MAXPOS = 16, 8, 2, 128, 64, 8, 64, 160
DT = torch.bfloat16
SCALE = D ** -0.5


def dense_pool(seqs):
    """Each sequence's logical context laid out in its own consecutive blocks."""
    nb = sum((len(t) + BS - 1) // BS for t in seqs)
    kc = torch.zeros(max(nb, 1), BS, HKV, D, dtype=DT)
    vc = torch.zeros_like(kc)
    tables, b0 = [], 0
    for toks in seqs:
        n = (len(toks) + BS - 1) // BS
        tables.append(list(range(b0, b0 + n)) + [-1] * (MAXB - n))
        for p, t in enumerate(toks):
            kc[b0 + p // BS, p % BS] = KT[t, p]
            vc[b0 + p // BS, p % BS] = VT[t, p]
        b0 += n
    return kc, vc, torch.tensor(tables, dtype=torch.int32)


g = torch.Generator().manual_seed(2024)
KT = torch.randn(VOCAB, MAXPOS, HKV, D, generator=g).to(DT)
VT = torch.randn(VOCAB, MAXPOS, HKV, D, generator=g).to(DT)


def test_prefix_shared_prefill_and_decode_steps(pa):
    from paged_kv_cache_bs_gb300.block_manager import BlockManager
    rng = torch.Generator().manual_seed(7)
    bm = BlockManager(NBLK, BS)
    kc = torch.full((NBLK, BS, HKV, D), float("nan"), dtype=DT, device="cuda")
    vc = torch.full_like(kc, float("nan"))
    toks = {}
    A = torch.randint(0, VOCAB, (40,), generator=rng).tolist()
    toks[0] = A
    toks[1] = A[:32] + torch.randint(0, VOCAB, (20,), generator=rng).tolist()   # shares 2 full blocks
    toks[2] = torch.randint(0, VOCAB, (25,), generator=rng).tolist()
    for s, t in toks.items():
        bm.add_sequence(s, t)

    def prefill(sids):
        sched = [len(toks[s]) - bm.num_cached_tokens(s) for s in sids]
        slots, cq, ck, tables = bm.prefill_inputs(sids, sched, MAXB)
        pos = [p for s, n in zip(sids, sched) for p in range(len(toks[s]) - n, len(toks[s]))]
        tk = [toks[s][p] for s, n in zip(sids, sched) for p in range(len(toks[s]) - n, len(toks[s]))]
        k_new = KT[tk, pos]
        v_new = VT[tk, pos]
        q = torch.randn(len(tk), HQ, D, generator=rng).to(DT)
        pa.store_kv(k_new.cuda(), v_new.cuda(), kc, vc, slots.cuda())
        out = pa.prefill_paged(q.cuda(), k_new.cuda(), v_new.cuda(), kc, vc, cq.cuda(), ck.cuda(), max(sched),
                               int((ck[1:] - ck[:-1]).max()), tables.cuda(), SCALE)
        torch.cuda.synchronize()
        dk, dv, dtab = dense_pool([toks[s] for s in sids])
        ref = oracle.prefill_paged(q, k_new, v_new, dk, dv, cq, ck, dtab, SCALE)
        assert max_err(out, ref) <= TOL[DT]
        for s, n in zip(sids, sched):
            bm.postprocess(s, n)

    for s in (0, 2):
        assert bm.can_allocate(s) == 0
        bm.allocate(s, 0)
    prefill([0, 2])
    # sequence 1 finds sequence 0's two full blocks registered and shares them
    assert bm.can_allocate(1) == 2
    bm.allocate(1, 2)
    assert bm.block_table(1)[:2] == bm.block_table(0)[:2] and bm.ref_count(bm.block_table(0)[0]) == 2
    assert bm.num_cached_tokens(1) == 32
    prefill([1])                                    # 20 new rows over a 32-token shared prefix

    ws = None
    for step in range(24):                          # decode steps; pages grow at block boundaries
        sids = [0, 1, 2]
        for s in sids:
            t = int(torch.randint(0, VOCAB, (1,), generator=rng))
            toks[s].append(t)
            bm.append_token(s, t)
            assert bm.can_append(s)
            bm.may_append(s)
        slots, lens, tables = bm.decode_inputs(sids, MAXB)
        k_new = torch.stack([KT[toks[s][-1], len(toks[s]) - 1] for s in sids])
        v_new = torch.stack([VT[toks[s][-1], len(toks[s]) - 1] for s in sids])
        q = torch.randn(len(sids), HQ, D, generator=rng).to(DT)
        if ws is None:
            ws = pa.alloc_decode_workspace(q.cuda(), kc, tables.cuda())
        out = pa.store_decode(k_new.cuda(), v_new.cuda(), slots.cuda(), q.cuda(), kc, vc, tables.cuda(), lens.cuda(),
                              SCALE, workspace=ws)
        torch.cuda.synchronize()
        dk, dv, dtab = dense_pool([toks[s] for s in sids])
        ref = oracle.decode(q, dk, dv, dtab, lens, SCALE)
        assert max_err(out, ref) <= TOL[DT], f"decode step {step}"
        for s in sids:
            bm.postprocess(s, 1)
    assert [len(bm.block_table(s)) for s in (0, 1, 2)] == [(len(toks[s]) + BS - 1) // BS for s in (0, 1, 2)]
    # releasing the sharer keeps the shared blocks alive for the other sequence
    shared = bm.block_table(0)[:2]
    bm.deallocate(0)
    assert [bm.ref_count(b) for b in shared] == [1, 1]
