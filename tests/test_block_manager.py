"""The native page directory (C++, through the C ABI) and its plain-Python
oracle, on the pages' BlockManager walk-through and on random request
streams.  The oracle is pinned by the walk-through; the native manager must
match the printed values and the oracle step by step."""

import json
import os
import random

import pytest
import torch

from oracle.block_manager import OracleBlockManager

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "block_manager_trace.json")


@pytest.fixture(scope="module")
def native(pa_host):
    from paged_kv_cache_bs_gb300.block_manager import BlockManager
    return BlockManager


def _run_trace(bm):
    g = json.load(open(GOLDEN))
    ids = {}
    for st in g["steps"]:
        want = st.get("printed", st.get("derived"))
        op = st["op"]
        sid = ids.setdefault(st["seq"], len(ids)) if "seq" in st else None
        if op == "add":
            bm.add_sequence(sid, st["tokens"])
        elif op == "append":
            bm.append_token(sid, st["token"])
        elif op == "can_allocate":
            assert bm.can_allocate(sid) == want, st
        elif op == "allocate":
            bm.allocate(sid, st["hits"])
        elif op == "can_append":
            assert bool(bm.can_append(sid)) == want, st
        elif op == "may_append":
            bm.may_append(sid)
        elif op == "postprocess":
            bm.postprocess(sid, st["scheduled"])
        elif op == "deallocate":
            bm.deallocate(sid)
        elif op == "prefill_inputs":
            slots, cq, ck, tables = bm.prefill_inputs([ids[s] for s in st["seqs"]], st["scheduled"], st["max_blocks"])
            got = {"slot_mapping": list(slots), "cu_seqlens_q": list(cq), "cu_seqlens_k": list(ck),
                   "block_tables": [list(r) for r in tables]}
            for k, v in want.items():
                assert [int(x) for x in got[k]] == v if k != "block_tables" else \
                    [[int(x) for x in r] for r in got[k]] == v, (st, k)
        elif op == "decode_inputs":
            slots, lens, tables = bm.decode_inputs([ids[s] for s in st["seqs"]], st["max_blocks"])
            got = {"slot_mapping": [int(x) for x in slots], "context_lens": [int(x) for x in lens],
                   "block_tables": [[int(x) for x in r] for r in tables]}
            for k, v in want.items():
                assert got[k] == v, (st, k)
        if isinstance(want, dict):  # state checks after the step
            for k, v in want.items():
                if k == "block_table":
                    assert list(bm.block_table(sid)) == v, st
                elif k == "ref_counts":
                    for b, c in v.items():
                        assert bm.ref_count(int(b)) == c, (st, b)
                elif k == "num_free":
                    assert bm.num_free_blocks() == v, st
                elif k == "num_cached_tokens":
                    assert bm.num_cached_tokens(sid) == v, st
        if "derived" in st and isinstance(st["derived"], dict) and "printed" in st:
            for k, v in st["derived"].items():
                if k == "num_free":
                    assert bm.num_free_blocks() == v, st


def test_oracle_follows_the_pages_walkthrough():
    g = json.load(open(GOLDEN))
    _run_trace(OracleBlockManager(g["num_blocks"], g["block_size"]))


def test_native_follows_the_pages_walkthrough(native):
    g = json.load(open(GOLDEN))
    _run_trace(native(g["num_blocks"], g["block_size"]))


def test_last_block_is_never_a_hit_and_same_step_prefixes_do_not_share(native):
    # "the final partial page is never considered a prefix-cache hit"; a request equal to a
    # cached two-block prefix reuses only its first block, a longer one reuses both; blocks
    # are registered only after the step that computed them (nano-vLLM section 12.4, 12.6)
    for bm in (OracleBlockManager(16, 4), native(16, 4)):
        first = [1, 2, 3, 4, 5, 6, 7, 8]
        bm.add_sequence(0, first)
        bm.add_sequence(1, first)
        assert bm.can_allocate(0) == 0
        bm.allocate(0, 0)
        assert bm.can_allocate(1) == 0          # sequence 0 not postprocessed yet: nothing registered
        bm.postprocess(0, 8)
        assert bm.can_allocate(1) == 1          # same two blocks: only the first can hit
        bm.add_sequence(2, first + [9])
        assert bm.can_allocate(2) == 2          # a longer request reuses both


@pytest.mark.parametrize("seed", range(12))
def test_native_matches_the_oracle_on_random_request_streams(native, seed):
    rng = random.Random(seed)
    bs = rng.choice([2, 4, 16])
    nblocks = rng.choice([12, 40])
    o, n = OracleBlockManager(nblocks, bs), native(nblocks, bs)
    prefixes = [[rng.randrange(50) for _ in range(rng.randrange(1, 3 * bs))] for _ in range(4)]
    live, waiting, next_id = [], [], 0
    for step in range(120):
        r = rng.random()
        if r < 0.25:  # a new request, often with a shared prefix
            toks = (rng.choice(prefixes) if rng.random() < 0.7 else []) + [rng.randrange(50) for _ in range(rng.randrange(1, 2 * bs))]
            for m in (o, n):
                m.add_sequence(next_id, toks)
            waiting.append(next_id)
            next_id += 1
        elif r < 0.45 and waiting:  # admit one: can_allocate + allocate + prefill postprocess
            sid = waiting[0]
            hits = o.can_allocate(sid)
            assert n.can_allocate(sid) == hits
            if hits < 0:
                continue
            waiting.pop(0)
            for m in (o, n):
                m.allocate(sid, hits)
            sched = len(o.seqs[sid].tokens) - o.num_cached_tokens(sid)
            mb = len(o.block_table(sid))
            a = o.prefill_inputs([sid], [sched], mb)
            b = n.prefill_inputs([sid], [sched], mb)
            assert [list(map(int, x)) if not hasattr(x, "tolist") else x.tolist() for x in b[:3]] == [list(v) for v in a[:3]]
            assert b[3].tolist() == a[3]
            for m in (o, n):
                m.postprocess(sid, sched)
            live.append(sid)
        elif r < 0.85 and live:  # a decode step of a random subset
            batch = [s for s in live if rng.random() < 0.6]
            ok = []
            for sid in batch:
                tok = rng.randrange(50)
                for m in (o, n):
                    m.append_token(sid, tok)
                assert n.can_append(sid) == o.can_append(sid)
                if not o.can_append(sid):  # preempt: release and requeue
                    for m in (o, n):
                        m.deallocate(sid)
                    live.remove(sid)
                    waiting.append(sid)
                    continue
                for m in (o, n):
                    m.may_append(sid)
                ok.append(sid)
            if ok:
                mb = max(len(o.block_table(s)) for s in ok)
                a = o.decode_inputs(ok, mb)
                b = n.decode_inputs(ok, mb)
                assert b[0].tolist() == a[0] and b[1].tolist() == a[1] and b[2].tolist() == a[2]
                for sid in ok:
                    for m in (o, n):
                        m.postprocess(sid, 1)
        elif live:  # a request finishes
            sid = live.pop(rng.randrange(len(live)))
            for m in (o, n):
                m.remove_sequence(sid)
        for sid in live:
            assert n.block_table(sid) == o.block_table(sid)
            assert n.num_cached_tokens(sid) == o.num_cached_tokens(sid)
        assert n.num_free_blocks() == o.num_free_blocks()
        assert [n.ref_count(b) for b in range(nblocks)] == [o.ref_count(b) for b in range(nblocks)]


def test_native_rejects_misuse(native):
    from paged_kv_cache_bs_gb300 import PagedAttentionError
    bm = native(4, 4)
    bm.add_sequence(0, [1, 2, 3])
    with pytest.raises(PagedAttentionError):
        bm.add_sequence(0, [1])
    with pytest.raises(PagedAttentionError):
        bm.allocate(0, 1)                       # no block of a 1-block sequence can be a hit
    with pytest.raises(PagedAttentionError):
        bm.may_append(0)                        # holds no blocks yet
    with pytest.raises(PagedAttentionError):
        bm.decode_inputs([7], 4)                # unknown sequence
    with pytest.raises(PagedAttentionError):
        bm.can_allocate(7)                      # an error, not "not enough blocks"
    bm.allocate(0, 0)
    with pytest.raises(PagedAttentionError):
        bm.postprocess(0, 9)                    # more tokens than the sequence has


# ------------------------------------------------------------- prefix groups

def _pg_native(tables, ctx, bs, min_pages=1):
    from paged_kv_cache_bs_gb300.block_manager import prefix_groups as native
    width = max([len(t) for t in tables] + [1])
    bt = torch.tensor([list(t) + [-1] * (width - len(t)) for t in tables] or [[-1]], dtype=torch.int32)[:len(tables)]
    g = native(bt.reshape(len(tables), width), torch.tensor(ctx, dtype=torch.int32), bs, min_pages)
    return g.group_offsets.tolist(), g.group_seqs[:g.group_offsets[-1]].tolist(), g.prefix_lens.tolist(), g


@pytest.mark.parametrize("seed", range(40))
def test_native_prefix_groups_equal_the_oracle(seed):
    import random
    from oracle.prefix_groups import prefix_groups as ref
    from tests.test_prefix_groups import _built_batch
    rng = random.Random(seed)
    bs = rng.choice([1, 3, 4, 12, 16, 256])  # any positive block size, powers of two or not
    if seed % 2:
        tables, ctx, _ = _built_batch(rng, bs)
    else:   # random tables over a small page alphabet: accidental equal entries are common
        B = rng.randint(0, 30)
        ctx = [rng.choice([0, rng.randint(1, 9 * bs)]) for _ in range(B)]
        tables = [[rng.randint(0, 4) for _ in range(-(-L // bs))] for L in ctx]
    width = max([-(-L // bs) for L in ctx] + [1])
    tables = [list(t) + [-1] * (width - len(t)) for t in tables]
    min_pages = rng.choice([1, 1, 2, 3])
    off, seqs, pre, g = _pg_native(tables, ctx, bs, min_pages)
    assert (off, seqs, pre) == ref(tables, ctx, bs, min_pages)
    sizes = [off[i + 1] - off[i] for i in range(len(off) - 1)]
    assert g.max_group_size == max(sizes, default=0) and g.max_prefix_len == max(pre, default=0)


@pytest.mark.parametrize("batch", [600, 5, 2000, 64])
def test_native_prefix_groups_many_candidates(batch):
    # first pages that differ only in high bits, or only in low bits, many of them, and batches
    # of changing size one after the other (the native lookup table is reused between calls)
    import random
    from oracle.prefix_groups import prefix_groups as ref
    rng = random.Random(batch)
    bs = 4
    starts = [k << 20 for k in range(40)] + [k for k in range(40)] + [rng.randrange(2**31) for _ in range(40)]
    tables, ctx = [], []
    for b in range(batch):
        p0 = rng.choice(starts)
        L = rng.randint(1, 6 * bs)
        tables.append([p0] + [rng.choice([p0 + 1, p0 + 2]) for _ in range(5)])
        ctx.append(L)
    off, seqs, pre, _ = _pg_native(tables, ctx, bs)
    assert (off, seqs, pre) == ref(tables, ctx, bs)
    assert len(off) > 2 or batch < 64  # several groups in the larger batches


def test_native_prefix_groups_pages_example():
    import json
    gold = json.load(open(os.path.join(os.path.dirname(__file__), "golden", "prefix_groups_example.json")))
    ctx = [gold["context_lens"]["A"]["printed"], gold["context_lens"]["B"]["derived"]]
    off, seqs, pre, _ = _pg_native(gold["block_tables"]["printed"], ctx, gold["block_size"])
    e = gold["expect"]
    assert (off, seqs, pre) == (e["group_offsets"], e["group_seqs"], e["prefix_lens"])


def test_native_prefix_groups_rejects_bad_lengths():
    import paged_kv_cache_bs_gb300 as pa
    from paged_kv_cache_bs_gb300.block_manager import prefix_groups as native
    with pytest.raises(pa.PagedAttentionError):
        native(torch.zeros(2, 3, dtype=torch.int32), torch.tensor([5, 13], dtype=torch.int32), 4)  # 13 > 3 * 4
