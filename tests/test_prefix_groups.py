"""Pins of the shared-prefix grouping oracle (``oracle/prefix_groups.py``): the
pages' two-prompt example, batches built with a known sharing structure
(recovered exactly), the cap at the page of each sequence's newest token,
and the rule's invariants on random tables with accidental collisions."""

import json
import os
import random

import pytest

from oracle.prefix_groups import prefix_groups

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "prefix_groups_example.json")


def test_pages_example_groups_a_and_b_on_page_0():
    g = json.load(open(GOLDEN))
    tables = g["block_tables"]["printed"]
    ctx = [g["context_lens"]["A"]["printed"], g["context_lens"]["B"]["derived"]]
    off, seqs, pre = prefix_groups(tables, ctx, g["block_size"])
    e = g["expect"]
    assert (off, seqs, pre) == (e["group_offsets"], e["group_seqs"], e["prefix_lens"])


def test_pages_example_a_alone_is_no_group():
    off, seqs, pre = prefix_groups([[0, 1, 2]], [12], 4)
    assert (off, seqs, pre) == ([0], [], [0])


def _built_batch(rng, bs):
    """A batch with known groups: group g has s_g >= 2 members sharing n_g fresh pages,
    every member then has private pages; plus singletons and padding rows, shuffled."""
    next_id = [0]

    def fresh(n):
        ids = list(range(next_id[0], next_id[0] + n))
        next_id[0] += n
        return ids

    rows, truth = [], []
    for g in range(rng.randint(1, 5)):
        n = rng.randint(1, 6)
        shared = fresh(n)
        for _ in range(rng.randint(2, 9)):
            L = rng.randint(n * bs + 1, (n + 4) * bs)      # (L - 1) // bs >= n: the newest token is private
            pages = shared + fresh(-(-L // bs) - n)
            rows.append((pages, L, g, n))
    for _ in range(rng.randint(0, 4)):                      # singletons
        L = rng.randint(1, 5 * bs)
        rows.append((fresh(-(-L // bs)), L, None, 0))
    for _ in range(rng.randint(0, 2)):                      # padding rows
        rows.append(([], 0, None, 0))
    rng.shuffle(rows)
    width = max(len(p) for p, *_ in rows) or 1
    tables = [p + [-1] * (width - len(p)) for p, *_ in rows]
    return tables, [L for _, L, _, _ in rows], [(g, n) for *_, g, n in rows]


@pytest.mark.parametrize("seed", range(20))
@pytest.mark.parametrize("bs", [4, 16, 256])
def test_known_sharing_is_recovered_exactly(seed, bs):
    rng = random.Random(seed * 1000 + bs)
    tables, ctx, truth = _built_batch(rng, bs)
    off, seqs, pre = prefix_groups(tables, ctx, bs)
    expect_groups = {}
    for b, (g, n) in enumerate(truth):
        if g is not None:
            expect_groups.setdefault(g, []).append(b)
    got_groups = [seqs[off[i]:off[i + 1]] for i in range(len(off) - 1)]
    assert sorted(got_groups) == sorted(expect_groups.values())
    # groups listed in the order their first member appears in the batch
    assert [m[0] for m in got_groups] == sorted(m[0] for m in got_groups)
    assert pre == [n * bs if g is not None else 0 for g, n in truth]


def test_cap_at_the_page_of_the_newest_token():
    # three sequences share 3 pages, but one has context 9 with block size 4: its newest token
    # (position 8) sits in the third page, so only (9 - 1) // 4 = 2 pages are shared
    tables = [[7, 8, 9, 10], [7, 8, 9, 11], [7, 8, 9, -1]]
    assert prefix_groups(tables, [16, 15, 9], 4) == ([0, 3], [0, 1, 2], [8, 8, 8])
    # context 8: position 7 ends page 1, so pages 0 and 1 (8 tokens)... minus the newest
    # token's page: (8 - 1) // 4 = 1 page
    assert prefix_groups(tables, [16, 15, 8], 4) == ([0, 3], [0, 1, 2], [4, 4, 4])
    # context 4: the newest token sits in page 0 itself: that sequence shares nothing and is left
    # out, the other two share their 3 common pages
    assert prefix_groups(tables, [16, 15, 4], 4) == ([0, 2], [0, 1], [12, 12, 0])
    assert prefix_groups(tables, [16, 4, 4], 4) == ([0], [], [0, 0, 0])


def test_min_shared_pages_dissolves_short_groups():
    tables = [[3, 4, 5], [3, 6, 7], [8, 9, 10], [8, 9, 11]]
    ctx = [12, 12, 12, 12]
    assert prefix_groups(tables, ctx, 4, min_shared_pages=2) == ([0, 2], [2, 3], [0, 0, 8, 8])
    assert prefix_groups(tables, ctx, 4) == ([0, 2, 4], [0, 1, 2, 3], [4, 4, 8, 8])


@pytest.mark.parametrize("seed", range(30))
def test_invariants_on_random_tables_with_collisions(seed):
    rng = random.Random(seed)
    bs = rng.choice([1, 2, 4, 16])
    B = rng.randint(1, 24)
    ctx = [rng.choice([0, rng.randint(1, 12 * bs)]) for _ in range(B)]
    width = max(1, max(-(-L // bs) for L in ctx))
    # a small page alphabet makes accidental equal entries common
    tables = [[rng.randint(0, 3) for _ in range(-(-L // bs))] + [-1] * (width - (-(-L // bs))) for L in ctx]
    off, seqs, pre = prefix_groups(tables, ctx, bs)
    assert len(set(seqs)) == len(seqs) and off[0] == 0 and off[-1] == len(seqs)
    member = set(seqs)
    for b in range(B):
        if b not in member:
            assert pre[b] == 0
    for i in range(len(off) - 1):
        m = seqs[off[i]:off[i + 1]]
        assert len(m) >= 2 and m == sorted(m)
        n = pre[m[0]] // bs
        assert n >= 1 and all(pre[b] == n * bs for b in m)
        assert all(ctx[b] > 0 and (ctx[b] - 1) // bs >= n for b in m)
        assert all(tables[b][:n] == tables[m[0]][:n] for b in m)
        cap = min((ctx[b] - 1) // bs for b in m)
        if n < cap:  # maximal: the next page differs somewhere
            assert len({tables[b][n] for b in m}) > 1
        # every non-padding sequence with the same first page is in this group
        assert {b for b in range(B) if ctx[b] > bs and tables[b][0] == tables[m[0]][0]} == set(m)


def test_shared_prefix_decode_workload_is_32_groups_of_8():
    # the Qwen3-8B-like decode workload: groups of 8 consecutive sequences share a 512-token prefix
    from tests import inputs
    st = inputs.qwen3_8b_shared_decode()
    off, seqs, pre = prefix_groups(st.block_tables.tolist(), st.context_lens.tolist(), st.pool.block_size)
    assert off == list(range(0, 257, 8)) and seqs == list(range(256)) and pre == [512] * 256
