"""Pins the runner-side index preparation of the input generator against the
worked examples the pages print (tests/golden/slot_examples.json)."""

import json
import os

import torch

from tests import inputs

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "slot_examples.json")


def _golden():
    with open(GOLDEN) as f:
        return json.load(f)


def test_position_to_slot_examples():
    for ex in _golden()["position"]:
        assert inputs.slot_of(ex["block_table"], ex["block_size"], ex["position"]) == ex["slot"], ex["cite"]


def test_prefill_slot_loop_examples():
    for ex in _golden()["range"]:
        got = inputs.slots_for_range(ex["block_table"], ex["block_size"], ex["start"], ex["end"])
        assert got == ex["slot_mapping"], ex["cite"]
        # the loop agrees with the per-position formula on every token
        per = [inputs.slot_of(ex["block_table"], ex["block_size"], p) for p in range(ex["start"], ex["end"])]
        assert got == per


def test_cu_seqlens_examples():
    for ex in _golden()["cu_seqlens"]:
        q = inputs.cu_seqlens(ex["scheduled"]).tolist()
        k = inputs.cu_seqlens([c + s for c, s in zip(ex["cached"], ex["scheduled"])]).tolist()
        assert q == ex["cu_seqlens_q"], ex["cite"]
        assert k == ex["cu_seqlens_k"], ex["cite"]


def test_decode_slot_examples():
    for ex in _golden()["decode"]:
        assert inputs.decode_slot(ex["block_table"], ex["block_size"], ex["seq_len"]) == ex["slot"], ex["cite"]
        # decode's context length is the sequence length (it includes the stored token)
        assert ex["context_len"] == ex["seq_len"]


def test_block_table_padding_examples():
    for ex in _golden()["tables"]:
        got = inputs.pad_block_tables(ex["tables"])
        assert got.dtype == torch.int32
        assert got.tolist() == ex["padded"], ex["cite"]


def test_prefill_slots_cross_pages_with_partial_ends():
    # a range starting and ending mid-page over a fragmented table
    bt, bs = [9, 2, 5, 7], 4
    got = inputs.slots_for_range(bt, bs, 3, 14)
    assert got == [inputs.slot_of(bt, bs, p) for p in range(3, 14)]
    assert inputs.slots_for_range(bt, bs, 5, 5) == []


def test_generated_pools_are_consistent():
    st = inputs.tiny_decode()
    p = st.pool
    # every table entry is a distinct physical block inside the pool
    ids = [b for t in p.tables for b in t]
    assert len(ids) == len(set(ids)) == 26
    assert all(0 <= b < p.num_blocks for b in ids)
    # the store slot of each sequence is its last logical position
    for t, L, s in zip(p.tables, st.context_lens.tolist(), st.slot_mapping.tolist()):
        assert s == inputs.slot_of(t, p.block_size, L - 1)
    # before the store, the slot holds the sentinel and earlier positions do not
    kf = p.k_cache.view(torch.int16).reshape(-1, p.num_kv_heads * p.head_dim)
    for t, L, s in zip(p.tables, st.context_lens.tolist(), st.slot_mapping.tolist()):
        assert (kf[s] == inputs.SENTINEL_BITS).all()
        for j in range(L - 1):
            assert not (kf[inputs.slot_of(t, p.block_size, j)] == inputs.SENTINEL_BITS).all()


def test_shared_prefix_tables():
    st = inputs.make_decode([40, 37, 50, 33], num_q_heads=4, num_kv_heads=2, head_dim=16, block_size=8,
                            dtype=torch.bfloat16, seed=7, share_groups=2, share_tokens=32)
    t = st.pool.tables
    assert t[0][:4] == t[1][:4] and t[2][:4] == t[3][:4]
    assert t[0][:4] != t[2][:4]
    assert not set(t[0][4:]) & set(t[1][4:])
    assert st.unique_kv_bytes() < st.kv_bytes()
