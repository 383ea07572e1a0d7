"""pa_stage_decode_step on the host (no GPU): a decode step's slot mapping, context lengths and
block tables written into a captured bucket's staging with the rows past the batch padded
("nano-vLLM Part 2: Block Tables, KV Cache, and the Path to the GPU", section 4.2), the
shared-prefix groups staged as their mode says, and the gather list or the decode's operands
array pointed at the caller's buffers.  The staging arrays here are ordinary host tensors: the call never touches a GPU."""

import ctypes
import random

import pytest
import torch

ROWS, MAX_BLOCKS, BS = 16, 12, 16
SENTINEL = 777


class Staging:
    """Host arrays of one bucket and the pa_decode_staging naming them."""

    def __init__(self, pa, rows=ROWS, max_blocks=MAX_BLOCKS, caps=None, segments=False):
        self.slot = torch.full((rows,), SENTINEL, dtype=torch.int32)
        self.ctx = torch.full((rows,), SENTINEL, dtype=torch.int32)
        self.tables = torch.full((rows, max_blocks), SENTINEL, dtype=torch.int32)
        self.st = pa.DecodeStaging(rows=rows, max_blocks=max_blocks, block_size=BS,
                                   slot_mapping=self.slot.data_ptr(), context_lens=self.ctx.data_ptr(),
                                   block_tables=self.tables.data_ptr())
        if caps is not None:
            ng = caps[0]
            self.offsets = torch.full((ng + 1,), SENTINEL, dtype=torch.int32)
            self.seqs = torch.full((rows,), SENTINEL, dtype=torch.int32)
            self.prefix = torch.full((rows,), SENTINEL, dtype=torch.int32)
            self.st.max_groups, self.st.max_group_size, self.st.max_prefix_len = caps
            self.st.group_offsets = self.offsets.data_ptr()
            self.st.group_seqs = self.seqs.data_ptr()
            self.st.prefix_lens = self.prefix.data_ptr()
        if segments:
            self.segs = (pa.CopySegment * 3)()
            for i in range(3):
                self.segs[i].dst = 0x1000 * (i + 1)
                self.st.segment_row_bytes[i] = 256 * (i + 1)
            self.st.segments = ctypes.addressof(self.segs)
            self.st.num_segments = 3


def step(batch, max_blocks=MAX_BLOCKS, seed=0, shared=0):
    """A step's metadata: batch sequences, the first ``shared`` of each pair of rows sharing pages."""
    rnd = random.Random(seed)
    ctx = torch.tensor([rnd.randint(0, max_blocks * BS) for _ in range(batch)], dtype=torch.int32)
    tables = torch.tensor([[rnd.randrange(1000) for _ in range(max_blocks)] for _ in range(batch)],
                          dtype=torch.int32).reshape(batch, max_blocks)
    for b in range(1, batch, 2):
        tables[b, :shared] = tables[b - 1, :shared]
    slot = torch.tensor([rnd.randrange(-1, 5000) for _ in range(batch)], dtype=torch.int32)
    return slot, ctx, tables


@pytest.mark.parametrize("batch", [0, 1, 7, ROWS])
def test_metadata_copied_and_padded(pa_host, batch):
    s = Staging(pa_host)
    slot, ctx, tables = step(batch, seed=batch)
    pa_host.stage_decode_step(s.st, slot, ctx, tables)
    assert torch.equal(s.slot[:batch], slot) and torch.equal(s.ctx[:batch], ctx)
    assert torch.equal(s.tables[:batch], tables)
    assert (s.slot[batch:] == -1).all() and (s.ctx[batch:] == 0).all()
    assert (s.tables[batch:] == SENTINEL).all()  # a context of 0 reads no page: pad rows untouched


def test_narrow_tables_padded_with_minus_one(pa_host):
    s = Staging(pa_host)
    slot, ctx, tables = step(5, max_blocks=4, seed=3)
    pa_host.stage_decode_step(s.st, slot, ctx, tables)
    assert torch.equal(s.tables[:5, :4], tables)
    assert (s.tables[:5, 4:] == -1).all()


def test_no_groups_empties_the_group_arrays(pa_host):
    s = Staging(pa_host, caps=(4, 8, 160))
    pa_host.stage_decode_step(s.st, *step(6, seed=4))
    assert (s.offsets == 0).all() and (s.prefix == 0).all()
    assert (s.seqs == SENTINEL).all()  # no member is read past the last offset


def test_keep_groups_leaves_them(pa_host):
    s = Staging(pa_host, caps=(4, 8, 160))
    pa_host.stage_decode_step(s.st, *step(6, seed=5), groups=pa_host.STAGE_KEEP_GROUPS)
    assert (s.offsets == SENTINEL).all() and (s.prefix == SENTINEL).all()


@pytest.mark.parametrize("batch", [0, 2, 9, ROWS])
def test_derived_groups_match_prefix_groups(pa_host, batch):
    from paged_kv_cache_bs_gb300.block_manager import prefix_groups
    s = Staging(pa_host, caps=(ROWS // 2, ROWS, MAX_BLOCKS * BS))
    slot, ctx, tables = step(batch, seed=10 + batch, shared=5)
    pa_host.stage_decode_step(s.st, slot, ctx, tables, groups=pa_host.STAGE_DERIVE_GROUPS)
    g = prefix_groups(tables, ctx, BS)
    n = g.num_groups
    assert torch.equal(s.offsets[:n + 1], g.group_offsets[:n + 1])
    last = int(g.group_offsets[n])
    assert (s.offsets[n + 1:] == last).all()  # unused groups are empty
    assert torch.equal(s.seqs[:last], g.group_seqs[:last])
    assert torch.equal(s.prefix[:batch], g.prefix_lens[:batch])
    assert (s.prefix[batch:] == 0).all()
    if batch >= 9:
        assert n >= 1  # the shared pairs form groups


def test_derived_groups_beyond_capacity_rejected(pa_host):
    s = Staging(pa_host, caps=(1, 2, MAX_BLOCKS * BS))
    slot, ctx, tables = step(ROWS, seed=20, shared=6)
    ctx.fill_(MAX_BLOCKS * BS)  # every pair shares 6 complete pages: 8 groups
    with pytest.raises(pa_host.PagedAttentionError, match="capacities"):
        pa_host.stage_decode_step(s.st, slot, ctx, tables, groups=pa_host.STAGE_DERIVE_GROUPS)
    s = Staging(pa_host, caps=(ROWS, ROWS, 4 * BS))
    with pytest.raises(pa_host.PagedAttentionError, match="capacities"):
        pa_host.stage_decode_step(s.st, slot, ctx, tables, groups=pa_host.STAGE_DERIVE_GROUPS)


def test_gather_list_pointed_at_sources(pa_host):
    s = Staging(pa_host, segments=True)
    pa_host.stage_decode_step(s.st, *step(5, seed=6), sources=[0xA000, 0xB000, 0xC000])
    for i, src in enumerate((0xA000, 0xB000, 0xC000)):
        assert s.segs[i].src == src
        assert s.segs[i].bytes == 5 * 256 * (i + 1)
        assert s.segs[i].dst == 0x1000 * (i + 1)
    pa_host.stage_decode_step(s.st, *step(3, seed=7))  # no sources: the list is left as it is
    assert s.segs[0].bytes == 5 * 256


def test_operands_array_pointed_at_sources(pa_host):
    s = Staging(pa_host)
    ops = torch.zeros(3, dtype=torch.int64)
    s.st.operands = ops.data_ptr()
    pa_host.stage_decode_step(s.st, *step(4, seed=9), sources=[0xA000, 0xB010, 0xC020])
    assert ops.tolist() == [0xA000, 0xB010, 0xC020]
    pa_host.stage_decode_step(s.st, *step(4, seed=9))  # no sources: left as it is
    assert ops.tolist() == [0xA000, 0xB010, 0xC020]
    # with both a gather list and an operands array, both are written
    s = Staging(pa_host, segments=True)
    s.st.operands = ops.data_ptr()
    pa_host.stage_decode_step(s.st, *step(2, seed=10), sources=[0x1, 0x2, 0x3])
    assert ops.tolist() == [1, 2, 3] and s.segs[2].src == 3


def test_invalid_arguments_rejected_before_any_write(pa_host):
    s = Staging(pa_host, caps=(4, 8, 160))
    slot, ctx, tables = step(4, seed=8)
    err = pa_host.PagedAttentionError
    lib = pa_host.library()
    addr = ctypes.addressof(s.st)

    def call(batch=4, cols=MAX_BLOCKS, mode=0, sources=None, staging=addr, c=ctx):
        return lib.pa_stage_decode_step(staging, batch, slot.data_ptr(), c.data_ptr(), tables.data_ptr(), cols,
                                        mode, sources)
    assert call(batch=ROWS + 1) == -1
    assert call(batch=-1) == -1
    assert call(cols=0) == -1 and call(cols=MAX_BLOCKS + 1) == -1
    assert call(mode=3) == -1
    assert call(sources=ctypes.addressof((ctypes.c_void_p * 3)())) == -1  # no gather list or operands array
    assert call(staging=None) == -1
    bad = ctx.clone()
    bad[2] = MAX_BLOCKS * BS + 1
    assert call(c=bad) == -1
    bad[2] = -1
    assert call(c=bad) == -1
    assert (s.slot == SENTINEL).all() and (s.ctx == SENTINEL).all()  # nothing written
    plain = Staging(pa_host)
    with pytest.raises(err, match="no shared-prefix groups"):
        pa_host.stage_decode_step(plain.st, slot, ctx, tables, groups=pa_host.STAGE_DERIVE_GROUPS)
    narrow = tables[:, :3].contiguous()
    with pytest.raises(err, match="outside its 48-token table"):
        pa_host.stage_decode_step(plain.st, slot, ctx.clamp(max=MAX_BLOCKS * BS).fill_(100), narrow)
