"""Plain-Python page directory -- TEST INFRASTRUCTURE ONLY (the oracle of
the native BlockManager in ``paged_kv_cache_bs_gb300/csrc/block_manager.cpp``;
the two share no code).

Written from the BlockManager walk-through of "Inference engine: inside
nano-vLLM" / "nano-vLLM Part 2: Block Tables, KV Cache, and the Path to the
GPU" (sections 2 and 3), step by step in the pages' order:

* can_allocate: chained hashes over every logical block but the last; stop at
  the first miss or token mismatch; hits on blocks in use need no free block.
* allocate: share the hits (count + 1, or revive a freed block), then take
  fresh blocks from the front of the free list (dropping a stale hash entry).
* can_append / may_append: a decode step needs a block when the last token
  starts a page (length 1 mod block size).
* postprocess: hash the blocks a step completed, from the previous block's
  hash; advance num_cached_tokens.
* deallocate: reverse walk, blocks reaching 0 go to the back of the free list
  with their hash kept.
* the kernel inputs: decode slot of the last token, -1-padded tables, and the
  prefill slot loop over the scheduled range.

Its hash is BLAKE2b with an 8-byte digest (from hashlib), unlike the native
FNV-1a: the observable behaviour is the same unless a hash collides.
"""

from __future__ import annotations

import hashlib
import struct
from collections import deque


def _h(tokens, prev):
    m = hashlib.blake2b(digest_size=8)
    if prev is not None:
        m.update(struct.pack("<Q", prev))
    m.update(struct.pack(f"<{len(tokens)}i", *tokens))
    return struct.unpack("<Q", m.digest())[0]


class _Block:
    def __init__(self):
        self.ref_count = 0
        self.hash = None
        self.tokens = None


class _Seq:
    def __init__(self, tokens):
        self.tokens = list(tokens)
        self.block_table = []
        self.num_cached_tokens = 0


class OracleBlockManager:
    def __init__(self, num_blocks, block_size):
        self.bs = block_size
        self.blocks = [_Block() for _ in range(num_blocks)]
        self.free = deque(range(num_blocks))
        self.used = set()
        self.hash_to_block = {}
        self.seqs = {}

    # ---- helpers
    def _nblocks(self, s):
        return (len(s.tokens) + self.bs - 1) // self.bs

    def _block(self, s, i):
        return s.tokens[i * self.bs:(i + 1) * self.bs]

    def _hit(self, h, tokens):
        b = self.hash_to_block.get(h)
        if b is None or self.blocks[b].tokens != tokens:
            return None
        return b

    def _fresh(self):
        b = self.free.popleft()
        blk = self.blocks[b]
        if blk.hash is not None and self.hash_to_block.get(blk.hash) == b:
            del self.hash_to_block[blk.hash]
        blk.hash, blk.tokens, blk.ref_count = None, None, 1
        self.used.add(b)
        return b

    # ---- the calls
    def add_sequence(self, sid, tokens):
        self.seqs[sid] = _Seq(tokens)

    def append_token(self, sid, t):
        self.seqs[sid].tokens.append(t)

    def can_allocate(self, sid):
        s = self.seqs[sid]
        h, hits, need = None, 0, self._nblocks(s)
        for i in range(self._nblocks(s) - 1):
            tok = self._block(s, i)
            h = _h(tok, h)
            b = self._hit(h, tok)
            if b is None:
                break
            hits += 1
            if b in self.used:
                need -= 1
        return -1 if len(self.free) < need else hits

    def allocate(self, sid, hits):
        s = self.seqs[sid]
        h = None
        for i in range(hits):
            tok = self._block(s, i)
            h = _h(tok, h)
            b = self.hash_to_block[h]
            if b in self.used:
                self.blocks[b].ref_count += 1
            else:
                self.blocks[b].ref_count = 1
                self.free.remove(b)
                self.used.add(b)
            s.block_table.append(b)
        for _ in range(hits, self._nblocks(s)):
            s.block_table.append(self._fresh())
        s.num_cached_tokens = hits * self.bs

    def deallocate(self, sid):
        s = self.seqs[sid]
        for b in reversed(s.block_table):
            self.blocks[b].ref_count -= 1
            if self.blocks[b].ref_count == 0:
                self.used.remove(b)
                self.free.append(b)
        s.block_table = []
        s.num_cached_tokens = 0

    def remove_sequence(self, sid):
        self.deallocate(sid)
        del self.seqs[sid]

    def can_append(self, sid):
        return len(self.free) >= (1 if len(self.seqs[sid].tokens) % self.bs == 1 % self.bs else 0)

    def may_append(self, sid):
        s = self.seqs[sid]
        if len(s.tokens) % self.bs == 1 % self.bs:
            s.block_table.append(self._fresh())

    def postprocess(self, sid, scheduled):
        s = self.seqs[sid]
        start, end = s.num_cached_tokens // self.bs, (s.num_cached_tokens + scheduled) // self.bs
        h = self.blocks[s.block_table[start - 1]].hash if start > 0 else None
        for i in range(start, end):
            tok = self._block(s, i)
            h = _h(tok, h)
            blk = self.blocks[s.block_table[i]]
            blk.hash, blk.tokens = h, tok
            self.hash_to_block[h] = s.block_table[i]
        s.num_cached_tokens += scheduled

    # ---- queries and kernel inputs
    def num_free_blocks(self):
        return len(self.free)

    def ref_count(self, b):
        return self.blocks[b].ref_count

    def block_table(self, sid):
        return list(self.seqs[sid].block_table)

    def num_cached_tokens(self, sid):
        return self.seqs[sid].num_cached_tokens

    def decode_inputs(self, sids, max_blocks):
        slots, lens, tables = [], [], []
        for sid in sids:
            s = self.seqs[sid]
            n = len(s.tokens)
            slots.append(s.block_table[(n - 1) // self.bs] * self.bs + (n - 1) % self.bs)
            lens.append(n)
            tables.append(s.block_table + [-1] * (max_blocks - len(s.block_table)))
        return slots, lens, tables

    def prefill_inputs(self, sids, scheduled, max_blocks):
        slots, cq, ck, tables = [], [0], [0], []
        for sid, n in zip(sids, scheduled):
            s = self.seqs[sid]
            start, end = s.num_cached_tokens, s.num_cached_tokens + n
            for pos in range(start, end):  # each scheduled position's slot, one by one
                slots.append(s.block_table[pos // self.bs] * self.bs + pos % self.bs)
            cq.append(cq[-1] + n)
            ck.append(ck[-1] + end)
            tables.append(s.block_table + [-1] * (max_blocks - len(s.block_table)))
        return slots, cq, ck, tables
