"""Python binding of the native page directory (``include/pa_block_manager.h``):
argument marshalling only; every rule runs in the library's C++ code.

The manager decides which physical blocks of the paged KV pool each sequence
uses (with prefix caching) and emits the host-side kernel inputs of a step:
``slot_mapping``, ``cu_seqlens_q/k``, ``context_lens`` and ``-1``-padded
``block_tables`` as int32 tensors, ready for a pinned copy to the GPU.
"""

from __future__ import annotations

import ctypes

import torch

from . import _lib, PagedAttentionError, PrefixGroups

_p, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_I32P = ctypes.POINTER(ctypes.c_int32)
_I64P = ctypes.POINTER(ctypes.c_int64)

_lib.pa_bm_create.restype = _p
_lib.pa_bm_create.argtypes = [_i32, _i32]
_lib.pa_bm_destroy.restype = None
_lib.pa_bm_destroy.argtypes = [_p]
for _name, _args in (("pa_bm_add_sequence", [_p, _i64, _I32P, _i32]), ("pa_bm_append_token", [_p, _i64, _i32]),
                     ("pa_bm_remove_sequence", [_p, _i64]), ("pa_bm_can_allocate", [_p, _i64, _I32P]),
                     ("pa_bm_allocate", [_p, _i64, _i32]), ("pa_bm_deallocate", [_p, _i64]),
                     ("pa_bm_can_append", [_p, _i64]), ("pa_bm_may_append", [_p, _i64]),
                     ("pa_bm_postprocess", [_p, _i64, _i32]), ("pa_bm_num_free_blocks", [_p]),
                     ("pa_bm_ref_count", [_p, _i32]), ("pa_bm_block_table", [_p, _i64, _I32P, _i32]),
                     ("pa_bm_decode_inputs", [_p, _I64P, _i32, _i32, _I32P, _I32P, _I32P]),
                     ("pa_bm_prefill_inputs", [_p, _I64P, _I32P, _i32, _i32, _I32P, _I32P, _I32P, _I32P])):
    getattr(_lib, _name).restype = ctypes.c_int
    getattr(_lib, _name).argtypes = _args
_lib.pa_prefix_groups.restype = ctypes.c_int
_lib.pa_prefix_groups.argtypes = [_I32P, _i32, _I32P, _i32, _i32, _i32, _I32P, _I32P, _I32P, _I32P, _I32P, _I32P]
for _name in ("pa_bm_seq_len", "pa_bm_num_cached_tokens"):
    getattr(_lib, _name).restype = ctypes.c_int64
    getattr(_lib, _name).argtypes = [_p, _i64]


def _ok(fn: str, rc: int) -> int:
    if rc < 0:
        raise PagedAttentionError(fn, rc)
    return rc


def _i32buf(t: torch.Tensor):
    return ctypes.cast(t.data_ptr(), _I32P)


class BlockManager:
    """Prefix-cached block allocator over ``num_blocks`` blocks of ``block_size`` tokens."""

    def __init__(self, num_blocks: int, block_size: int):
        self._h = _lib.pa_bm_create(num_blocks, block_size)
        if not self._h:
            raise PagedAttentionError("pa_bm_create", -1)
        self.num_blocks, self.block_size = num_blocks, block_size

    def __del__(self):
        h, self._h = getattr(self, "_h", None), None
        if h:
            _lib.pa_bm_destroy(h)

    # ---- sequences
    def add_sequence(self, seq_id: int, token_ids: list[int]) -> None:
        arr = (ctypes.c_int32 * len(token_ids))(*token_ids)
        _ok("pa_bm_add_sequence", _lib.pa_bm_add_sequence(self._h, seq_id, arr, len(token_ids)))

    def append_token(self, seq_id: int, token_id: int) -> None:
        _ok("pa_bm_append_token", _lib.pa_bm_append_token(self._h, seq_id, token_id))

    def remove_sequence(self, seq_id: int) -> None:
        _ok("pa_bm_remove_sequence", _lib.pa_bm_remove_sequence(self._h, seq_id))

    # ---- allocation
    def can_allocate(self, seq_id: int) -> int:
        """Prefix-cache hits if the sequence can be allocated, -1 if the free blocks do not suffice."""
        hits = ctypes.c_int32()
        _ok("pa_bm_can_allocate", _lib.pa_bm_can_allocate(self._h, seq_id, ctypes.byref(hits)))
        return hits.value

    def allocate(self, seq_id: int, num_cached_blocks: int) -> None:
        _ok("pa_bm_allocate", _lib.pa_bm_allocate(self._h, seq_id, num_cached_blocks))

    def deallocate(self, seq_id: int) -> None:
        _ok("pa_bm_deallocate", _lib.pa_bm_deallocate(self._h, seq_id))

    def can_append(self, seq_id: int) -> bool:
        return bool(_ok("pa_bm_can_append", _lib.pa_bm_can_append(self._h, seq_id)))

    def may_append(self, seq_id: int) -> None:
        _ok("pa_bm_may_append", _lib.pa_bm_may_append(self._h, seq_id))

    def postprocess(self, seq_id: int, num_scheduled_tokens: int) -> None:
        _ok("pa_bm_postprocess", _lib.pa_bm_postprocess(self._h, seq_id, num_scheduled_tokens))

    # ---- queries
    def num_free_blocks(self) -> int:
        return _ok("pa_bm_num_free_blocks", _lib.pa_bm_num_free_blocks(self._h))

    def ref_count(self, block_id: int) -> int:
        return _ok("pa_bm_ref_count", _lib.pa_bm_ref_count(self._h, block_id))

    def block_table(self, seq_id: int) -> list[int]:
        n = _ok("pa_bm_block_table", _lib.pa_bm_block_table(self._h, seq_id, None, 0))
        out = (ctypes.c_int32 * max(n, 1))()
        _lib.pa_bm_block_table(self._h, seq_id, out, n)
        return list(out[:n])

    def seq_len(self, seq_id: int) -> int:
        return _ok("pa_bm_seq_len", _lib.pa_bm_seq_len(self._h, seq_id))

    def num_cached_tokens(self, seq_id: int) -> int:
        return _ok("pa_bm_num_cached_tokens", _lib.pa_bm_num_cached_tokens(self._h, seq_id))

    # ---- kernel inputs (host int32 tensors)
    def decode_inputs(self, seq_ids: list[int], max_blocks: int):
        """(slot_mapping [n], context_lens [n], block_tables [n, max_blocks])."""
        n = len(seq_ids)
        ids = (ctypes.c_int64 * max(n, 1))(*seq_ids)
        slots = torch.empty(n, dtype=torch.int32)
        lens = torch.empty(n, dtype=torch.int32)
        tables = torch.empty(n, max_blocks, dtype=torch.int32)
        _ok("pa_bm_decode_inputs", _lib.pa_bm_decode_inputs(self._h, ids, n, max_blocks, _i32buf(slots),
                                                            _i32buf(lens), _i32buf(tables)))
        return slots, lens, tables

    def prefill_inputs(self, seq_ids: list[int], num_scheduled: list[int], max_blocks: int):
        """(slot_mapping [sum scheduled], cu_seqlens_q [n+1], cu_seqlens_k [n+1], block_tables [n, max_blocks])."""
        n = len(seq_ids)
        ids = (ctypes.c_int64 * max(n, 1))(*seq_ids)
        sched = (ctypes.c_int32 * max(n, 1))(*num_scheduled)
        slots = torch.empty(max(sum(num_scheduled), 1), dtype=torch.int32)
        cq = torch.empty(n + 1, dtype=torch.int32)
        ck = torch.empty(n + 1, dtype=torch.int32)
        tables = torch.empty(n, max_blocks, dtype=torch.int32)
        _ok("pa_bm_prefill_inputs", _lib.pa_bm_prefill_inputs(self._h, ids, sched, n, max_blocks, _i32buf(slots),
                                                              _i32buf(cq), _i32buf(ck), _i32buf(tables)))
        return slots[:sum(num_scheduled)], cq, ck, tables


__all__ = ["BlockManager"]


def prefix_groups(block_tables: torch.Tensor, context_lens: torch.Tensor, block_size: int,
                  min_shared_pages: int = 1) -> PrefixGroups:
    """``pa_prefix_groups``: the shared-prefix groups of a decode batch from its host block
    tables ([B, max_blocks] int32, -1 padded) and context lengths ([B] int32), as host int32
    tensors (``.to(device)`` for the decode call)."""
    bt = block_tables.to(torch.int32).contiguous()
    cl = context_lens.to(torch.int32).contiguous()
    if bt.device.type != "cpu" or cl.device.type != "cpu" or bt.dim() != 2 or cl.numel() != bt.shape[0]:
        raise ValueError("block_tables [B, max_blocks] and context_lens [B] must be host tensors")
    B = bt.shape[0]
    off = torch.zeros(B // 2 + 1, dtype=torch.int32)
    seqs = torch.zeros(max(B, 1), dtype=torch.int32)
    pre = torch.zeros(max(B, 1), dtype=torch.int32)
    n, big, longest = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    rc = _lib.pa_prefix_groups(_i32buf(bt), bt.shape[1], _i32buf(cl), B, block_size, min_shared_pages, _i32buf(off),
                               _i32buf(seqs), _i32buf(pre), ctypes.byref(n), ctypes.byref(big), ctypes.byref(longest))
    if rc != 0:
        raise PagedAttentionError("pa_prefix_groups", rc)
    g = n.value
    # group_seqs keeps room for B entries (the decode call reads it within [0, batch))
    return PrefixGroups(off[:g + 1].clone(), seqs[:max(B, 1)].clone(), pre[:B].clone(), big.value, longest.value)
