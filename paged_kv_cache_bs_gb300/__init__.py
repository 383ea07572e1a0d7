"""Paged-KV attention for GB300 (sm_103a): Python binding of libpa.so.

Argument marshalling only: every step of the store, decode and prefill path
runs in the library's CUDA kernels.  torch supplies device memory and the
current stream.  Importing this package loads ``libpa.so`` and raises if it is
missing -- there is no fallback path.  Build it with
``python paged_kv_cache_bs_gb300/build.py``.

The functions mirror the C ABI in ``include/pa_api.h``:

* :func:`store_kv`       -- ``pa_store_kv``
* :func:`decode`         -- ``pa_decode`` (+ ``pa_decode_workspace_bytes``)
* :func:`store_decode`   -- ``pa_store_decode`` (the decode step's store fused into decode)
* :func:`store_kv_fp8`   -- ``pa_store_kv_fp8`` (quantising store into an E4M3 pool)
* :func:`decode_fp8`     -- ``pa_decode_fp8`` (+ ``pa_decode_fp8_workspace_bytes``)
* :func:`store_decode_fp8` -- ``pa_store_decode_fp8`` (the fp8 store fused into fp8 decode)
* :func:`prefill_paged`  -- ``pa_prefill_paged``
* :func:`mixed_step`     -- ``pa_mixed_step`` (store, chunked prefill and decode of one step;
  with an :class:`SmSplit` (``pa_sm_split_*``) the prefill and the decode run side by side)
* :func:`sample`         -- ``pa_sample`` (temperature sampling, exponential race)

``paged_kv_cache_bs_gb300.graphs.DecodeGraphRunner`` replays the decode step of a layer
from CUDA graphs captured per padded batch size; ``paged_kv_cache_bs_gb300.block_manager``
binds the native page directory.
"""

from __future__ import annotations

import ctypes
import os

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libpa.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(f"{LIB_PATH} is not built; run `python paged_kv_cache_bs_gb300/build.py`")

_lib = ctypes.CDLL(LIB_PATH)

_p, _i32, _i64, _f32, _sz = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_size_t
_lib.pa_last_error.restype = ctypes.c_char_p
_lib.pa_last_error.argtypes = []
_lib.pa_version.restype = ctypes.c_int
_lib.pa_store_kv.restype = ctypes.c_int
_lib.pa_store_kv.argtypes = [_p, _p, _i64, _i64, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _p, _p]
_lib.pa_decode_workspace_bytes.restype = _sz
_lib.pa_decode_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
_lib.pa_decode.restype = ctypes.c_int
_lib.pa_decode.argtypes = [_p, _i64, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _p, _p, _sz,
                           ctypes.c_int, _p, _p]
_lib.pa_store_decode.restype = ctypes.c_int
_lib.pa_store_decode.argtypes = [_p, _p, _i64, _i64, _p, _p, _i64, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32,
                                 _i32, _f32, _p, _p, _sz, ctypes.c_int, _p, _p]


class _Options(ctypes.Structure):
    """Mirror of pa_decode_options."""
    _fields_ = [("partition", _i32), ("stages", _i32), ("num_groups", _i32), ("max_group_size", _i32),
                ("max_prefix_len", _i32), ("prefix_partition", _i32), ("group_offsets", _p), ("group_seqs", _p),
                ("prefix_lens", _p), ("operands", _p)]


_opt_p = ctypes.POINTER(_Options)
_lib.pa_decode_ex_workspace_bytes.restype = _sz
_lib.pa_decode_ex_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _opt_p]
_lib.pa_decode_ex.restype = ctypes.c_int
_lib.pa_decode_ex.argtypes = [_p, _i64, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _p, _p, _sz,
                              _opt_p, ctypes.c_int, _p, _p]
_lib.pa_store_decode_ex.restype = ctypes.c_int
_lib.pa_store_decode_ex.argtypes = [_p, _p, _i64, _i64, _p, _p, _i64, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32,
                                    _i32, _i32, _f32, _p, _p, _sz, _opt_p, ctypes.c_int, _p, _p]
_lib.pa_store_kv_fp8.restype = ctypes.c_int
_lib.pa_store_kv_fp8.argtypes = [_p, _p, _i64, _i64, _p, _p, _p, _i32, _i32, _i32, _i32, _i32, ctypes.c_int, _f32, _f32,
                                 _p, _p]
_lib.pa_decode_fp8_workspace_bytes.restype = _sz
_lib.pa_decode_fp8_workspace_bytes.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32]
_lib.pa_decode_fp8.restype = ctypes.c_int
_lib.pa_decode_fp8.argtypes = [_p, _i64, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32, _i32, _i32, _f32, _f32, _f32, _p,
                               _p, _sz, ctypes.c_int, _p, _p]
_lib.pa_store_decode_fp8.restype = ctypes.c_int
_lib.pa_store_decode_fp8.argtypes = [_p, _p, _i64, _i64, _p, _p, _i64, _p, _p, _p, _i32, _p, _i32, _i32, _i32, _i32,
                                     _i32, _i32, _f32, _f32, _f32, _p, _p, _sz, ctypes.c_int, _p, _p]
_lib.pa_store_decode_fp8_ex.restype = ctypes.c_int
_lib.pa_store_decode_fp8_ex.argtypes = [_p, _p, _i64, _i64, _p, _p, _i64, _p, _p, _p, _i32, _p, _i32, _i32, _i32,
                                        _i32, _i32, _i32, _f32, _f32, _f32, _p, _p, _sz, _opt_p, ctypes.c_int, _p, _p]
_lib.pa_sample.restype = ctypes.c_int
_lib.pa_sample.argtypes = [_p, _i64, _i32, _i32, ctypes.c_int, _p, _p, ctypes.c_uint64, ctypes.c_uint64, _p, _p, _p]
_lib.pa_selftest_wait_timeout.restype = ctypes.c_int
_lib.pa_selftest_wait_timeout.argtypes = [_i64, _p, _p]
_lib.pa_sm_split_create.restype = ctypes.c_int
_lib.pa_sm_split_create.argtypes = [_i32, ctypes.POINTER(ctypes.c_void_p)]
_lib.pa_sm_split_info.restype = ctypes.c_int
_lib.pa_sm_split_info.argtypes = [_p, ctypes.POINTER(_i32), ctypes.POINTER(_i32), _p, _p]
_lib.pa_sm_split_destroy.restype = None
_lib.pa_sm_split_destroy.argtypes = [_p]
_lib.pa_mixed_step.restype = ctypes.c_int
_lib.pa_mixed_step.argtypes = [_p, _p, _i64, _i64, _p, _i32, _p, _p, _p, _i32, _i32, _i32, _i32, _p, _i32, _p, _p, _i64,
                               _p, _i32, _p, _i32, _p, _p, _sz, _p, _p, _i32, _i32, _i32, _i32, _i32, _f32,
                               ctypes.c_int, _p, _p, _p]
_lib.pa_prefill_paged.restype = ctypes.c_int
_lib.pa_prefill_paged.argtypes = [_p, _p, _p, _p, _p, _p, _p, _i32, _i32, _i32, _i32, _p, _i32, _i32, _i32, _i32,
                                  _i32, _i32, _f32, _p, ctypes.c_int, _p, _p]


class _PrefillOptions(ctypes.Structure):
    _fields_ = [("max_ctas", ctypes.c_int32)]


_lib.pa_prefill_paged_ex.restype = ctypes.c_int
_lib.pa_prefill_paged_ex.argtypes = _lib.pa_prefill_paged.argtypes[:-1] + [ctypes.POINTER(_PrefillOptions), _p]

class CopySegment(ctypes.Structure):
    """Mirror of pa_copy_segment."""
    _fields_ = [("src", _p), ("dst", _p), ("bytes", ctypes.c_uint64)]


_lib.pa_copy_segments.restype = ctypes.c_int
_lib.pa_copy_segments.argtypes = [_p, _i32, _p]


class DecodeStaging(ctypes.Structure):
    """Mirror of pa_decode_staging (the host arrays of one captured decode bucket)."""
    _fields_ = [("rows", _i32), ("max_blocks", _i32), ("block_size", _i32),
                ("slot_mapping", _p), ("context_lens", _p), ("block_tables", _p),
                ("max_groups", _i32), ("max_group_size", _i32), ("max_prefix_len", _i32),
                ("group_offsets", _p), ("group_seqs", _p), ("prefix_lens", _p),
                ("segments", _p), ("num_segments", _i32), ("segment_row_bytes", ctypes.c_uint64 * 4),
                ("operands", _p)]


STAGE_NO_GROUPS, STAGE_DERIVE_GROUPS, STAGE_KEEP_GROUPS = 0, 1, 2
_lib.pa_stage_decode_step.restype = ctypes.c_int
_lib.pa_stage_decode_step.argtypes = [_p, _i32, _p, _p, _p, _i32, _i32, _p]

PA_F16, PA_BF16, PA_F32, PA_E4M3 = 0, 1, 2, 3
_FP8_POOL = (torch.uint8, torch.float8_e4m3fn)  # E4M3 codes, one byte per element
_DTYPES = {torch.float16: PA_F16, torch.bfloat16: PA_BF16}
FLAG_BAD_SLOT, FLAG_BAD_BLOCK, FLAG_BAD_LENGTH, FLAG_TIMEOUT, FLAG_INTERNAL, FLAG_BAD_VALUE = 1, 2, 4, 8, 16, 32
FLAG_BAD_GROUP = 64


class PagedAttentionError(RuntimeError):
    """A libpa call returned an error code."""

    def __init__(self, fn: str, code: int):
        super().__init__(f"{fn} failed ({code}): {_lib.pa_last_error().decode()}")
        self.code = code


def library() -> ctypes.CDLL:
    """The loaded libpa.so handle (for direct C-ABI calls)."""
    return _lib


def _ptr(t) -> ctypes.c_void_p | None:
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(t: torch.Tensor) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _check(fn: str, rc: int) -> None:
    if rc != 0:
        raise PagedAttentionError(fn, rc)


def _dtype(t: torch.Tensor) -> int:
    if t.dtype not in _DTYPES:
        raise TypeError(f"unsupported dtype {t.dtype}; use float16 or bfloat16")
    return _DTYPES[t.dtype]


def _cache_shape(k_cache: torch.Tensor, v_cache: torch.Tensor):
    if k_cache.dim() != 4 or k_cache.shape != v_cache.shape:
        raise ValueError("k_cache / v_cache must both be [num_blocks, block_size, H_kv, D]")
    if not (k_cache.is_contiguous() and v_cache.is_contiguous()):
        raise ValueError("k_cache / v_cache must be contiguous")
    if not (k_cache.is_cuda and v_cache.is_cuda):
        raise ValueError("k_cache / v_cache must be CUDA tensors")
    return k_cache.shape


def _rows(t: torch.Tensor, name: str) -> int:
    """Row stride (elements) of a [T, H, D] tensor whose heads/dims are contiguous."""
    if t.dim() != 3 or t.stride(2) != 1 or t.stride(1) != t.shape[2]:
        raise ValueError(f"{name} must be [T, H, D] with contiguous heads and dims")
    return t.stride(0)


def store_kv(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
             slot_mapping: torch.Tensor, err_flag: torch.Tensor | None = None) -> None:
    """Write rows of k/v ([T, H_kv, D]) to cache rows ``slot_mapping`` (int32; -1 skips)."""
    n, bs, hkv, d = _cache_shape(k_cache, v_cache)
    if slot_mapping.dtype != torch.int32 or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int32")
    if k.shape[0] != slot_mapping.numel() or v.shape[0] != slot_mapping.numel():
        raise ValueError("k/v rows must match slot_mapping")
    if k.shape[1:] != (hkv, d) or v.shape[1:] != (hkv, d):
        raise ValueError("k/v must be [T, H_kv, D] matching the cache")
    if k.dtype != k_cache.dtype or v.dtype != k_cache.dtype:
        raise TypeError("k/v dtype must match the cache")
    _step_operands(k_cache, k=k, v=v, slot_mapping=slot_mapping)
    rc = _lib.pa_store_kv(_ptr(k), _ptr(v), _rows(k, "k"), _rows(v, "v"), _ptr(k_cache), _ptr(v_cache),
                          _ptr(slot_mapping), slot_mapping.numel(), hkv, d, n, bs, _dtype(k_cache), _ptr(err_flag),
                          _stream(k_cache))
    _check("pa_store_kv", rc)


class PrefixGroups:
    """Shared-prefix groups of a decode batch (``pa_prefix_groups``): the members of group g are
    ``group_seqs[group_offsets[g]:group_offsets[g + 1]]`` (``group_seqs`` has room for the whole
    batch; entries past the last offset are unused); ``prefix_lens[b]`` tokens at the start
    of sequence b's context are read once for its whole group (0: not grouped).  int32 tensors,
    on the host as computed, on the device for a decode call (:meth:`to`)."""

    def __init__(self, group_offsets: torch.Tensor, group_seqs: torch.Tensor, prefix_lens: torch.Tensor,
                 max_group_size: int, max_prefix_len: int):
        self.group_offsets, self.group_seqs, self.prefix_lens = group_offsets, group_seqs, prefix_lens
        self.max_group_size, self.max_prefix_len = int(max_group_size), int(max_prefix_len)

    @property
    def num_groups(self) -> int:
        return self.group_offsets.numel() - 1

    def to(self, device) -> "PrefixGroups":
        return PrefixGroups(self.group_offsets.to(device), self.group_seqs.to(device), self.prefix_lens.to(device),
                            self.max_group_size, self.max_prefix_len)


class DecodeOptions:
    """Optional settings of :func:`decode` / :func:`store_decode` (``pa_decode_options``).

    ``partition``: tokens per split-K partition (a multiple of 64; 0 = the library's plan).
    ``stages``: TMA ring depth of the partition kernel, 2 or 3 (0 = the plan).
    ``groups``: shared-prefix groups (:class:`PrefixGroups` on the call's device, or in pinned
    host memory): each group's shared pages are read once for all its sequences.
    ``prefix_partition``: tokens per partition of a shared prefix (0 = the plan).
    ``operands``: the address of three pointers {q, k, v} in device-readable memory (page-locked
    host or device), read by the kernels when they run in place of the call's q, k and v (0 = the
    call's own)."""

    def __init__(self, partition: int = 0, stages: int = 0, groups: PrefixGroups | None = None,
                 prefix_partition: int = 0, operands: int = 0):
        self.partition, self.stages = int(partition), int(stages)
        self.groups, self.prefix_partition = groups, int(prefix_partition)
        self.operands = int(operands)

    def _c(self) -> _Options:
        g = self.groups
        ops = self.operands or None
        if g is None or g.num_groups == 0:
            return _Options(self.partition, self.stages, 0, 0, 0, self.prefix_partition, None, None, None, ops)
        for name in ("group_offsets", "group_seqs", "prefix_lens"):
            t = getattr(g, name)
            if t.dtype != torch.int32 or not t.is_contiguous():
                raise ValueError(f"groups.{name} must be contiguous int32")
        return _Options(self.partition, self.stages, g.num_groups, max(g.max_group_size, 1),
                        max(g.max_prefix_len, 1), self.prefix_partition, g.group_offsets.data_ptr(),
                        g.group_seqs.data_ptr(), g.prefix_lens.data_ptr(), ops)


def _opts(options: DecodeOptions | None):
    return None if options is None else ctypes.byref(options._c())


def decode_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                           max_blocks_per_seq: int, block_size: int, options: DecodeOptions | None = None) -> int:
    if options is None:
        return int(_lib.pa_decode_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                                  block_size))
    return int(_lib.pa_decode_ex_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                                 block_size, _opts(options)))


def alloc_decode_workspace(q: torch.Tensor, k_cache: torch.Tensor, block_tables: torch.Tensor,
                           options: DecodeOptions | None = None) -> torch.Tensor:
    n, bs, hkv, d = k_cache.shape
    nbytes = decode_workspace_bytes(q.shape[0], q.shape[1], hkv, d, block_tables.shape[1], bs, options)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=k_cache.device)


def _step_operands(k_cache: torch.Tensor, **tensors) -> None:
    """The per-step operands of the store, the fused decode calls and the sampler (q, the new k/v
    rows, slot mapping, block tables, context lengths, logits, temperatures, out) may live on the
    device or in page-locked host memory, which the kernels then read and write directly over the
    CPU-GPU link (with unified addressing a pinned host pointer is also a device pointer).
    Pageable host memory is refused.  ``k_cache``: any tensor on the device the call runs on."""
    for name, t in tensors.items():
        if t is None:
            continue
        if t.device == k_cache.device:
            continue
        if t.device.type == "cpu" and t.is_pinned():
            continue
        raise ValueError(f"{name} must be on {k_cache.device} or in pinned host memory")


def _device_only(k_cache: torch.Tensor, **tensors) -> None:
    """Operands a kernel reads by TMA or that the C ABI takes as device memory only: on the device of
    the call (``k_cache``'s).  A host tensor would reach the kernel as a host pointer."""
    for name, t in tensors.items():
        if t is not None and t.device != k_cache.device:
            raise ValueError(f"{name} must be on {k_cache.device}")


def _decode_checks(q, k_cache, v_cache, block_tables, context_lens):
    n, bs, hkv, d = _cache_shape(k_cache, v_cache)
    B = q.shape[0]
    if q.dim() != 3 or q.shape[2] != d:
        raise ValueError("q must be [B, H_q, D]")
    for name, t in (("block_tables", block_tables), ("context_lens", context_lens)):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
    if block_tables.dim() != 2 or block_tables.shape[0] != B or context_lens.numel() != B:
        raise ValueError("block_tables must be [B, max_blocks] and context_lens [B]")
    return n, bs, hkv, d


def decode(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
           context_lens: torch.Tensor, scale: float, out: torch.Tensor | None = None,
           workspace: torch.Tensor | None = None, err_flag: torch.Tensor | None = None,
           options: DecodeOptions | None = None) -> torch.Tensor:
    """Paged decode attention: q [B, H_q, D] -> out [B, H_q, D] (``pa_decode``, or
    ``pa_decode_ex`` with ``options``)."""
    n, bs, hkv, d = _decode_checks(q, k_cache, v_cache, block_tables, context_lens)
    _device_only(k_cache, q=q, block_tables=block_tables, context_lens=context_lens, out=out)
    B, hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty(B, hq, d, dtype=q.dtype, device=q.device)
    if workspace is None:
        workspace = alloc_decode_workspace(q, k_cache, block_tables, options)
    args = (_ptr(q), _rows(q, "q"), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1],
            _ptr(context_lens), B, hq, hkv, d, n, bs, float(scale), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size())
    tail = (_dtype(q), _ptr(err_flag), _stream(q))
    if options is None:
        _check("pa_decode", _lib.pa_decode(*args, *tail))
    else:
        _check("pa_decode_ex", _lib.pa_decode_ex(*args, _opts(options), *tail))
    return out


def store_decode(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, q: torch.Tensor,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                 context_lens: torch.Tensor, scale: float, out: torch.Tensor | None = None,
                 workspace: torch.Tensor | None = None, err_flag: torch.Tensor | None = None,
                 options: DecodeOptions | None = None) -> torch.Tensor:
    """One decode step in one launch: store k/v ([B, H_kv, D]) at ``slot_mapping`` (the slot of
    each sequence's last context position, or -1) and attend: q [B, H_q, D] -> out [B, H_q, D]
    (``pa_store_decode``, or ``pa_store_decode_ex`` with ``options``)."""
    n, bs, hkv, d = _decode_checks(q, k_cache, v_cache, block_tables, context_lens)
    B, hq = q.shape[0], q.shape[1]
    if slot_mapping.dtype != torch.int32 or not slot_mapping.is_contiguous() or slot_mapping.numel() != B:
        raise ValueError("slot_mapping must be contiguous int32 [B]")
    if k.shape != (B, hkv, d) or v.shape != (B, hkv, d) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k/v must be [B, H_kv, D] of the cache dtype")
    _step_operands(k_cache, q=q, k=k, v=v, slot_mapping=slot_mapping, block_tables=block_tables,
                   context_lens=context_lens, out=out)
    if out is None:
        out = torch.empty(B, hq, d, dtype=q.dtype, device=k_cache.device)
    if workspace is None:
        workspace = alloc_decode_workspace(q, k_cache, block_tables, options)
    args = (_ptr(k), _ptr(v), _rows(k, "k"), _rows(v, "v"), _ptr(slot_mapping), _ptr(q), _rows(q, "q"),
            _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, hq, hkv,
            d, n, bs, float(scale), _ptr(out), _ptr(workspace), workspace.numel() * workspace.element_size())
    tail = (_dtype(q), _ptr(err_flag), _stream(k_cache))
    if options is None:
        _check("pa_store_decode", _lib.pa_store_decode(*args, *tail))
    else:
        _check("pa_store_decode_ex", _lib.pa_store_decode_ex(*args, _opts(options), *tail))
    return out


def prefill_paged(q: torch.Tensor, k: torch.Tensor | None, v: torch.Tensor | None, k_cache: torch.Tensor,
                  v_cache: torch.Tensor, cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor,
                  max_seqlen_q: int, max_seqlen_k: int, block_tables: torch.Tensor | None, scale: float,
                  out: torch.Tensor | None = None, err_flag: torch.Tensor | None = None,
                  max_ctas: int = 0) -> torch.Tensor:
    """Causal varlen prefill over a paged prefix: q [Tq, H_q, D] -> out [Tq, H_q, D].
    ``max_ctas`` > 0 caps the persistent grid (``pa_prefill_paged_ex``), e.g. at the SM count of
    a green-context partition."""
    n, bs, hkv, d = _cache_shape(k_cache, v_cache)
    _device_only(k_cache, q=q, k=k, v=v, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                 block_tables=block_tables)
    _step_operands(k_cache, out=out)  # written by plain stores: the device, or page-locked host memory
    tq, hq = q.shape[0], q.shape[1]
    if not q.is_contiguous():
        raise ValueError("q must be contiguous [Tq, H_q, D]")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k)):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
    if block_tables is not None and (block_tables.dtype != torch.int32 or not block_tables.is_contiguous()):
        raise ValueError("block_tables must be contiguous int32")
    for name, t in (("k", k), ("v", v)):
        if t is not None and not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous")
    if out is None:
        out = torch.empty(tq, hq, d, dtype=q.dtype, device=q.device)
    args = (_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache), _ptr(v_cache), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k),
            cu_seqlens_q.numel() - 1, tq, int(max_seqlen_q), int(max_seqlen_k), _ptr(block_tables),
            block_tables.shape[1] if block_tables is not None else 0, hq, hkv, d, n, bs, float(scale), _ptr(out),
            _dtype(q), _ptr(err_flag))
    if max_ctas:
        opt = _PrefillOptions(int(max_ctas))
        rc = _lib.pa_prefill_paged_ex(*args, ctypes.byref(opt), _stream(q))
        _check("pa_prefill_paged_ex", rc)
    else:
        rc = _lib.pa_prefill_paged(*args, _stream(q))
        _check("pa_prefill_paged", rc)
    return out


def copy_segments(segments_ptr: int, count: int, stream: int | None = None) -> None:
    """``pa_copy_segments``: ``count`` copies in one kernel, the :class:`CopySegment` list at
    address ``segments_ptr`` (page-locked host or device memory) read when the kernel runs;
    ``stream`` is a raw stream handle (default: the current stream)."""
    if stream is None:
        stream = torch.cuda.current_stream().cuda_stream
    _check("pa_copy_segments", _lib.pa_copy_segments(ctypes.c_void_p(segments_ptr), int(count),
                                                       ctypes.c_void_p(stream)))


def stage_decode_step(staging: DecodeStaging, slot_mapping: torch.Tensor, context_lens: torch.Tensor,
                      block_tables: torch.Tensor, groups: int = STAGE_NO_GROUPS, sources=None) -> None:
    """``pa_stage_decode_step``: one decode step's metadata (contiguous host int32 tensors, batch =
    ``slot_mapping.numel()``) into the pinned arrays ``staging`` names, rows past the batch padded;
    ``groups`` one of the STAGE_* modes; ``sources`` None or the addresses of the step's q and new
    K / V rows for the staging's gather list.  Host only."""
    batch = slot_mapping.numel()
    for name, t in (("slot_mapping", slot_mapping), ("context_lens", context_lens), ("block_tables", block_tables)):
        if t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be a contiguous host int32 tensor")
    if context_lens.numel() != batch or block_tables.dim() != 2 or block_tables.shape[0] != batch:
        raise ValueError(f"context_lens and block_tables must hold {batch} rows")
    src = None
    if sources is not None:
        src = (ctypes.c_void_p * max(len(sources), 1))(*sources)
    _check("pa_stage_decode_step", _lib.pa_stage_decode_step(
        ctypes.addressof(staging), batch, slot_mapping.data_ptr(), context_lens.data_ptr(), block_tables.data_ptr(),
        block_tables.shape[1], int(groups), None if src is None else ctypes.addressof(src)))


def selftest_wait_timeout(err_flag: torch.Tensor, max_cycles: int = 2_000_000) -> None:
    """``pa_selftest_wait_timeout``: a bounded wait that nothing satisfies gives up after
    ``max_cycles`` and ORs FLAG_TIMEOUT into ``err_flag`` (a CUDA int32 tensor)."""
    if err_flag.dtype != torch.int32 or not err_flag.is_cuda:
        raise ValueError("err_flag must be a CUDA int32 tensor")
    _check("pa_selftest_wait_timeout", _lib.pa_selftest_wait_timeout(int(max_cycles), _ptr(err_flag),
                                                                      _stream(err_flag)))


class SmSplit:
    """``pa_sm_split``: the current device's SMs as two disjoint partitions with their own streams
    (``first_sms`` SMs, a multiple of 8, and the rest), for :func:`mixed_step`.  Create one at
    start-up and reuse it; :meth:`close` (or garbage collection) releases it."""

    def __init__(self, first_sms: int):
        self._h = None
        h = ctypes.c_void_p()
        _check("pa_sm_split_create", _lib.pa_sm_split_create(int(first_sms), ctypes.byref(h)))
        self._h = h
        a, b = ctypes.c_int32(), ctypes.c_int32()
        _check("pa_sm_split_info", _lib.pa_sm_split_info(h, ctypes.byref(a), ctypes.byref(b), None, None))
        self.sms = (a.value, b.value)

    @property
    def handle(self) -> ctypes.c_void_p:
        if self._h is None:
            raise ValueError("the SM split is closed")
        return self._h

    def close(self) -> None:
        if getattr(self, "_h", None) is not None:
            _lib.pa_sm_split_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:  # interpreter shutdown: the library may already be unloaded
            pass


def mixed_step(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, prefill_q: torch.Tensor,
               cu_seqlens_q: torch.Tensor, cu_seqlens_k: torch.Tensor, max_seqlen_q: int, max_seqlen_k: int,
               prefill_block_tables: torch.Tensor, decode_q: torch.Tensor, decode_block_tables: torch.Tensor,
               context_lens: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, scale: float,
               prefill_out: torch.Tensor | None = None, decode_out: torch.Tensor | None = None,
               workspace: torch.Tensor | None = None, split: SmSplit | None = None,
               err_flag: torch.Tensor | None = None) -> tuple[torch.Tensor, torch.Tensor]:
    """``pa_mixed_step``: store every new token (k/v [T, H_kv, D] at ``slot_mapping``), then the
    chunked prefill of ``prefill_q`` [Tq, H_q, D] over the pool and the decode of ``decode_q``
    [B, H_q, D]; with ``split`` the prefill and the decode run at once on its two SM partitions.
    Returns (prefill_out, decode_out)."""
    n, bs, hkv, d = _decode_checks(decode_q, k_cache, v_cache, decode_block_tables, context_lens)
    _device_only(k_cache, prefill_q=prefill_q, cu_seqlens_q=cu_seqlens_q, cu_seqlens_k=cu_seqlens_k,
                 prefill_block_tables=prefill_block_tables, workspace=workspace)
    _step_operands(k_cache, k=k, v=v, slot_mapping=slot_mapping, decode_q=decode_q,
                   decode_block_tables=decode_block_tables, context_lens=context_lens, prefill_out=prefill_out,
                   decode_out=decode_out)
    B, hq = decode_q.shape[0], decode_q.shape[1]
    tq = prefill_q.shape[0]
    if slot_mapping.dtype != torch.int32 or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int32")
    if k.shape != (slot_mapping.numel(), hkv, d) or v.shape != k.shape or k.dtype != k_cache.dtype or v.dtype != k.dtype:
        raise ValueError("k/v must be [T, H_kv, D] of the cache dtype, one row per slot")
    if not prefill_q.is_contiguous() or prefill_q.dim() != 3 or prefill_q.shape[1:] != (hq, d):
        raise ValueError("prefill_q must be contiguous [Tq, H_q, D]")
    for name, t in (("cu_seqlens_q", cu_seqlens_q), ("cu_seqlens_k", cu_seqlens_k),
                    ("prefill_block_tables", prefill_block_tables)):
        if t.dtype != torch.int32 or not t.is_contiguous():
            raise ValueError(f"{name} must be contiguous int32")
    if prefill_out is None:
        prefill_out = torch.empty(tq, hq, d, dtype=prefill_q.dtype, device=k_cache.device)
    if decode_out is None:
        decode_out = torch.empty(B, hq, d, dtype=decode_q.dtype, device=k_cache.device)
    if workspace is None:
        workspace = alloc_decode_workspace(decode_q, k_cache, decode_block_tables)
    rc = _lib.pa_mixed_step(
        _ptr(k), _ptr(v), _rows(k, "k"), _rows(v, "v"), _ptr(slot_mapping), slot_mapping.numel(),
        _ptr(prefill_q), _ptr(cu_seqlens_q), _ptr(cu_seqlens_k), cu_seqlens_q.numel() - 1, tq, int(max_seqlen_q),
        int(max_seqlen_k), _ptr(prefill_block_tables), prefill_block_tables.shape[1], _ptr(prefill_out),
        _ptr(decode_q), _rows(decode_q, "decode_q"), _ptr(decode_block_tables), decode_block_tables.shape[1],
        _ptr(context_lens), B, _ptr(decode_out), _ptr(workspace), workspace.numel() * workspace.element_size(),
        _ptr(k_cache), _ptr(v_cache), hq, hkv, d, n, bs, float(scale), _dtype(decode_q), _ptr(err_flag),
        split.handle if split is not None else None, _stream(k_cache))
    _check("pa_mixed_step", rc)
    return prefill_out, decode_out


def _fp8_pool(k_cache: torch.Tensor, v_cache: torch.Tensor):
    if k_cache.dtype not in _FP8_POOL or v_cache.dtype not in _FP8_POOL:
        raise TypeError("an fp8 pool holds E4M3 codes: torch.uint8 or torch.float8_e4m3fn")
    return _cache_shape(k_cache, v_cache)


def store_kv_fp8(k: torch.Tensor, v: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                 slot_mapping: torch.Tensor, k_scale: float, v_scale: float,
                 err_flag: torch.Tensor | None = None) -> None:
    """Quantise rows of k/v ([T, H_kv, D], fp16/bf16) to E4M3 codes (x / scale, nearest even,
    saturating) into the fp8 pool at ``slot_mapping`` (int32; -1 skips)."""
    n, bs, hkv, d = _fp8_pool(k_cache, v_cache)
    if slot_mapping.dtype != torch.int32 or not slot_mapping.is_contiguous():
        raise ValueError("slot_mapping must be contiguous int32")
    if k.shape[0] != slot_mapping.numel() or v.shape[0] != slot_mapping.numel():
        raise ValueError("k/v rows must match slot_mapping")
    if k.shape[1:] != (hkv, d) or v.shape[1:] != (hkv, d):
        raise ValueError("k/v must be [T, H_kv, D] matching the cache")
    if k.dtype != v.dtype:
        raise TypeError("k and v must have one dtype")
    rc = _lib.pa_store_kv_fp8(_ptr(k), _ptr(v), _rows(k, "k"), _rows(v, "v"), _ptr(k_cache), _ptr(v_cache),
                              _ptr(slot_mapping), slot_mapping.numel(), hkv, d, n, bs, _dtype(k), float(k_scale),
                              float(v_scale), _ptr(err_flag), _stream(k_cache))
    _check("pa_store_kv_fp8", rc)


def decode_fp8_workspace_bytes(batch: int, num_q_heads: int, num_kv_heads: int, head_dim: int,
                               max_blocks_per_seq: int, block_size: int) -> int:
    return int(_lib.pa_decode_fp8_workspace_bytes(batch, num_q_heads, num_kv_heads, head_dim, max_blocks_per_seq,
                                                  block_size))


def decode_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
               context_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float,
               out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
               err_flag: torch.Tensor | None = None) -> torch.Tensor:
    """Paged decode over an fp8 pool (K = code * k_scale, V = code * v_scale): q [B, H_q, D] -> out."""
    _fp8_pool(k_cache, v_cache)
    n, bs, hkv, d = _decode_checks(q, k_cache, v_cache, block_tables, context_lens)
    _device_only(k_cache, q=q, block_tables=block_tables, context_lens=context_lens, out=out)
    B, hq = q.shape[0], q.shape[1]
    if out is None:
        out = torch.empty(B, hq, d, dtype=q.dtype, device=q.device)
    workspace = _fp8_workspace(q, hkv, d, block_tables, bs, workspace)
    rc = _lib.pa_decode_fp8(_ptr(q), _rows(q, "q"), _ptr(k_cache), _ptr(v_cache), _ptr(block_tables),
                            block_tables.shape[1], _ptr(context_lens), B, hq, hkv, d, n, bs, float(scale),
                            float(k_scale), float(v_scale), _ptr(out), _ptr(workspace),
                            workspace.numel() * workspace.element_size(), _dtype(q), _ptr(err_flag), _stream(q))
    _check("pa_decode_fp8", rc)
    return out


def _fp8_workspace(q, hkv, d, block_tables, bs, workspace, device=None):
    if workspace is None:
        nbytes = decode_fp8_workspace_bytes(q.shape[0], q.shape[1], hkv, d, block_tables.shape[1], bs)
        workspace = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device or q.device)
    return workspace


def store_decode_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor, q: torch.Tensor,
                     k_cache: torch.Tensor, v_cache: torch.Tensor, block_tables: torch.Tensor,
                     context_lens: torch.Tensor, scale: float, k_scale: float, v_scale: float,
                     out: torch.Tensor | None = None, workspace: torch.Tensor | None = None,
                     err_flag: torch.Tensor | None = None, operands: int = 0) -> torch.Tensor:
    """One decode step over an fp8 pool in one launch: quantise k/v ([B, H_kv, D]) into slot
    ``slot_mapping`` (each sequence's last context position, or -1) and attend.  ``operands``: as
    :class:`DecodeOptions` (``pa_store_decode_fp8_ex``; the only option an E4M3 pool takes)."""
    _fp8_pool(k_cache, v_cache)
    n, bs, hkv, d = _decode_checks(q, k_cache, v_cache, block_tables, context_lens)
    B, hq = q.shape[0], q.shape[1]
    if slot_mapping.dtype != torch.int32 or not slot_mapping.is_contiguous() or slot_mapping.numel() != B:
        raise ValueError("slot_mapping must be contiguous int32 [B]")
    if k.shape != (B, hkv, d) or v.shape != (B, hkv, d) or k.dtype != q.dtype or v.dtype != q.dtype:
        raise ValueError("k/v must be [B, H_kv, D] of the query dtype")
    _step_operands(k_cache, q=q, k=k, v=v, slot_mapping=slot_mapping, block_tables=block_tables,
                   context_lens=context_lens, out=out)
    if out is None:
        out = torch.empty(B, hq, d, dtype=q.dtype, device=k_cache.device)
    workspace = _fp8_workspace(q, hkv, d, block_tables, bs, workspace, k_cache.device)
    args = (_ptr(k), _ptr(v), _rows(k, "k"), _rows(v, "v"), _ptr(slot_mapping), _ptr(q), _rows(q, "q"),
            _ptr(k_cache), _ptr(v_cache), _ptr(block_tables), block_tables.shape[1], _ptr(context_lens), B, hq, hkv,
            d, n, bs, float(scale), float(k_scale), float(v_scale), _ptr(out), _ptr(workspace),
            workspace.numel() * workspace.element_size())
    if operands:
        rc = _lib.pa_store_decode_fp8_ex(*args, _opts(DecodeOptions(operands=operands)), _dtype(q), _ptr(err_flag),
                                         _stream(k_cache))
        _check("pa_store_decode_fp8_ex", rc)
    else:
        rc = _lib.pa_store_decode_fp8(*args, _dtype(q), _ptr(err_flag), _stream(k_cache))
        _check("pa_store_decode_fp8", rc)
    return out


def sample(logits: torch.Tensor, temperatures: torch.Tensor, noise: torch.Tensor | None = None, seed: int = 0,
           offset: int = 0, out: torch.Tensor | None = None, err_flag: torch.Tensor | None = None,
           device: torch.device | None = None) -> torch.Tensor:
    """One token per row of logits [B, V] (fp32/bf16/fp16): argmax of softmax(logits / T) / max(E, 1e-10),
    E ~ Exp(1) from ``noise`` [B, V] fp32 or, if None, drawn in-kernel from Philox4x32-10 at (seed, offset).
    The operands may be on the GPU or in pinned host memory (read and written by the kernel directly);
    ``device`` (default: that of ``logits`` if on the GPU, else the current device) runs the kernel."""
    if device is None:
        device = logits.device if logits.is_cuda else torch.device("cuda", torch.cuda.current_device())
    anchor = torch.empty(0, device=device)
    if logits.dim() != 2 or logits.stride(1) != 1:
        raise ValueError("logits must be a [B, V] tensor with contiguous rows")
    _step_operands(anchor, logits=logits, temperatures=temperatures, noise=noise, out=out)
    dt = {torch.float32: PA_F32, torch.bfloat16: PA_BF16, torch.float16: PA_F16}.get(logits.dtype)
    if dt is None:
        raise TypeError("logits must be fp32, bf16 or fp16")
    B, V = logits.shape
    if temperatures.dtype != torch.float32 or temperatures.numel() != B or not temperatures.is_contiguous():
        raise ValueError("temperatures must be contiguous fp32 [B]")
    if noise is not None and (noise.dtype != torch.float32 or tuple(noise.shape) != (B, V) or not noise.is_contiguous()):
        raise ValueError("noise must be contiguous fp32 [B, V]")
    if out is None:
        out = torch.empty(B, dtype=torch.int32, device=device)
    rc = _lib.pa_sample(_ptr(logits), logits.stride(0), B, V, dt, _ptr(temperatures), _ptr(noise), seed, offset,
                        _ptr(out), _ptr(err_flag), _stream(anchor))
    _check("pa_sample", rc)
    return out


__all__ = ["copy_segments", "CopySegment", "stage_decode_step", "DecodeStaging", "STAGE_NO_GROUPS", "STAGE_DERIVE_GROUPS",
           "STAGE_KEEP_GROUPS", "store_kv", "decode", "store_decode", "prefill_paged", "sample", "store_kv_fp8", "decode_fp8",
           "store_decode_fp8", "mixed_step", "SmSplit",
           "decode_workspace_bytes", "decode_fp8_workspace_bytes", "alloc_decode_workspace", "library",
           "PagedAttentionError", "LIB_PATH", "PA_F16", "PA_BF16", "PA_F32", "PA_E4M3", "FLAG_BAD_SLOT", "FLAG_BAD_BLOCK",
           "FLAG_BAD_LENGTH", "FLAG_TIMEOUT", "FLAG_INTERNAL", "FLAG_BAD_VALUE"]
