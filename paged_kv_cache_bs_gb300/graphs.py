"""Bucketed CUDA-graph replay of the decode step.

"nano-vLLM Part 2: Block Tables, KV Cache, and the Path to the GPU", section
4.2: decode has one input token per live sequence, so the runner records one
CUDA graph per padded batch size at start-up (1, 2, 4, 8, 16, 32, ... up to the
batch limit), and a step copies its slot mapping, context lengths and block
tables into the graph's fixed buffers, pads the unused rows (slot -1, context
length 0), replays the smallest graph that fits and keeps the first rows of
the output.

Here one graph holds the whole step of one attention layer.  By default
(``zero_copy=True``) it is the fused store + decode (``pa_store_decode``, or
``pa_store_decode_fp8`` over an E4M3 pool) with its per-step operands in host
memory, read over the CPU-GPU link (NVLink-C2C on a Grace-based GB300): the
kernels read the slot mapping, context lengths and block tables from the
pinned staging and write the output into pinned memory directly, so the step
has no copy-engine transfer, whose start-up latency is longer than the
transfer of these few MB.  q and the new K/V rows come one of two ways, each
bucket holding a graph for both: when the caller's tensors are page-locked,
the kernels read them where they are, taking the three addresses from a pinned
array (the decode options' ``operands``) rewritten each step; otherwise they
are copied into the pinned staging and the kernels read them there.  With ``zero_copy=False`` the
graph holds a host-to-device copy of the packed inputs, the fused call on
device buffers and a device-to-host copy of the output.  A step's host side is
one native call (``pa_stage_decode_step``: metadata rows, padding, shared-prefix
groups, the addresses of the caller's buffers) and one ``cuGraphLaunch``.  Argument marshalling only:
every step of the path runs in the library's kernels.
"""

from __future__ import annotations

import bisect
import ctypes

import torch

from . import (_fp8_pool, _FP8_POOL, _lib, DecodeOptions, DecodeStaging, PagedAttentionError,
               PrefixGroups, STAGE_DERIVE_GROUPS, STAGE_KEEP_GROUPS, STAGE_NO_GROUPS, decode_fp8_workspace_bytes,
               decode_workspace_bytes, store_decode, store_decode_fp8)


def graph_batch_sizes(max_batch: int) -> list[int]:
    """Bucket sizes: 1, 2, 4, 8, then multiples of 16 up to ``max_batch`` (and ``max_batch``
    itself, so every batch up to it has a graph)."""
    if max_batch < 1:
        raise ValueError("max_batch must be positive")
    sizes = [b for b in (1, 2, 4, 8) if b <= max_batch] + list(range(16, max_batch + 1, 16))
    if sizes[-1] != max_batch:
        sizes.append(max_batch)
    return sizes


def _align(n: int) -> int:
    return (n + 255) // 256 * 256


_cu_graph_launch = None


def _graph_launch(graph_exec: int, stream: int) -> None:
    """cuGraphLaunch of an instantiated graph on a stream.  torch's ``CUDAGraph.replay`` first
    refreshes the captured random-generator state with two small fill kernels; the runner's
    graphs draw no random numbers, so they are launched directly."""
    global _cu_graph_launch
    if _cu_graph_launch is None:
        f = ctypes.CDLL("libcuda.so.1").cuGraphLaunch
        f.argtypes, f.restype = [ctypes.c_void_p, ctypes.c_void_p], ctypes.c_int
        _cu_graph_launch = f
    rc = _cu_graph_launch(graph_exec, stream)
    if rc != 0:
        raise RuntimeError(f"cuGraphLaunch failed with CUresult {rc}")


def _raw_stream(device_index: int) -> int:
    """The current stream's handle on a device (torch's direct query where it has one)."""
    get = getattr(torch._C, "_cuda_getCurrentRawStream", None)
    if get is not None:
        return get(device_index)
    return torch.cuda.current_stream(device_index).cuda_stream


def _host_i32(t: torch.Tensor) -> torch.Tensor:
    """t as a contiguous host int32 tensor (itself when it already is one)."""
    if t.is_cuda or t.dtype != torch.int32 or not t.is_contiguous():
        t = t.to("cpu", torch.int32).contiguous()
    return t


class DecodeGraphRunner:
    """Fixed buffers and one captured graph per bucket for the fused decode step of one layer.

    ``k_cache`` / ``v_cache``: the layer's pool (16-bit, or E4M3 codes as ``torch.uint8`` /
    ``torch.float8_e4m3fn`` with ``k_scale`` and ``v_scale`` given).  ``dtype``: the type of q,
    the new K/V rows and the output.  ``zero_copy``: the kernels read the step's inputs from, and
    write its output to, the pinned staging (default), or the graph copies them to and from
    device buffers.  ``group_caps``: (groups, members per group, prefix tokens) -- the largest
    shared-prefix groups a step may pass (:class:`PrefixGroups`, 16-bit pools); the graphs are
    captured for them (unused groups are empty and cost a CTA exit each).  Steps are issued on
    the current stream of the pool's device; one runner serves one step at a time.
    """

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, num_q_heads: int, max_batch: int,
                 max_blocks_per_seq: int, scale: float, dtype: torch.dtype = torch.bfloat16,
                 k_scale: float | None = None, v_scale: float | None = None, zero_copy: bool = True,
                 group_caps: tuple[int, int, int] | None = None):
        self.fp8 = k_cache.dtype in _FP8_POOL
        if self.fp8:
            if k_scale is None or v_scale is None:
                raise ValueError("an E4M3 pool needs k_scale and v_scale")
            _fp8_pool(k_cache, v_cache)
        n, bs, hkv, d = k_cache.shape
        self.k_cache, self.v_cache = k_cache, v_cache
        self.num_q_heads, self.num_kv_heads, self.head_dim = num_q_heads, hkv, d
        self.max_blocks = max_blocks_per_seq
        self.scale, self.k_scale, self.v_scale = float(scale), k_scale, v_scale
        self.dtype = dtype
        self.zero_copy = zero_copy
        if group_caps is not None and (self.fp8 or min(group_caps) < 1):
            raise ValueError("group_caps: positive (groups, members, prefix tokens), 16-bit pools only")
        self.group_caps = group_caps
        self.sizes = graph_batch_sizes(max_batch)
        dev = k_cache.device
        esz = torch.empty(0, dtype=dtype).element_size()
        # per-bucket packed layout (the same in pinned host memory and on the device)
        self._layout = {b: self._pack_layout(b, esz) for b in self.sizes}
        self._staged_views, self._staged_out = {}, {}
        in_bytes = max(lay["_bytes"] for lay in self._layout.values())
        out_bytes = max(self.sizes) * num_q_heads * d * esz
        self.host_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
        self.host_out = torch.zeros(out_bytes, dtype=torch.uint8).pin_memory()
        # zero_copy: when the caller's q and new K/V rows are page-locked, the kernels read them
        # where they are, through a pinned array of their three addresses (the decode options'
        # operands) that each step rewrites
        self._qkv_names = ("q", "k_new", "v_new")
        self._operands = None
        if zero_copy:
            self.dev_in = self.dev_out = None
            self._operands = torch.zeros(3, dtype=torch.int64).pin_memory()
        else:
            self.dev_in = torch.zeros(in_bytes, dtype=torch.uint8, device=dev)
            self.dev_out = torch.zeros(out_bytes, dtype=torch.uint8, device=dev)
        ws_fn = decode_fp8_workspace_bytes if self.fp8 else decode_workspace_bytes
        if group_caps is not None:
            ws = max(decode_workspace_bytes(b, num_q_heads, hkv, d, max_blocks_per_seq, bs, self._options(b, None))
                     for b in self.sizes)
        else:
            ws = max(ws_fn(b, num_q_heads, hkv, d, max_blocks_per_seq, bs) for b in self.sizes)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev)
        # per bucket: the pa_decode_staging a step's metadata are written into (one native call)
        self._stagings = {b: self._make_staging(b) for b in self.sizes}
        self._staging_addr = {b: ctypes.addressof(st) for b, st in self._stagings.items()}
        self._sources = (ctypes.c_void_p * 3)()
        self._sources_addr = ctypes.addressof(self._sources)
        self._row_shapes = ((num_q_heads, d), (hkv, d), (hkv, d))  # a row of q, k_new, v_new
        # per bucket: the graph whose kernels read q and the new rows from the pinned staging, and
        # (zero_copy) the one that first pulls them from the caller's page-locked tensors
        self.graphs: dict[int, torch.cuda.CUDAGraph] = {}
        self._inplace_graphs: dict[int, torch.cuda.CUDAGraph] = {}
        self._use_inplace: dict[int, bool] = {}
        self._execs: dict[tuple[int, bool], int] = {}  # (bucket, in place) -> the instantiated graph
        self._device_index = dev.index if dev.index is not None else torch.cuda.current_device()
        self._capture()

    # ------------------------------------------------------------------ layout
    def _pack_layout(self, b: int, esz: int) -> dict:
        hq, hkv, d, mb = self.num_q_heads, self.num_kv_heads, self.head_dim, self.max_blocks
        fields = [("q", (b, hq, d), self.dtype, b * hq * d * esz),
                  ("k_new", (b, hkv, d), self.dtype, b * hkv * d * esz),
                  ("v_new", (b, hkv, d), self.dtype, b * hkv * d * esz),
                  ("slot_mapping", (b,), torch.int32, 4 * b),
                  ("context_lens", (b,), torch.int32, 4 * b),
                  ("block_tables", (b, mb), torch.int32, 4 * b * mb)]
        if self.group_caps is not None:
            ng = self.group_caps[0]
            fields += [("group_offsets", (ng + 1,), torch.int32, 4 * (ng + 1)),
                       ("group_seqs", (b,), torch.int32, 4 * b),
                       ("prefix_lens", (b,), torch.int32, 4 * b)]
        lay, off = {}, 0
        for name, shape, dt, nbytes in fields:
            lay[name] = (off, shape, dt, nbytes)
            off = _align(off + nbytes)
        lay["_bytes"] = off
        return lay

    def _views(self, buf: torch.Tensor, b: int) -> dict:
        out = {}
        for name, val in self._layout[b].items():
            if name == "_bytes":
                continue
            off, shape, dt, nbytes = val
            out[name] = buf[off:off + nbytes].view(dt).view(shape)
        return out

    def _out_view(self, buf: torch.Tensor, b: int) -> torch.Tensor:
        n = b * self.num_q_heads * self.head_dim
        return buf.view(self.dtype)[:n].view(b, self.num_q_heads, self.head_dim)

    def _options(self, b: int, views: dict | None, operands: int = 0) -> DecodeOptions | None:
        """The decode options of bucket b: the staged groups at their captured capacities, and the
        operands array when the kernels read the caller's q and new rows in place."""
        if self.group_caps is None:
            return DecodeOptions(operands=operands) if operands else None
        ng, members, prefix = self.group_caps
        if views is None:  # sizing only
            z = torch.zeros(max(b, ng + 1), dtype=torch.int32)
            return DecodeOptions(groups=PrefixGroups(z[:ng + 1], z[:b], z[:b], members, prefix))
        return DecodeOptions(groups=PrefixGroups(views["group_offsets"], views["group_seqs"], views["prefix_lens"],
                                                 members, prefix), operands=operands)

    # ----------------------------------------------------------------- capture
    def _make_staging(self, b: int) -> DecodeStaging:
        """The pa_decode_staging of bucket b over its pinned views (and the operands array)."""
        h = self._staged(b)
        st = DecodeStaging(rows=b, max_blocks=self.max_blocks, block_size=self.k_cache.shape[1],
                           slot_mapping=h["slot_mapping"].data_ptr(), context_lens=h["context_lens"].data_ptr(),
                           block_tables=h["block_tables"].data_ptr())
        if self.group_caps is not None:
            st.max_groups, st.max_group_size, st.max_prefix_len = self.group_caps
            st.group_offsets = h["group_offsets"].data_ptr()
            st.group_seqs = h["group_seqs"].data_ptr()
            st.prefix_lens = h["prefix_lens"].data_ptr()
        if self.zero_copy:
            st.operands = self._operands.data_ptr()
        return st

    def _launch(self, b: int, inplace: bool = False) -> None:
        lay = self._layout[b]
        operands = 0
        if self.zero_copy:
            v = dict(self._views(self.host_in, b))
            if inplace:
                # the kernels read q and the new rows through the operands array: captured (and
                # warmed up) pointing at the staging's own, valid memory; steps rewrite it
                for i, n in enumerate(self._qkv_names):
                    self._operands[i] = v[n].data_ptr()
                operands = self._operands.data_ptr()
            out = self._out_view(self.host_out, b)
        else:
            self.dev_in[:lay["_bytes"]].copy_(self.host_in[:lay["_bytes"]], non_blocking=True)
            v = self._views(self.dev_in, b)
            out = self._out_view(self.dev_out, b)
        if self.fp8:
            store_decode_fp8(v["k_new"], v["v_new"], v["slot_mapping"], v["q"], self.k_cache, self.v_cache,
                             v["block_tables"], v["context_lens"], self.scale, self.k_scale, self.v_scale,
                             out=out, workspace=self.workspace, operands=operands)
        else:
            store_decode(v["k_new"], v["v_new"], v["slot_mapping"], v["q"], self.k_cache, self.v_cache,
                         v["block_tables"], v["context_lens"], self.scale, out=out, workspace=self.workspace,
                         options=self._options(b, v, operands))
        if not self.zero_copy:
            self._out_view(self.host_out, b).copy_(out, non_blocking=True)

    def _capture(self) -> None:
        # capture with every row padded (slot -1, context 0): no page is read, nothing is stored
        for b in self.sizes:
            h = self._views(self.host_in, b)
            h["slot_mapping"].fill_(-1)
            h["context_lens"].zero_()
            if self.group_caps is not None:  # empty groups, no shared prefix
                h["group_offsets"].zero_()
                h["prefix_lens"].zero_()
        stream = torch.cuda.Stream(device=self.k_cache.device)
        stream.wait_stream(torch.cuda.current_stream(self.k_cache.device))
        modes = (False, True) if self.zero_copy else (False,)
        with torch.cuda.stream(stream):
            for b in self.sizes:  # warm-up: function attributes and tensor maps are set outside capture
                for m in modes:
                    self._launch(b, m)
        stream.synchronize()
        for b in reversed(self.sizes):
            for m in modes:
                g = torch.cuda.CUDAGraph()
                with torch.cuda.graph(g, stream=stream):
                    self._launch(b, m)
                (self._inplace_graphs if m else self.graphs)[b] = g
                self._execs[(b, m)] = g.raw_cuda_graph_exec()
        torch.cuda.current_stream(self.k_cache.device).wait_stream(stream)

    # -------------------------------------------------------------------- step
    def bucket(self, batch: int) -> int:
        i = bisect.bisect_left(self.sizes, batch)
        if i == len(self.sizes):
            raise ValueError(f"batch {batch} exceeds the largest captured size {self.sizes[-1]}")
        return self.sizes[i]

    def host_inputs(self, batch: int) -> dict:
        """Pinned host views of the step inputs for a batch (the bucket's rows; fill the first
        ``batch``, or use :meth:`set_inputs`)."""
        return self._views(self.host_in, self.bucket(batch))

    def _staged(self, b: int) -> dict:
        """The pinned staging views of bucket b (built once: the step path reuses them)."""
        views = self._staged_views.get(b)
        if views is None:
            views = self._staged_views[b] = self._views(self.host_in, b)
        return views

    def set_inputs(self, q, k_new, v_new, slot_mapping, context_lens, block_tables,
                   groups: PrefixGroups | None = None, share_prefixes: bool = False) -> int:
        """Write one step's host tensors into the pinned staging of its bucket and pad the rest
        (slot -1, context length 0; groups past the step's are empty).  The shared-prefix groups
        are ``groups``, or with ``share_prefixes`` derived by ``pa_prefix_groups`` from the staged
        block tables.  The metadata, the groups and the addresses of the caller's buffers go by one
        native call, ``pa_stage_decode_step``.  With ``zero_copy`` and page-locked, contiguous,
        16-byte aligned q / k_new / v_new of the runner's dtype, those three are not copied: the
        next :meth:`replay` reads them where they are, so keep them unchanged until its stream has
        completed (:meth:`step` synchronises).  Returns the bucket size."""
        batch = q.shape[0]
        b = self.bucket(batch)
        if share_prefixes:
            if self.group_caps is None:
                raise ValueError("this runner was built without group_caps")
            mode = STAGE_DERIVE_GROUPS
        elif groups is not None and groups.num_groups:
            if self.group_caps is None:
                raise ValueError("this runner was built without group_caps")
            self._stage_groups(b, batch, groups)
            mode = STAGE_KEEP_GROUPS
        else:
            mode = STAGE_NO_GROUPS
        slot_mapping, context_lens, block_tables = (_host_i32(slot_mapping), _host_i32(context_lens),
                                                    _host_i32(block_tables))
        if (slot_mapping.numel() != batch or context_lens.numel() != batch or block_tables.dim() != 2
                or block_tables.shape[0] != batch):
            raise ValueError(f"slot_mapping {tuple(slot_mapping.shape)}, context_lens {tuple(context_lens.shape)} "
                             f"and block_tables {tuple(block_tables.shape)} must hold {batch} rows")
        dt, shapes = self.dtype, self._row_shapes
        inplace = self.zero_copy and all(t.dtype == dt and t.shape[1:] == shp and t.data_ptr() % 16 == 0
                                         and t.is_contiguous() and t.is_pinned()
                                         for t, shp in zip((q, k_new, v_new), shapes))
        self._use_inplace[b] = inplace
        if inplace:
            # page-locked tensors: the graph reads them where they are
            src = self._sources
            src[0], src[1], src[2] = q.data_ptr(), k_new.data_ptr(), v_new.data_ptr()
            sources = self._sources_addr
        else:
            h = self._staged(b)
            h["q"][:batch].copy_(q)
            h["k_new"][:batch].copy_(k_new)
            h["v_new"][:batch].copy_(v_new)
            sources = None
        rc = _lib.pa_stage_decode_step(self._staging_addr[b], batch, slot_mapping.data_ptr(),
                                       context_lens.data_ptr(), block_tables.data_ptr(), block_tables.shape[1],
                                       mode, sources)
        if rc != 0:
            raise PagedAttentionError("pa_stage_decode_step", rc)
        return b

    def _stage_groups(self, b: int, batch: int, groups: PrefixGroups) -> None:
        """Caller-given groups into bucket b's staged group fields, unused entries empty."""
        ng, members, prefix = self.group_caps
        if groups.num_groups > ng or groups.max_group_size > members or groups.max_prefix_len > prefix:
            raise ValueError(f"groups ({groups.num_groups}, {groups.max_group_size}, {groups.max_prefix_len}) "
                             f"exceed the captured capacities {self.group_caps}")
        h = self._staged(b)
        g = groups.num_groups
        off = groups.group_offsets
        h["group_offsets"][:g + 1].copy_(off)
        h["group_offsets"][g + 1:].fill_(int(off[g]))
        n = int(off[g])
        h["group_seqs"][:n].copy_(groups.group_seqs[:n])
        h["prefix_lens"].zero_()
        h["prefix_lens"][:batch].copy_(groups.prefix_lens[:batch])

    def replay(self, batch: int) -> torch.Tensor:
        """Replay the bucket's graph (inputs from the pinned staging) on the current stream; the
        returned pinned host view of the output is valid once that stream has synchronised."""
        b = self.bucket(batch)
        _graph_launch(self._execs[(b, self._use_inplace.get(b, False))], _raw_stream(self._device_index))
        out = self._staged_out.get(batch)
        if out is None:  # the first `batch` rows of the bucket's output, one view per batch size
            out = self._staged_out[batch] = self._out_view(self.host_out, b)[:batch]
        return out

    def step(self, q, k_new, v_new, slot_mapping, context_lens, block_tables,
             groups: PrefixGroups | None = None, share_prefixes: bool = False) -> torch.Tensor:
        """One decode step from host tensors to the host output [batch, H_q, D] (synchronises);
        groups as :meth:`set_inputs`."""
        self.set_inputs(q, k_new, v_new, slot_mapping, context_lens, block_tables, groups, share_prefixes)
        out = self.replay(q.shape[0])
        torch.cuda.current_stream(self.k_cache.device).synchronize()
        return out

    def h2d_bytes(self, batch: int) -> int:
        return self._layout[self.bucket(batch)]["_bytes"]

    def d2h_bytes(self, batch: int) -> int:
        return self.bucket(batch) * self.num_q_heads * self.head_dim * torch.empty(0, dtype=self.dtype).element_size()


__all__ = ["DecodeGraphRunner", "graph_batch_sizes"]
