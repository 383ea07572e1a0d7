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
``pa_store_decode_fp8`` over an E4M3 pool) with its small per-step operands in
pinned host memory: the kernels read q, the new K/V rows, the slot mapping,
context lengths and block tables from the pinned staging and write the output
into pinned memory directly over the CPU-GPU link (NVLink-C2C on a Grace-based
GB300), so the step has no copy-engine transfer, whose start-up latency is
longer than the transfer of these few hundred KB.  With ``zero_copy=False``
the graph holds a host-to-device copy of the packed inputs, the fused call on
device buffers and a device-to-host copy of the output.  Argument marshalling
only: every step of the path runs in the library's kernels.
"""

from __future__ import annotations

import torch

from . import (_fp8_pool, _FP8_POOL, decode_fp8_workspace_bytes, decode_workspace_bytes, store_decode,
               store_decode_fp8)


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


class DecodeGraphRunner:
    """Fixed buffers and one captured graph per bucket for the fused decode step of one layer.

    ``k_cache`` / ``v_cache``: the layer's pool (16-bit, or E4M3 codes as ``torch.uint8`` /
    ``torch.float8_e4m3fn`` with ``k_scale`` and ``v_scale`` given).  ``dtype``: the type of q,
    the new K/V rows and the output.  ``zero_copy``: the kernels read the step's inputs from, and
    write its output to, the pinned staging (default), or the graph copies them to and from
    device buffers.  Steps are issued on the current stream of the pool's device; one runner
    serves one step at a time.
    """

    def __init__(self, k_cache: torch.Tensor, v_cache: torch.Tensor, num_q_heads: int, max_batch: int,
                 max_blocks_per_seq: int, scale: float, dtype: torch.dtype = torch.bfloat16,
                 k_scale: float | None = None, v_scale: float | None = None, zero_copy: bool = True):
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
        self.sizes = graph_batch_sizes(max_batch)
        dev = k_cache.device
        esz = torch.empty(0, dtype=dtype).element_size()
        # per-bucket packed layout (the same in pinned host memory and on the device)
        self._layout = {b: self._pack_layout(b, esz) for b in self.sizes}
        in_bytes = max(lay["_bytes"] for lay in self._layout.values())
        out_bytes = max(self.sizes) * num_q_heads * d * esz
        self.host_in = torch.zeros(in_bytes, dtype=torch.uint8).pin_memory()
        self.host_out = torch.zeros(out_bytes, dtype=torch.uint8).pin_memory()
        if zero_copy:
            self.dev_in = self.dev_out = None
        else:
            self.dev_in = torch.zeros(in_bytes, dtype=torch.uint8, device=dev)
            self.dev_out = torch.zeros(out_bytes, dtype=torch.uint8, device=dev)
        ws_fn = decode_fp8_workspace_bytes if self.fp8 else decode_workspace_bytes
        ws = max(ws_fn(b, num_q_heads, hkv, d, max_blocks_per_seq, bs) for b in self.sizes)
        self.workspace = torch.zeros(max(ws, 256), dtype=torch.uint8, device=dev)
        self.graphs: dict[int, torch.cuda.CUDAGraph] = {}
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

    # ----------------------------------------------------------------- capture
    def _launch(self, b: int) -> None:
        lay = self._layout[b]
        if self.zero_copy:
            v = self._views(self.host_in, b)
            out = self._out_view(self.host_out, b)
        else:
            self.dev_in[:lay["_bytes"]].copy_(self.host_in[:lay["_bytes"]], non_blocking=True)
            v = self._views(self.dev_in, b)
            out = self._out_view(self.dev_out, b)
        if self.fp8:
            store_decode_fp8(v["k_new"], v["v_new"], v["slot_mapping"], v["q"], self.k_cache, self.v_cache,
                             v["block_tables"], v["context_lens"], self.scale, self.k_scale, self.v_scale,
                             out=out, workspace=self.workspace)
        else:
            store_decode(v["k_new"], v["v_new"], v["slot_mapping"], v["q"], self.k_cache, self.v_cache,
                         v["block_tables"], v["context_lens"], self.scale, out=out, workspace=self.workspace)
        if not self.zero_copy:
            self._out_view(self.host_out, b).copy_(out, non_blocking=True)

    def _capture(self) -> None:
        # capture with every row padded (slot -1, context 0): no page is read, nothing is stored
        for b in self.sizes:
            h = self._views(self.host_in, b)
            h["slot_mapping"].fill_(-1)
            h["context_lens"].zero_()
        stream = torch.cuda.Stream(device=self.k_cache.device)
        stream.wait_stream(torch.cuda.current_stream(self.k_cache.device))
        with torch.cuda.stream(stream):
            for b in self.sizes:  # warm-up: function attributes and tensor maps are set outside capture
                self._launch(b)
        stream.synchronize()
        for b in reversed(self.sizes):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                self._launch(b)
            self.graphs[b] = g
        torch.cuda.current_stream(self.k_cache.device).wait_stream(stream)

    # -------------------------------------------------------------------- step
    def bucket(self, batch: int) -> int:
        for b in self.sizes:
            if b >= batch:
                return b
        raise ValueError(f"batch {batch} exceeds the largest captured size {self.sizes[-1]}")

    def host_inputs(self, batch: int) -> dict:
        """Pinned host views of the step inputs for a batch (the bucket's rows; fill the first
        ``batch``, or use :meth:`set_inputs`)."""
        return self._views(self.host_in, self.bucket(batch))

    def set_inputs(self, q, k_new, v_new, slot_mapping, context_lens, block_tables) -> int:
        """Copy one step's host tensors into the pinned staging of its bucket and pad the rest
        (slot -1, context length 0).  Returns the bucket size."""
        batch = q.shape[0]
        b = self.bucket(batch)
        h = self._views(self.host_in, b)
        h["q"][:batch].copy_(q)
        h["k_new"][:batch].copy_(k_new)
        h["v_new"][:batch].copy_(v_new)
        h["slot_mapping"].fill_(-1)
        h["slot_mapping"][:batch].copy_(slot_mapping)
        h["context_lens"].zero_()
        h["context_lens"][:batch].copy_(context_lens)
        h["block_tables"][:batch, :block_tables.shape[1]].copy_(block_tables)
        return b

    def replay(self, batch: int) -> torch.Tensor:
        """Replay the bucket's graph (inputs from the pinned staging) on the current stream; the
        returned pinned host view of the output is valid once that stream has synchronised."""
        b = self.bucket(batch)
        self.graphs[b].replay()
        return self._out_view(self.host_out, b)[:batch]

    def step(self, q, k_new, v_new, slot_mapping, context_lens, block_tables) -> torch.Tensor:
        """One decode step from host tensors to the host output [batch, H_q, D] (synchronises)."""
        self.set_inputs(q, k_new, v_new, slot_mapping, context_lens, block_tables)
        out = self.replay(q.shape[0])
        torch.cuda.current_stream(self.k_cache.device).synchronize()
        return out

    def h2d_bytes(self, batch: int) -> int:
        return self._layout[self.bucket(batch)]["_bytes"]

    def d2h_bytes(self, batch: int) -> int:
        return self.bucket(batch) * self.num_q_heads * self.head_dim * torch.empty(0, dtype=self.dtype).element_size()


__all__ = ["DecodeGraphRunner", "graph_batch_sizes"]
