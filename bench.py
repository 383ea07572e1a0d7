#!/usr/bin/env python3
"""Benchmark of the paged-KV hot path on GB300.

One step = one pass of the layer's hot path over one batch of synthetic input
resident in HBM: the store of the step's new K/V rows, then the attention
call(s) of that step (decode; the mixed chunked-prefill workload also runs
the chunked prefill).  Every decode workload reads more than 4x the 129 MB L2
of KV per step, streamed in the same order each step, so each step starts cold
without any flush; a workload with less than twice the L2 of KV is flushed
between steps by reading a 256 MB buffer, outside the timed events.  (A write
flush leaves the L2 full of dirty lines whose write-back then lands inside the
next step, an artefact a real multi-layer step does not have.)

Prints ONE JSON line.  The headline workload (default: the Qwen3-8B-like
decode whose sequences share a 512-token prefix in groups of 8, the largest
decode workload) gives ``value`` = K+V bytes DRAM must supply per step (each
physical page once) / step time; ``value_logical`` counts every sequence's
context.  Unless ``--no-configs``, the same run then times every other
workload (tiny decode, the Qwen3-0.6B-like decode over 16-bit and E4M3 pools,
long-context decode, the mixed chunked-prefill step, the 16384-token store
and the sampler) and reports each under ``configs``, with its own roofline,
clocks and CPU baselines.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--no-configs]
  python bench.py --impl reference ...   # the CPU oracle, timed on the host

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path needs no exchange); the step time is the max over ranks.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

METRIC = "paged decode KV GB/s (% of GB300 HBM peak) and decode tokens/s on 1 GPU"
UNIT = "GB/s"
L2_FLUSH_BYTES = 256 << 20
L2_BYTES = 129 << 20
NOMINAL_HBM_GBS = 7900.0  # GB300 HBM3e, nominal (the measured copy peak is the roofline's denominator)
# GPU-side delay queued before each timed step (outside its events) so that the
# host has enqueued the whole step before the GPU reaches it: the events then
# time the kernels, not the host's launch latency.
PRE_STEP_SPIN_CYCLES = 400_000
DEFAULT_WORKLOAD = "qwen3_8b_shared_decode"
# the other workloads a default run reports under "configs", in this order
# workloads whose sequences share prefix pages: decoded with their shared-prefix groups
SHARED_PREFIX_WORKLOADS = {"qwen3_8b_shared_decode"}
SUB_CONFIGS = ["tiny_decode", "qwen3_0p6b_decode", "long_context_decode", "mixed_chunked_prefill",
               "qwen3_0p6b_decode_fp8", "store_stress", "sampler_qwen3_vocab"]

# DRAM bytes (read + write) of the dominant kernel per launch, from one ncu
# capture of the current kernels on that workload; a workload missing here
# reports null.
TRAFFIC_PER_CALL = {
    "qwen3_0p6b_decode": 575_843_072 + 4_158_720,       # decode_partition_kernel (store fused)
    "qwen3_0p6b_decode_fp8": 288_197_120 + 4_085_248,   # decode_partition_kernel, E4M3 pool (store fused)
    "long_context_decode": 536_962_560 + 3_218_944,     # decode_partition_kernel (store fused)
    # both grids of the step with shared-prefix groups: decode_partition_kernel (sequences; store fused)
    # + decode_prefix_kernel (each group's shared pages once)
    "qwen3_8b_shared_decode": 805_121_536 + 2_861_056 + 69_261_056 + 66_304,
}
PREFILL_TRAFFIC_PER_CALL = {"mixed_chunked_prefill": 126_953_728 + 13_033_728}  # prefill_kernel (ncu, current code)
# store_kv_kernel on store_stress: DRAM read + write inside the launch (the L2 holds most written
# rows as dirty lines until after the launch, so this is below the algorithmic 134,217,728 B)
STORE_TRAFFIC_PER_CALL = 67_182_848 + 15_672_576

WORKLOAD_CONFIG = {
    "tiny_decode": dict(batch=4, context="{1,17,100,255}", H_q=4, H_kv=2, D=64, block_size=16, dtype="fp16"),
    "qwen3_0p6b_decode": dict(batch=64, context="U[128,4096]", H_q=16, H_kv=8, D=128, block_size=256,
                              dtype="bf16", pool="1.25x need, shuffled"),
    "qwen3_8b_shared_decode": dict(batch=256, context="U[513,2048]", H_q=32, H_kv=8, D=128, block_size=16,
                                   dtype="bf16", sharing="groups of 8 share a 512-token prefix"),
    "long_context_decode": dict(batch=4, context="32768", H_q=32, H_kv=8, D=128, block_size=256, dtype="bf16",
                                pool="600 blocks, shuffled"),
    "mixed_chunked_prefill": dict(batch=128, prefill="8 x 512-token chunks over prefixes U[0,3584]",
                                  decode="120 sequences, context U[256,4096]", H_q=32, H_kv=8, D=128,
                                  block_size=256, dtype="bf16"),
    "qwen3_0p6b_decode_fp8": dict(batch=64, context="U[128,4096]", H_q=16, H_kv=8, D=128, block_size=256,
                                  dtype="e4m3 KV (per-tensor scales), bf16 q/out", pool="1.25x need, shuffled"),
    "store_stress": dict(tokens=16384, H_kv=8, D=128, block_size=256, dtype="bf16",
                         slots="distinct random slots of a 1.25x pool"),
    "sampler_qwen3_vocab": dict(batch=64, vocab=151936, dtype="bf16", logits="3 * N(0,1)",
                                temperature="U[0.5, 1.5]", noise="in-kernel Philox4x32-10, new offset per step"),
}
SAMPLER_METRIC = "temperature-sampling logits GB/s and rows/s on 1 GPU"
STORE_METRIC = "slot-mapped KV store GB/s (read + write) on 1 GPU"
# Warp instructions one pa_sample launch executes on the sampler workload (ncu
# smsp__inst_executed.sum of sample_kernel on this workload): the
# kernel is issue-bound (Philox4x32-10 and two accurate logarithms per vocabulary entry;
# 36 warp instructions per entry).
SAMPLER_INSTRUCTIONS_PER_CALL = 10_966_336
SAMPLER_TRAFFIC_PER_CALL = 19_469_824  # sample_kernel DRAM read + write (ncu, one launch)
ISSUE_PER_SM_PER_CLK = 4  # warp instructions: four schedulers per SM


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOAD_CONFIG))
    ap.add_argument("--cpu-seconds", type=float, default=6.0,
                    help="budget of the single-threaded oracle baseline (headline workload)")
    ap.add_argument("--cpu-all-seconds", type=float, default=3.0,
                    help="budget of the all-core (OpenMP) oracle baseline (headline workload)")
    ap.add_argument("--sub-cpu-seconds", type=float, default=2.0,
                    help="budget of each oracle baseline of the other workloads")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="time the chosen workload only")
    ap.add_argument("--split-sms", type=int, default=88,
                    help="mixed chunked-prefill step: SMs of the prefill's partition (0: no SM split)")
    ap.add_argument("--unfused", action="store_true",
                    help="decode workloads: time pa_store_kv + pa_decode as two calls instead of pa_store_decode")
    return ap.parse_args()


def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except OSError:
        return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


# ----------------------------------------------------------------- clocks

class ClockSampler:
    """nvidia-smi clock / throttle samples of this process's GPU while running."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device: int):
        self.uuid = None
        try:
            self.uuid = str(torch.cuda.get_device_properties(device).uuid)
        except Exception:
            pass
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.5)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [r.split(", ") for r in out.strip().splitlines() if r.count(",") >= 8]
        if self.uuid:
            mine = [r for r in rows if self.uuid in r[0]]
            rows = mine or rows
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({n for r in rows for n, v in zip(names, r[5:9]) if v.strip() == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


# --------------------------------------------------------------- workloads

_INPUTS: dict = {}


def workload_inputs(name: str):
    """The workload's seeded synthetic inputs, generated once per run (the timed device
    copies, the end-to-end path and the CPU baselines all read the same objects, which
    nothing mutates: every consumer copies what it writes)."""
    if name not in _INPUTS:
        from tests import inputs
        _INPUTS[name] = inputs.WORKLOADS[name]()
    return _INPUTS[name]

class L2Flush:
    """Evicts the L2 between timed steps by READING a 256 MB buffer (a sum into one float):
    a write flush would leave ~129 MB of dirty lines whose write-back lands in the next
    timed step; read lines are clean, and the previous step's dirty lines are written back
    during the flush, outside the events."""

    def __init__(self, dev: torch.device, enabled: bool = True):
        self.buf = torch.ones(L2_FLUSH_BYTES // 4 if enabled else 1, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)
        self.enabled = enabled

    def __call__(self):
        if self.enabled:
            torch.sum(self.buf, dim=0, out=self.out)


def pack_inputs(host: dict, dev: torch.device):
    """A step's inputs in one device buffer (each tensor 256-byte aligned), as a
    caller stages them for a single host-to-device copy.  Returns the device
    buffer, typed views into it keyed like `host`, and the layout."""
    layout, off = {}, 0
    for k, v in host.items():
        nb = v.numel() * v.element_size()
        layout[k] = (off, nb)
        off = (off + nb + 255) // 256 * 256
    buf = torch.empty(off, dtype=torch.uint8, device=dev)
    views = {}
    for k, v in host.items():
        o, nb = layout[k]
        views[k] = buf[o:o + nb].view(v.dtype).view(v.shape)
        views[k].copy_(v.to(dev))
    return buf, views, layout


def pinned_inputs(host: dict, layout: dict, nbytes: int) -> torch.Tensor:
    """The same layout in pinned host memory."""
    buf = torch.zeros(nbytes, dtype=torch.uint8).pin_memory()
    for k, v in host.items():
        o, nb = layout[k]
        buf[o:o + nb].view(v.dtype).view(v.shape).copy_(v)
    return buf


class DecodeWorkload:
    """A decode step (store of one token per sequence + paged decode) with
    all inputs resident on the device."""

    groups = None    # shared-prefix groups (host), for workloads whose sequences share pages
    options = None   # the decode options carrying them (device)

    def __init__(self, name: str, dev: torch.device, fused: bool = True):
        import paged_kv_cache_bs_gb300 as pa
        self.pa = pa
        self.name = name
        self.st = st = workload_inputs(name)
        p = st.pool
        self.dev = dev
        self.kc, self.vc = p.k_cache.to(dev), p.v_cache.to(dev)
        self.host = {"q": st.q, "k_new": st.k_new, "v_new": st.v_new, "slot_mapping": st.slot_mapping,
                     "block_tables": st.block_tables, "context_lens": st.context_lens}
        # sequences sharing prefix pages: their groups, derived on the host from the block tables
        # (pa_prefix_groups), are one more input of the step, and each shared page is read once
        self.groups = None
        if name in SHARED_PREFIX_WORKLOADS:
            from paged_kv_cache_bs_gb300.block_manager import prefix_groups
            self.groups = prefix_groups(st.block_tables, st.context_lens, p.block_size)
            self.host.update(group_offsets=self.groups.group_offsets, group_seqs=self.groups.group_seqs,
                             prefix_lens=self.groups.prefix_lens)
        self.inputs, self.d, self.layout = pack_inputs(self.host, dev)
        self.options = None
        if self.groups is not None:
            g = self.groups
            self.options = pa.DecodeOptions(groups=pa.PrefixGroups(self.d["group_offsets"], self.d["group_seqs"],
                                                                   self.d["prefix_lens"], g.max_group_size,
                                                                   g.max_prefix_len))
        self.out = torch.empty_like(self.d["q"])
        self.ws = pa.alloc_decode_workspace(self.d["q"], self.kc, self.d["block_tables"], self.options)
        self.kv_bytes = st.kv_bytes()
        # each physical row counted once (differs when sequences share prefix pages)
        self.kv_unique_bytes = st.unique_kv_bytes() if name == "qwen3_8b_shared_decode" else self.kv_bytes
        self.batch = st.batch
        row = p.num_kv_heads * p.head_dim * st.q.element_size()
        self.store_bytes = 2 * 2 * int((st.slot_mapping >= 0).sum()) * row   # k and v, read + write
        self.prefill_flops = 0
        self.fused = fused
        if fused:   # one call: pa_store_decode (store fused into the partition kernel) + merge kernel
            # (with shared prefixes: the prefix grid, then the sequences' grid, which merges)
            self.launches_per_step = 2
            self.phases = [("store+decode", self.store_and_attend)]
        else:
            self.launches_per_step = 3   # store, decode partitions, log-sum-exp merge
            self.phases = [("store", self.store), ("decode", self.attend)]

    def store(self):
        d = self.d
        self.pa.store_kv(d["k_new"], d["v_new"], self.kc, self.vc, d["slot_mapping"])

    def attend(self):
        d = self.d
        self.pa.decode(d["q"], self.kc, self.vc, d["block_tables"], d["context_lens"], self.st.scale,
                       out=self.out, workspace=self.ws, options=self.options)

    def store_and_attend(self):
        d = self.d
        self.pa.store_decode(d["k_new"], d["v_new"], d["slot_mapping"], d["q"], self.kc, self.vc, d["block_tables"],
                             d["context_lens"], self.st.scale, out=self.out, workspace=self.ws, options=self.options)

    e2e_path = ("one packed H2D copy of the step's inputs from pinned memory, the step's calls, "
                "D2H of the output, stream sync; host wall clock")

    def make_runner(self, zero_copy: bool):
        from paged_kv_cache_bs_gb300.graphs import DecodeGraphRunner
        st, fs, g = self.st, getattr(self, "fs", None), getattr(self, "groups", None)
        caps = (g.num_groups, g.max_group_size, g.max_prefix_len) if g is not None else None
        return DecodeGraphRunner(self.kc, self.vc, st.num_q_heads, st.batch, st.block_tables.shape[1],
                                 st.scale, st.q.dtype, k_scale=fs.k_scale if fs else None,
                                 v_scale=fs.v_scale if fs else None, zero_copy=zero_copy, group_caps=caps)

    @staticmethod
    def runner_args(st):
        return st.q, st.k_new, st.v_new, st.slot_mapping, st.context_lens, st.block_tables

    def runner_step(self, runner, args):
        """DecodeGraphRunner.step from a step's host tensors; for workloads that share prefix
        pages the runner derives the groups from the staged block tables (pa_prefix_groups),
        every step, as a caller's step would."""
        return runner.step(*args, share_prefixes=self.groups is not None)

    def e2e_buffers(self):
        if self.fused:
            # the engine's decode path: one CUDA graph per padded batch size holding the fused store +
            # decode (captured here, untimed); a step is DecodeGraphRunner.step() from the caller's host
            # tensors, alternating between this step and the next one over the same pool
            from tests import inputs
            st = self.st
            self.runner = self.make_runner(zero_copy=True)
            # the caller's step inputs in page-locked host memory (allocated once, outside the timing)
            pin = lambda args: tuple(t.contiguous().pin_memory() for t in args)  # noqa: E731
            self.e2e_inputs = [pin(self.runner_args(st)), pin(self.runner_args(inputs.next_decode_step(st, seed=4242)))]
            self.e2e_path = ("DecodeGraphRunner.step() from the caller's page-locked host tensors, alternating two "
                             "seeded decode steps over the same pool: slot mapping, context lengths and block tables "
                             "written into the pinned staging by one native call (pa_stage_decode_step, C++), "
                             "CUDA-graph replay of the fused store + decode, whose kernels read q and the new K/V "
                             "rows from the caller's tensors over NVLink-C2C (their addresses in a pinned operands "
                             "array the same call writes) and write the output into pinned host memory, stream "
                             "sync; host wall "
                             "clock" + ("; the shared-prefix groups derived from the staged block tables "
                                        "inside that call every step" if self.groups is not None else ""))
            return None, None, self.runner.h2d_bytes(st.batch), self.runner.d2h_bytes(st.batch)
        pinned = pinned_inputs(self.host, self.layout, self.inputs.numel())
        out_host = torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()
        return pinned, out_host, pinned.numel(), out_host.numel() * out_host.element_size()

    def e2e_step(self, pinned, out_host, i: int = 0):
        if self.fused:
            self.runner_step(self.runner, self.e2e_inputs[i % 2])
            return
        self.inputs.copy_(pinned, non_blocking=True)   # the step's inputs, one copy
        for _, fn in self.phases:
            fn()
        out_host.copy_(self.out, non_blocking=True)


class Fp8DecodeWorkload(DecodeWorkload):
    """A decode step over an E4M3 pool: pa_store_decode_fp8 (the quantising store of one
    token per sequence fused into the split-K partition kernel, + merge), or with
    fused=False pa_store_kv_fp8 then pa_decode_fp8."""

    def __init__(self, name: str, dev: torch.device, fused: bool = True):
        import paged_kv_cache_bs_gb300 as pa
        self.pa = pa
        self.name = name
        fs = workload_inputs(name)
        self.fs, self.st = fs, fs.step
        st = fs.step
        p = st.pool
        self.dev = dev
        self.kc, self.vc = fs.k_cache.to(dev), fs.v_cache.to(dev)
        self.host = {"q": st.q, "k_new": st.k_new, "v_new": st.v_new, "slot_mapping": st.slot_mapping,
                     "block_tables": st.block_tables, "context_lens": st.context_lens}
        self.inputs, self.d, self.layout = pack_inputs(self.host, dev)
        self.out = torch.empty_like(self.d["q"])
        nbytes = pa.decode_fp8_workspace_bytes(st.batch, st.num_q_heads, p.num_kv_heads, p.head_dim,
                                               st.block_tables.shape[1], p.block_size)
        self.ws = torch.empty(max(nbytes, 256), dtype=torch.uint8, device=dev)
        self.kv_bytes = fs.kv_bytes()
        self.kv_unique_bytes = self.kv_bytes
        self.batch = st.batch
        row = p.num_kv_heads * p.head_dim
        # k and v: 16-bit rows read, one-byte codes written
        self.store_bytes = 2 * int((st.slot_mapping >= 0).sum()) * row * (st.q.element_size() + 1)
        self.prefill_flops = 0
        self.fused = fused
        if fused:
            self.launches_per_step = 2   # partitions (with the store) + log-sum-exp merge
            self.phases = [("store+decode", self.store_and_attend)]
        else:
            self.launches_per_step = 3   # quantising store, decode partitions, log-sum-exp merge
            self.phases = [("store", self.store), ("decode", self.attend)]

    def store(self):
        d, fs = self.d, self.fs
        self.pa.store_kv_fp8(d["k_new"], d["v_new"], self.kc, self.vc, d["slot_mapping"], fs.k_scale, fs.v_scale)

    def attend(self):
        d, fs = self.d, self.fs
        self.pa.decode_fp8(d["q"], self.kc, self.vc, d["block_tables"], d["context_lens"], self.st.scale,
                           fs.k_scale, fs.v_scale, out=self.out, workspace=self.ws)

    def store_and_attend(self):
        d, fs = self.d, self.fs
        self.pa.store_decode_fp8(d["k_new"], d["v_new"], d["slot_mapping"], d["q"], self.kc, self.vc,
                                 d["block_tables"], d["context_lens"], self.st.scale, fs.k_scale, fs.v_scale,
                                 out=self.out, workspace=self.ws)


class MixedWorkload(DecodeWorkload):
    """A mixed chunked-prefill step over one pool: store of every new token
    (prefill chunks and decode tokens), causal prefill of the chunks over
    their cached prefixes, decode of the other sequences."""

    def __init__(self, name: str, dev: torch.device, split_sms: int = 0):
        import paged_kv_cache_bs_gb300 as pa
        self.pa = pa
        self.name = name
        # the whole step in one call, the prefill and the decode side by side on disjoint SM sets
        self.split = pa.SmSplit(split_sms) if split_sms else None
        m = workload_inputs(name)
        self.st = st = m.decode
        pf = m.prefill
        self.pf = pf
        p = pf.pool
        self.dev = dev
        self.kc, self.vc = p.k_cache.to(dev), p.v_cache.to(dev)
        self.host = {"q": st.q, "block_tables": st.block_tables, "context_lens": st.context_lens,
                     "k_all": m.k_new, "v_all": m.v_new, "slot_all": m.slot_mapping, "pq": pf.q,
                     "cu_q": pf.cu_seqlens_q, "cu_k": pf.cu_seqlens_k, "pbt": pf.block_tables}
        self.inputs, self.d, self.layout = pack_inputs(self.host, dev)
        self.out = torch.empty_like(self.d["q"])
        self.pout = torch.empty_like(self.d["pq"])
        self.ws = pa.alloc_decode_workspace(self.d["q"], self.kc, self.d["block_tables"])
        self.kv_bytes = st.kv_bytes()
        self.kv_unique_bytes = self.kv_bytes
        self.batch = st.batch + (pf.cu_seqlens_q.numel() - 1)
        row = p.num_kv_heads * p.head_dim * st.q.element_size()
        self.store_bytes = 2 * 2 * int((m.slot_mapping >= 0).sum()) * row
        # store, prefill, decode partitions (960 (sequence, kv head) pairs fill two waves: no split-K,
        # so no merge launch)
        self.launches_per_step = 3
        self.phases = [("store", self.store), ("prefill", self.prefill), ("decode", self.attend)]
        self.prefill_flops = pf.flops()
        self.fused = False

    def store(self):
        d = self.d
        self.pa.store_kv(d["k_all"], d["v_all"], self.kc, self.vc, d["slot_all"])

    def prefill(self):
        d, pf = self.d, self.pf
        self.pa.prefill_paged(d["pq"], None, None, self.kc, self.vc, d["cu_q"], d["cu_k"], pf.max_seqlen_q,
                              pf.max_seqlen_k, d["pbt"], pf.scale, out=self.pout)

    def split_step(self, prefill_out=None, decode_out=None):
        d, pf = self.d, self.pf
        self.pa.mixed_step(d["k_all"], d["v_all"], d["slot_all"], d["pq"], d["cu_q"], d["cu_k"], pf.max_seqlen_q,
                           pf.max_seqlen_k, d["pbt"], d["q"], d["block_tables"], d["context_lens"], self.kc, self.vc,
                           pf.scale, prefill_out=self.pout if prefill_out is None else prefill_out,
                           decode_out=self.out if decode_out is None else decode_out, workspace=self.ws,
                           split=self.split)

    def e2e_buffers(self):
        pinned = pinned_inputs(self.host, self.layout, self.inputs.numel())
        outs = torch.empty(self.out.numel() + self.pout.numel(), dtype=self.out.dtype).pin_memory()
        if self.split is not None:
            # the outputs come back by copy-engine transfers: the kernels writing the 33.5 MB prefill
            # output into pinned memory themselves took the step from 688 to 1427 us end to end
            self.e2e_path = ("one packed H2D copy of the step's inputs from pinned memory, pa_mixed_step (store, then "
                             f"prefill on {self.split.sms[0]} SMs beside decode on {self.split.sms[1]}), D2H of the "
                             "outputs, stream sync; host wall clock")
        return pinned, outs, pinned.numel(), outs.numel() * outs.element_size()

    def e2e_step(self, pinned, out_host, i: int = 0):
        self.inputs.copy_(pinned, non_blocking=True)   # the step's inputs, one copy
        if self.split is not None:
            self.split_step()
        else:
            for _, fn in self.phases:
                fn()
        n = self.out.numel()
        out_host[:n].copy_(self.out.view(-1), non_blocking=True)
        out_host[n:].copy_(self.pout.view(-1), non_blocking=True)


# ------------------------------------------------------------------ timing

def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    return world, rank, local


def barrier(world, local):
    if world > 1:
        import torch.distributed as dist
        dist.barrier(device_ids=[local]) if dist.get_backend() == "nccl" else dist.barrier()


def max_over_ranks(x: float, world: int, dev) -> float:
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------ CPU baselines

def _decode_part(name: str):
    """The decode step of a workload (the decode rows of the mixed step)."""
    st = workload_inputs(name)
    return st.decode if hasattr(st, "decode") else st


def _oracle_step(name: str):
    """(decode step, fn(b), K + V bytes of one context token): the oracle's store + decode
    of sequence b of the workload."""
    import oracle
    st = _decode_part(name)
    if hasattr(st, "step"):  # E4M3 pool
        fs, st = st, st.step
        kc, vc = fs.k_cache.clone(), fs.v_cache.clone()

        def step(b):
            sl = slice(b, b + 1)
            oracle.store_kv_fp8(st.k_new[sl], st.v_new[sl], kc, vc, st.slot_mapping[sl], fs.k_scale, fs.v_scale)
            oracle.decode_fp8(st.q[sl], kc, vc, st.block_tables[sl], st.context_lens[sl], st.scale, fs.k_scale,
                              fs.v_scale)
        return st, step, 2 * st.pool.num_kv_heads * st.pool.head_dim  # one byte per element
    p = st.pool
    kc, vc = p.k_cache.clone(), p.v_cache.clone()

    def step(b):
        sl = slice(b, b + 1)
        oracle.store_kv(st.k_new[sl], st.v_new[sl], kc, vc, st.slot_mapping[sl])
        oracle.decode(st.q[sl], kc, vc, st.block_tables[sl], st.context_lens[sl], st.scale)
    return st, step, 2 * p.num_kv_heads * p.head_dim * st.q.element_size()


def cpu_baseline(name: str, seconds: float):
    """The oracle as it stands, single-threaded on this host: store + decode of
    the workload's sequences one at a time until the time budget is spent."""
    st, step, row = _oracle_step(name)
    done_bytes, n, t_total = 0, 0, 0.0
    while t_total < seconds:          # whole passes over the batch until the budget is spent
        b = n % st.batch
        t0 = time.perf_counter()
        step(b)
        t_total += time.perf_counter() - t0
        done_bytes += int(st.context_lens[b]) * row
        n += 1
    return {"value": done_bytes / t_total / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"store + decode of {n} sequences (round robin over the {st.batch} of the workload) "
                      f"({done_bytes / 1e6:.1f} MB of KV), single-threaded C oracle, "
                      f"{os.cpu_count()} host cores present"}


def cpu_baseline_all_cores(name: str, seconds: float):
    """The same oracle source built with OpenMP (bit-identical results), on all host cores:
    decode of 8 sequences per call, round robin over the batch, until the budget is spent
    (the store of the step's rows is done once, before the timing)."""
    import oracle
    lib = oracle.load_omp()
    st = _decode_part(name)
    fp8 = hasattr(st, "step")
    if fp8:
        fs, st = st, st.step
        kc, vc = fs.k_cache.clone(), fs.v_cache.clone()
        oracle.store_kv_fp8(st.k_new, st.v_new, kc, vc, st.slot_mapping, fs.k_scale, fs.v_scale)
        row = 2 * st.pool.num_kv_heads * st.pool.head_dim
    else:
        kc, vc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
        oracle.store_kv(st.k_new, st.v_new, kc, vc, st.slot_mapping)
        row = 2 * st.pool.num_kv_heads * st.pool.head_dim * st.q.element_size()
    chunk, B = 8, st.batch
    done_bytes, n, t_total = 0, 0, 0.0
    while t_total < seconds:
        b0 = (n * chunk) % B
        sl = slice(b0, min(b0 + chunk, B))
        t0 = time.perf_counter()
        if fp8:
            oracle.decode_fp8(st.q[sl], kc, vc, st.block_tables[sl], st.context_lens[sl], st.scale, fs.k_scale,
                              fs.v_scale, lib=lib)
        else:
            oracle.decode(st.q[sl], kc, vc, st.block_tables[sl], st.context_lens[sl], st.scale, lib=lib)
        t_total += time.perf_counter() - t0
        done_bytes += int(st.context_lens[sl].sum()) * row
        n += 1
    threads = lib.oracle_num_threads()
    return {"value": done_bytes / t_total / 1e9, "unit": UNIT, "cores": threads, "kind": "oracle (OpenMP build)",
            "sample": f"decode of {n} batches of up to {chunk} sequences (round robin over the {B} of the "
                      f"workload, {done_bytes / 1e6:.1f} MB of KV), {threads} threads over (query head) rows "
                      f"and gathered positions, {os.cpu_count()} host cores present"}


def decode_cpu_baselines(name: str, single_s: float, all_s: float):
    """Single-threaded oracle baseline with the all-core figure beside it."""
    base = cpu_baseline(name, single_s)
    base["all_cores"] = cpu_baseline_all_cores(name, all_s)
    return base


def prefill_cpu_baselines(single_s: float, all_s: float):
    """The oracle's chunked prefill of the mixed workload on the host, in TFLOP/s of the
    kernel's algorithmic work (masked work excluded): single-threaded on 16-row windows
    of the chunks (round robin), and the OpenMP build on whole chunks (round robin)."""
    import oracle
    m = workload_inputs("mixed_chunked_prefill")
    st = m.prefill
    okc, ovc = st.pool.k_cache.clone(), st.pool.v_cache.clone()
    oracle.store_kv(m.k_new, m.v_new, okc, ovc, m.slot_mapping)
    cq, ck = st.cu_seqlens_q.tolist(), st.cu_seqlens_k.tolist()
    S, H, D = len(cq) - 1, st.num_q_heads, st.q.shape[2]

    def window(i, r0, r1, lib=None):
        lq, lk = cq[i + 1] - cq[i], ck[i + 1] - ck[i]
        P = lk - lq
        rows = slice(cq[i] + r0, cq[i] + r1)
        t0 = time.perf_counter()
        oracle.prefill_paged(st.q[rows], st.k_new[rows], st.v_new[rows], okc, ovc,
                             torch.tensor([0, r1 - r0], dtype=torch.int32),
                             torch.tensor([0, P + r1], dtype=torch.int32), st.block_tables[i:i + 1], st.scale,
                             lib=lib)
        dt = time.perf_counter() - t0
        return dt, 4 * D * H * sum(P + r + 1 for r in range(r0, r1))

    out = {}
    for kind, budget in (("single", single_s), ("all", all_s)):
        lib = oracle.load_omp() if kind == "all" else None
        t_total, flops, n = 0.0, 0, 0
        while t_total < budget:
            i = n % S
            lq = cq[i + 1] - cq[i]
            if kind == "single":
                r0 = (16 * (n // S)) % max(lq - 15, 1)
                dt, f = window(i, r0, min(r0 + 16, lq))
            else:
                dt, f = window(i, 0, lq, lib)
            t_total += dt
            flops += f
            n += 1
        out[kind] = (flops / t_total / 1e12, n, flops)
    threads = oracle.load_omp().oracle_num_threads()
    v1, n1, f1 = out["single"]
    va, na, fa = out["all"]
    return {"value": v1, "unit": "TFLOP/s", "cores": 1, "kind": "oracle",
            "sample": f"{n1} 16-row windows of the 8 chunks (round robin), {f1 / 1e9:.1f} GFLOP, single-threaded "
                      f"C oracle, {os.cpu_count()} host cores present",
            "all_cores": {"value": va, "unit": "TFLOP/s", "cores": threads, "kind": "oracle (OpenMP build)",
                          "sample": f"{na} whole 512-row chunks (round robin), {fa / 1e9:.1f} GFLOP, {threads} "
                                    f"threads over (query row, head) rows"}}


def run_reference(args, world, rank):
    """The oracle timed as the reference arm: each step decodes one sequence of
    the workload (round robin) on the host."""
    if rank != 0:
        return
    import oracle
    if args.workload == "store_stress":
        k, v, kc, vc, slots = _store_inputs()
        row = k.shape[1] * k.shape[2] * k.element_size()
        T = k.shape[0]
        for i in range(args.warmup):
            oracle.store_kv(k[i % T:i % T + 1], v[i % T:i % T + 1], kc, vc, slots[i % T:i % T + 1])
        t0 = time.perf_counter()
        for i in range(args.steps):
            j = (args.warmup + i) % T
            oracle.store_kv(k[j:j + 1], v[j:j + 1], kc, vc, slots[j:j + 1])
        dt = time.perf_counter() - t0
        value = 4 * row * args.steps / dt / 1e9
        print(json.dumps({"metric": STORE_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                          "data": "synthetic", "impl": "reference",
                          "config": {"workload": args.workload, **WORKLOAD_CONFIG[args.workload],
                                     "sample": "one token per step"},
                          "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                                           "sample": "one token of the workload stored per step"},
                          "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    if args.workload == "sampler_qwen3_vocab":
        logits, temps = _sampler_inputs()
        g = torch.Generator().manual_seed(13)
        noise = torch.empty(1, logits.shape[1]).exponential_(1, generator=g)
        step_bytes = logits.shape[1] * logits.element_size()
        for i in range(args.warmup):
            oracle.sample(logits[i % 64:i % 64 + 1], temps[i % 64:i % 64 + 1], noise)
        t0 = time.perf_counter()
        for i in range(args.steps):
            b = (args.warmup + i) % logits.shape[0]
            oracle.sample(logits[b:b + 1], temps[b:b + 1], noise)
        dt = time.perf_counter() - t0
        value = args.steps * step_bytes / dt / 1e9
        print(json.dumps({"metric": SAMPLER_METRIC, "value": value, "unit": UNIT, "n_gpus": world,
                          "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps,
                          "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
                          "data": "synthetic", "impl": "reference",
                          "config": {"workload": args.workload, **WORKLOAD_CONFIG[args.workload],
                                     "sample": "one row per step"},
                          "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                                           "sample": "one row of the workload per step"},
                          "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                                  "d2h_bytes_per_step": 0}}), flush=True)
        return
    st, one, row = _oracle_step(args.workload)

    def step(i):
        b = i % st.batch
        one(b)
        return int(st.context_lens[b]) * row

    for i in range(args.warmup):
        step(i)
    nbytes, t0 = 0, time.perf_counter()
    for i in range(args.steps):
        nbytes += step(args.warmup + i)
    dt = time.perf_counter() - t0
    value = nbytes / dt / 1e9
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": dt * 1e3 / args.steps, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": WORKLOAD_CONFIG[args.workload]["dtype"],
            "data": "synthetic", "impl": "reference",
            "config": {"workload": args.workload, **WORKLOAD_CONFIG[args.workload],
                       "sample": "one sequence (round robin) per step"},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
                             "sample": "one sequence of the workload per step, store + decode"},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def _sampler_inputs():
    cfg = WORKLOAD_CONFIG["sampler_qwen3_vocab"]
    g = torch.Generator().manual_seed(9)
    logits = (3 * torch.randn(cfg["batch"], cfg["vocab"], generator=g)).to(torch.bfloat16)
    temps = 0.5 + torch.rand(cfg["batch"], generator=g)
    return logits, temps


def sampler_cpu_baseline(seconds: float):
    """The oracle sampler single-threaded on this host, row by row, with Exp(1) noise drawn by torch."""
    import oracle
    logits, temps = _sampler_inputs()
    g = torch.Generator().manual_seed(11)
    n, t_total = 0, 0.0
    while t_total < seconds:
        b = n % logits.shape[0]
        noise = torch.empty(1, logits.shape[1]).exponential_(1, generator=g)
        t0 = time.perf_counter()
        oracle.sample(logits[b:b + 1], temps[b:b + 1], noise)
        t_total += time.perf_counter() - t0
        n += 1
    nbytes = n * logits.shape[1] * logits.element_size()
    return {"value": nbytes / t_total / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} rows of the workload sampled one at a time (noise drawn outside the timing), "
                      f"single-threaded C oracle (the sampler oracle has no multi-threaded build), "
                      f"{os.cpu_count()} host cores present"}


def measure_sampler(name, args, world, rank, local, cpu_s):
    """pa_sample on 64 rows of a 151936-token vocabulary, in-kernel noise, a new offset every step."""
    import paged_kv_cache_bs_gb300 as pa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    logits_h, temps_h = _sampler_inputs()
    B, V = logits_h.shape
    logits, temps = logits_h.to(dev), temps_h.to(dev)
    tokens = torch.empty(B, dtype=torch.int32, device=dev)
    nbytes = B * V * logits.element_size()
    flush = L2Flush(dev)  # the logits fit in L2
    stream = torch.cuda.current_stream(dev)
    for i in range(args.warmup):
        pa.sample(logits, temps, seed=1, offset=i, out=tokens)
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world, local)
    torch.cuda.synchronize(dev)
    for i in range(K):
        flush()                                            # L2 flushed between steps, outside the events
        torch.cuda._sleep(PRE_STEP_SPIN_CYCLES)
        ev[i][0].record(stream)
        pa.sample(logits, temps, seed=1, offset=args.warmup + i, out=tokens)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, local)
    clk = clocks.stop()
    ms = sum(a.elapsed_time(b) for a, b in ev) / K
    ms_max = max_over_ranks(ms, world, dev)
    # end to end: the logits from pinned host memory (one copy), the call, the tokens back
    pin_l, pin_t, out_h = logits_h.pin_memory(), temps_h.pin_memory(), torch.empty(B, dtype=torch.int32).pin_memory()
    Ke = min(K, 300)
    e2e_s = 0.0
    for i in range(Ke):
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        logits.copy_(pin_l, non_blocking=True)
        temps.copy_(pin_t, non_blocking=True)
        pa.sample(logits, temps, seed=2, offset=i, out=tokens)
        out_h.copy_(tokens, non_blocking=True)
        stream.synchronize()
        e2e_s += time.perf_counter() - t0
    e2e_ms = max_over_ranks(e2e_s * 1e3 / Ke, world, dev)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    sm_mhz = clk.get("sm_mhz") or 2070.0
    sms = torch.cuda.get_device_properties(dev).multi_processor_count
    issue_peak = ISSUE_PER_SM_PER_CLK * sms * sm_mhz * 1e6
    achieved = SAMPLER_INSTRUCTIONS_PER_CALL / (ms / 1e3)
    roof = {"bound": "alu", "kernel": "sample_kernel (Philox4x32-10 + two logf per entry, issue-bound)",
            "achieved": achieved, "peak": issue_peak, "unit": "warp-instr/s", "frac": achieved / issue_peak,
            "peak_source": f"derived: {ISSUE_PER_SM_PER_CLK} warp instructions/clock/SM x {sms} SMs x "
                           f"{sm_mhz:.0f} MHz sampled", "traffic": SAMPLER_TRAFFIC_PER_CALL,
            "hbm_frac": nbytes / (ms / 1e3) / 1e9 / peaks["hbm_gbs"]}
    return {
        "metric": SAMPLER_METRIC, "value": world * nbytes / (ms_max / 1e3) / 1e9, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, **WORKLOAD_CONFIG[name],
                   "l2": "flushed (256 MB read) between steps, outside the timed events",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "rows_per_s": world * B / (ms_max / 1e3),
        "roofline": roof,
        "cpu_baseline": sampler_cpu_baseline(cpu_s) if world == 1 and cpu_s > 0 else None,
        "e2e": {"value": world * nbytes / (e2e_ms / 1e3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": nbytes + B * 4, "d2h_bytes_per_step": B * 4, "ms_per_step": e2e_ms},
        "gpu_launches": K,
        "clocks": clk,
    }


def _store_inputs():
    from tests import inputs
    return inputs.store_stress()


def store_cpu_baseline(seconds: float):
    """The oracle's store single-threaded on this host, token by token."""
    import oracle
    k, v, kc, vc, slots = _store_inputs()
    row = k.shape[1] * k.shape[2] * k.element_size()
    n, t_total = 0, 0.0
    while t_total < seconds:
        i = n % k.shape[0]
        t0 = time.perf_counter()
        oracle.store_kv(k[i:i + 1], v[i:i + 1], kc, vc, slots[i:i + 1])
        t_total += time.perf_counter() - t0
        n += 1
    return {"value": 4 * row * n / t_total / 1e9, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{n} tokens of the workload stored one at a time, single-threaded C oracle (the store "
                      f"oracle has no multi-threaded build), {os.cpu_count()} host cores present"}


def measure_store(name, args, world, rank, local, cpu_s):
    """pa_store_kv of 16384 tokens (the engine's max batched tokens) into distinct random slots."""
    import paged_kv_cache_bs_gb300 as pa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    k_h, v_h, kc_h, vc_h, slots_h = _store_inputs()
    k, v, kc, vc, slots = k_h.to(dev), v_h.to(dev), kc_h.to(dev), vc_h.to(dev), slots_h.to(dev)
    T, row = k.shape[0], k.shape[1] * k.shape[2] * k.element_size()
    nbytes = 2 * 2 * T * row  # K and V rows, read + written
    flush = L2Flush(dev)  # 134 MB of rows: about the L2
    stream = torch.cuda.current_stream(dev)
    for _ in range(args.warmup):
        pa.store_kv(k, v, kc, vc, slots)
    torch.cuda.synchronize(dev)
    K = args.steps
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world, local)
    torch.cuda.synchronize(dev)
    for i in range(K):
        flush()
        torch.cuda._sleep(PRE_STEP_SPIN_CYCLES)
        ev[i][0].record(stream)
        pa.store_kv(k, v, kc, vc, slots)
        ev[i][1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, local)
    clk = clocks.stop()
    times = [a.elapsed_time(b) for a, b in ev]
    ms = sum(times) / K
    ms_max = max_over_ranks(ms, world, dev)
    # end to end: the new rows and slots from pinned host memory, the store, a sync
    pin_k, pin_v, pin_s = k_h.pin_memory(), v_h.pin_memory(), slots_h.pin_memory()
    Ke = min(K, 300)
    e2e_s = 0.0
    for _ in range(Ke):
        flush()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        k.copy_(pin_k, non_blocking=True)
        v.copy_(pin_v, non_blocking=True)
        slots.copy_(pin_s, non_blocking=True)
        pa.store_kv(k, v, kc, vc, slots)
        stream.synchronize()
        e2e_s += time.perf_counter() - t0
    e2e_ms = max_over_ranks(e2e_s * 1e3 / Ke, world, dev)
    if rank != 0:
        return None
    peaks, peak_kind = measured_peaks()
    achieved = nbytes / (ms / 1e3) / 1e9
    return {
        "metric": STORE_METRIC, "value": world * nbytes / (ms_max / 1e3) / 1e9, "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms_max, "ms_per_step_median": statistics.median(times),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": name, **WORKLOAD_CONFIG[name],
                   "l2": "flushed (256 MB read) between steps, outside the timed events",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "tokens_per_s": world * T / (ms_max / 1e3),
        "roofline": {"bound": "hbm", "kernel": "store_kv_kernel (one warp per token, 16-byte vectors)",
                     "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                     "peak_source": f"{peak_kind} (hbm_gbs)", "traffic": STORE_TRAFFIC_PER_CALL},
        "cpu_baseline": store_cpu_baseline(cpu_s) if world == 1 and cpu_s > 0 else None,
        "e2e": {"value": world * nbytes / (e2e_ms / 1e3) / 1e9, "unit": UNIT,
                "h2d_bytes_per_step": 2 * T * row + 4 * T, "d2h_bytes_per_step": 0, "ms_per_step": e2e_ms,
                "path": "H2D copies of the new K/V rows and slots from pinned memory, pa_store_kv, stream sync; "
                        "host wall clock (a store returns nothing to read back)"},
        "gpu_launches": K,
        "clocks": clk,
    }


def measure_attention(name, args, world, rank, local, cpu_s, cpu_all_s):
    """A decode or mixed chunked-prefill workload: the device-resident timed steps, the
    mixed step on SM partitions, the end-to-end step through the public API, the roofline
    of the dominant kernel and the CPU baselines."""
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if name == "mixed_chunked_prefill":
        w = MixedWorkload(name, dev, split_sms=args.split_sms)
    elif name.endswith("_fp8"):
        w = Fp8DecodeWorkload(name, dev, fused=not args.unfused)
    else:
        w = DecodeWorkload(name, dev, fused=not args.unfused)
    flush_needed = w.kv_unique_bytes < 2 * L2_BYTES
    flush = L2Flush(dev, flush_needed)
    stream = torch.cuda.current_stream(dev)

    def between_steps():
        if flush_needed:
            flush()

    for _ in range(args.warmup):
        between_steps()
        for _, fn in w.phases:
            fn()
    torch.cuda.synchronize(dev)

    # ---- device-resident timed region
    K = args.steps
    nph = len(w.phases)
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(nph + 1)] for _ in range(K)]
    clocks = ClockSampler(local)
    clocks.start()
    barrier(world, local)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter()
    for i in range(K):
        between_steps()               # L2 flush (small workloads only), outside the events
        torch.cuda._sleep(PRE_STEP_SPIN_CYCLES)
        ev[i][0].record(stream)
        for j, (_, fn) in enumerate(w.phases):
            fn()
            ev[i][j + 1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world, local)
    t_wall = time.perf_counter() - t_wall
    clk = clocks.stop()
    phase_ms = {pn: sum(e[j].elapsed_time(e[j + 1]) for e in ev) / K for j, (pn, _) in enumerate(w.phases)}
    step_ms = sum(phase_ms.values())
    step_ms_median = statistics.median(e[0].elapsed_time(e[nph]) for e in ev)
    step_ms_max = max_over_ranks(step_ms, world, dev)
    store_ms = phase_ms.get("store")
    dec_ms_avg = phase_ms["decode"] if "decode" in phase_ms else phase_ms["store+decode"]

    # ---- the mixed step as one pa_mixed_step call with its prefill and decode side by side on
    # disjoint SM partitions: this is the step's time; the phases above (one after the other)
    # give each kernel's own rate for its roofline
    split_ms = None
    if getattr(w, "split", None) is not None:
        for _ in range(args.warmup):
            between_steps()
            w.split_step()
        torch.cuda.synchronize(dev)
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(K)]
        barrier(world, local)
        torch.cuda.synchronize(dev)
        for i in range(K):
            between_steps()
            torch.cuda._sleep(PRE_STEP_SPIN_CYCLES)
            evs[i][0].record(stream)
            w.split_step()
            evs[i][1].record(stream)
        torch.cuda.synchronize(dev)
        barrier(world, local)
        split_times = [a.elapsed_time(b) for a, b in evs]
        split_ms = sum(split_times) / K
        step_ms_sequential = step_ms
        step_ms_max = max_over_ranks(split_ms, world, dev)
        step_ms_median = statistics.median(split_times)

    # ---- end to end through the public API, as a caller sees it: host wall clock from the
    # step's inputs in host memory to its result back in host memory, launch overheads and
    # the final sync included.
    pinned, out_host, h2d, d2h = w.e2e_buffers()
    for i in range(args.warmup):
        w.e2e_step(pinned, out_host, i)
    torch.cuda.synchronize(dev)
    Ke = min(K, 500)
    barrier(world, local)
    e2e_s = 0.0
    for i in range(Ke):
        between_steps()
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        w.e2e_step(pinned, out_host, i)
        stream.synchronize()
        e2e_s += time.perf_counter() - t0
    barrier(world, local)
    e2e_ms = max_over_ranks(e2e_s * 1e3 / Ke, world, dev)
    # breakdown of the graph runner's step: the replay alone (inputs already staged), and the
    # step with the graph's copy-engine transfers instead of zero-copy operands
    e2e_replay_ms = e2e_copy_ms = None
    if getattr(w, "runner", None) is not None:
        w.runner_step(w.runner, w.e2e_inputs[0])
        e2e_s = 0.0
        for i in range(Ke):
            between_steps()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            w.runner.replay(w.st.batch)
            stream.synchronize()
            e2e_s += time.perf_counter() - t0
        e2e_replay_ms = max_over_ranks(e2e_s * 1e3 / Ke, world, dev)
        rc = w.make_runner(zero_copy=False)
        for i in range(args.warmup):
            w.runner_step(rc, w.e2e_inputs[i % 2])
        torch.cuda.synchronize(dev)
        e2e_s = 0.0
        for i in range(Ke):
            between_steps()
            torch.cuda.synchronize(dev)
            t0 = time.perf_counter()
            w.runner_step(rc, w.e2e_inputs[i % 2])
            e2e_s += time.perf_counter() - t0
        e2e_copy_ms = max_over_ranks(e2e_s * 1e3 / Ke, world, dev)
        del rc

    peaks, peak_kind = measured_peaks()
    # bytes DRAM must supply per step: each physical page once (pages shared by several
    # sequences are counted once; for unshared workloads this equals the logical KV bytes)
    value = world * w.kv_unique_bytes / (step_ms_max / 1e3) / 1e9
    if rank != 0:
        return None
    cpu = None
    if world == 1 and cpu_s > 0:
        cpu = decode_cpu_baselines(name, cpu_s, cpu_all_s)
    decode_gbs = w.kv_bytes / (dec_ms_avg / 1e3) / 1e9
    unique_gbs = w.kv_unique_bytes / (dec_ms_avg / 1e3) / 1e9
    dominant = max(phase_ms, key=phase_ms.get)
    if dominant == "prefill":
        achieved = w.prefill_flops / (phase_ms["prefill"] / 1e3) / 1e12
        roof = {"bound": "tensor", "kernel": "prefill_kernel (tcgen05, bf16, fp32 accumulate)", "achieved": achieved,
                "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / peaks["bf16_tflops"],
                "peak_source": f"{peak_kind} (bf16_tflops, burst: the kernel is timed by its own events)",
                "traffic": PREFILL_TRAFFIC_PER_CALL.get(name)}
    else:
        f8 = isinstance(w, Fp8DecodeWorkload)
        kern = ("pa_store_decode_fp8 (E4M3 store fused into the split-K partition kernel + merge)"
                if f8 and "store+decode" in phase_ms else
                "pa_decode_fp8 (E4M3 split-K partitions + merge)" if f8 else
                ("pa_store_decode_ex with shared-prefix groups (the groups' shared pages read once by a prefix "
                 "grid; the sequences' grid stores, attends over the private pages and folds in the prefix "
                 "partials)" if w.options is not None else
                 "pa_store_decode (store fused into the split-K partition kernel + merge)")
                if "store+decode" in phase_ms else "pa_decode (split-K partitions + merge)")
        roof = {"bound": "hbm", "kernel": kern, "achieved": unique_gbs,
                "achieved_logical": decode_gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": unique_gbs / peaks["hbm_gbs"], "peak_source": f"{peak_kind} (hbm_gbs)",
                "frac_of_nominal": unique_gbs / NOMINAL_HBM_GBS,
                "traffic": TRAFFIC_PER_CALL.get(name)}
    e2e = {"value": world * w.kv_unique_bytes / (e2e_ms / 1e3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": h2d,
           "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms, "path": w.e2e_path}
    if e2e_replay_ms is not None:
        e2e["breakdown"] = {"ms_per_step_replay_only": e2e_replay_ms,
                            "ms_per_step_with_copy_engine": e2e_copy_ms,
                            "note": "replay only: the graph replayed with the inputs already in the pinned "
                                    "staging; with copy engine: step() of a runner whose graph copies the "
                                    "inputs to and the output from device buffers"}
    line = {
        "metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world, "steps": K, "warmup": args.warmup,
        "ms_per_step": step_ms_max, "ms_per_step_median": step_ms_median, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": WORKLOAD_CONFIG[name]["dtype"], "data": "synthetic",
        "config": {"workload": name, **WORKLOAD_CONFIG[name],
                   "l2": ("flushed (256 MB read) between steps, outside the timed events" if flush_needed else
                          f"not flushed: inputs larger than L2 ({w.kv_unique_bytes / 2**20:.0f} MiB of KV per step "
                          f"vs 129 MB L2, read in the same order every step)"),
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "value_logical": world * w.kv_bytes / (step_ms_max / 1e3) / 1e9,
        "tokens_per_s": world * w.batch / (step_ms_max / 1e3),
        "pct_of_hbm_peak": 100.0 * value / world / peaks["hbm_gbs"],
        "phase_ms": phase_ms,
        **({"step_ms_phases_in_sequence": step_ms_sequential,
            "sm_split": {"prefill_sms": w.split.sms[0], "decode_sms": w.split.sms[1],
                         "note": "ms_per_step is pa_mixed_step with the prefill and the decode on disjoint SM "
                                 "partitions at once; phase_ms times the three calls one after the other"}}
           if split_ms is not None else {}),
        "decode_gbs": decode_gbs,
        "decode_unique_gbs": unique_gbs,
        "kv_unique_bytes_per_step": w.kv_unique_bytes,
        "store_gbs": w.store_bytes / (store_ms / 1e3) / 1e9 if store_ms else None,
        "store_fused_into_decode": "store+decode" in phase_ms,
        "kv_bytes_per_step": w.kv_bytes,
        "roofline": roof,
        "cpu_baseline": cpu,
        "e2e": e2e,
        "gpu_launches": K * w.launches_per_step,
        "clocks": clk,
        "wall_s_timed_region": t_wall,
    }
    if w.prefill_flops:
        tf = w.prefill_flops / (phase_ms["prefill"] / 1e3) / 1e12
        line["prefill_tflops"] = tf
        line["prefill_flops_per_step"] = w.prefill_flops
        line["roofline_prefill"] = {
            "bound": "tensor", "kernel": "prefill_kernel (tcgen05, bf16 in, fp32 accumulate)", "achieved": tf,
            "peak": peaks["bf16_tflops"], "unit": "TFLOP/s", "frac": tf / peaks["bf16_tflops"],
            "frac_of_sustained_peak": tf / peaks["bf16_tflops_sustained"],
            "peak_source": f"{peak_kind} (bf16_tflops, burst: the kernel is timed by its own events)",
            "traffic": PREFILL_TRAFFIC_PER_CALL.get(name)}
        if world == 1 and cpu_s > 0:
            line["cpu_baseline_prefill"] = prefill_cpu_baselines(cpu_s, cpu_all_s)
    del w
    torch.cuda.empty_cache()
    return line


def measure(name, args, world, rank, local, cpu_s, cpu_all_s):
    try:
        if name == "sampler_qwen3_vocab":
            return measure_sampler(name, args, world, rank, local, cpu_s)
        if name == "store_stress":
            return measure_store(name, args, world, rank, local, cpu_s)
        return measure_attention(name, args, world, rank, local, cpu_s, cpu_all_s)
    finally:
        _INPUTS.pop(name, None)


def run_ours(args, world, rank, local):
    cpu_s = 0.0 if args.no_cpu_baseline else args.cpu_seconds
    cpu_all_s = 0.0 if args.no_cpu_baseline else args.cpu_all_seconds
    line = measure(args.workload, args, world, rank, local, cpu_s, cpu_all_s)
    if not args.no_configs:
        sub_s = 0.0 if args.no_cpu_baseline else args.sub_cpu_seconds
        configs = {}
        for name in SUB_CONFIGS:
            if name == args.workload:
                continue
            rec = measure(name, args, world, rank, local, sub_s, sub_s)
            if rec is not None:
                configs[name] = rec
        if line is not None:
            line["configs"] = configs
    if line is not None:
        print(json.dumps(line), flush=True)


def main():
    args = parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    world, rank, local = dist_setup(args)
    try:
        if args.impl == "reference":
            run_reference(args, world, rank)
        else:
            run_ours(args, world, rank, local)
    finally:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()


if __name__ == "__main__":
    main()
