"""CPU oracle for the paged-KV hot path -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library and its Python binding
never touch it, and it never touches them: the two share no code.

``oracle.c`` is plain single-threaded fp32 C built with ``-O2 -fno-fast-math``.
This module compiles it (``build``) and wraps its entry points for torch CPU
tensors.  ``build_omp`` / ``load_omp`` give the same source built with
``-fopenmp`` (its independent rows spread over the host cores, each row's
arithmetic unchanged): the all-core CPU baseline of the benchmark.  Parity is pinned by ``tests/test_oracle_pins.py`` against
the pages' worked examples, closed forms, brute force and library attention.
"""

from __future__ import annotations

import ctypes
import os
import subprocess

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "oracle.c")
LIB = os.path.join(HERE, "liboracle.so")
LIB_OMP = os.path.join(HERE, "liboracle_omp.so")

F16, BF16 = 0, 1
_DT = {torch.float16: F16, torch.bfloat16: BF16}

_lib = None


def build(src: str = SRC, out: str = LIB, openmp: bool = False) -> str:
    """Compile the oracle (or a variant source) into a shared library (with ``openmp``: the
    multi-threaded build of the same source)."""
    if src == SRC and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    tmp = out + ".tmp"
    omp = ["-fopenmp"] if openmp else []
    subprocess.run(["gcc", "-O2", "-fno-fast-math", "-std=c11", *omp, "-shared", "-fPIC", src, "-o", tmp, "-lm"],
                   check=True)
    os.replace(tmp, out)
    return out


def build_omp() -> str:
    return build(SRC, LIB_OMP, openmp=True)


def _declare(lib):
    p, i32, i64, f32, ci = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_int
    lib.oracle_store_kv.argtypes = [p, p, i64, i64, p, p, p, i32, i32, i32, i32, i32]
    lib.oracle_store_kv.restype = ci
    lib.oracle_decode.argtypes = [p, p, p, p, i32, p, i32, i32, i32, i32, i32, i32, f32, ci, p]
    lib.oracle_decode.restype = ci
    lib.oracle_prefill_paged.argtypes = [p, p, p, p, p, p, p, i32, p, i32, i32, i32, i32, i32, i32, f32, ci, p]
    lib.oracle_prefill_paged.restype = ci
    lib.oracle_store_kv_fp8.argtypes = [p, p, i64, i64, p, p, p, i32, i32, i32, i32, i32, ci, f32, f32]
    lib.oracle_store_kv_fp8.restype = ci
    lib.oracle_decode_fp8.argtypes = [p, p, p, p, i32, p, i32, i32, i32, i32, i32, i32, f32, f32, f32, ci, p]
    lib.oracle_decode_fp8.restype = ci
    lib.oracle_e4m3_to_float.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_to_float.restype = f32
    lib.oracle_float_to_e4m3.argtypes = [f32]
    lib.oracle_float_to_e4m3.restype = ctypes.c_uint8
    lib.oracle_sample.argtypes = [p, i64, i32, i32, i32, p, p, p]
    lib.oracle_sample.restype = ci
    lib.oracle_half_to_float.argtypes = [ctypes.c_uint16, ci]
    lib.oracle_half_to_float.restype = f32
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = ci
    return lib


def load(path: str | None = None):
    """Load the oracle library (building it first if needed)."""
    global _lib
    if path is not None:
        return _declare(ctypes.CDLL(path))
    if _lib is None:
        _lib = _declare(ctypes.CDLL(build()))
    return _lib


_lib_omp = None


def load_omp():
    """The OpenMP build of the oracle (building it first if needed); pass it as ``lib=``."""
    global _lib_omp
    if _lib_omp is None:
        _lib_omp = _declare(ctypes.CDLL(build_omp()))
    return _lib_omp


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _cpu(t, dtype=None):
    assert t.device.type == "cpu"
    t = t.contiguous()
    return t if dtype is None else t.to(dtype)


class OracleError(RuntimeError):
    pass


def store_kv(k, v, k_cache, v_cache, slot_mapping, lib=None):
    """Store rows of k/v ([T, H_kv, D], row stride = stride(0)) into the
    caches in place at ``slot_mapping``.  Raises OracleError on a bad slot."""
    lib = lib or load()
    N, bs, hkv, d = k_cache.shape
    assert k_cache.is_contiguous() and v_cache.is_contiguous()
    assert k.stride(1) == d and k.stride(2) == 1 and v.stride(1) == d and v.stride(2) == 1
    sm = _cpu(slot_mapping, torch.int32)
    rc = lib.oracle_store_kv(_ptr(k), _ptr(v), k.stride(0), v.stride(0), _ptr(k_cache), _ptr(v_cache),
                             _ptr(sm), sm.numel(), hkv, d, N, bs)
    if rc:
        raise OracleError(f"oracle_store_kv rejected its input ({rc})")


def decode(q, k_cache, v_cache, block_tables, context_lens, scale, lib=None) -> torch.Tensor:
    """fp32 [B, H_q, D] decode attention over the paged context."""
    lib = lib or load()
    N, bs, hkv, d = k_cache.shape
    B, hq, _ = q.shape
    q = _cpu(q)
    bt = _cpu(block_tables, torch.int32)
    cl = _cpu(context_lens, torch.int32)
    out = torch.empty(B, hq, d, dtype=torch.float32)
    rc = lib.oracle_decode(_ptr(q), _ptr(k_cache.contiguous()), _ptr(v_cache.contiguous()), _ptr(bt),
                           bt.shape[1] if bt.dim() == 2 else 0, _ptr(cl), B, hq, hkv, d, N, bs,
                           float(scale), _DT[q.dtype], _ptr(out))
    if rc:
        raise OracleError(f"oracle_decode rejected its input ({rc})")
    return out


def prefill_paged(q, k, v, k_cache, v_cache, cu_seqlens_q, cu_seqlens_k, block_tables, scale,
                  lib=None) -> torch.Tensor:
    """fp32 [Tq, H_q, D] causal prefill over a paged prefix plus this step's k/v."""
    lib = lib or load()
    N, bs, hkv, d = k_cache.shape
    tq, hq, _ = q.shape
    q, k, v = _cpu(q), _cpu(k), _cpu(v)
    cq = _cpu(cu_seqlens_q, torch.int32)
    ck = _cpu(cu_seqlens_k, torch.int32)
    bt = _cpu(block_tables, torch.int32) if block_tables is not None else None
    out = torch.empty(tq, hq, d, dtype=torch.float32)
    rc = lib.oracle_prefill_paged(_ptr(q), _ptr(k), _ptr(v), _ptr(k_cache.contiguous()),
                                  _ptr(v_cache.contiguous()), _ptr(cq), _ptr(ck), cq.numel() - 1,
                                  _ptr(bt), bt.shape[1] if bt is not None else 0, hq, hkv, d, N, bs,
                                  float(scale), _DT[q.dtype], _ptr(out))
    if rc:
        raise OracleError(f"oracle_prefill_paged rejected its input ({rc})")
    return out


def half_to_float(bits: int, dtype: torch.dtype, lib=None) -> float:
    lib = lib or load()
    return lib.oracle_half_to_float(bits, _DT[dtype])


def sample(logits: torch.Tensor, temperatures: torch.Tensor, noise: torch.Tensor, lib=None) -> torch.Tensor:
    """Exponential-race sampling of one token per row: logits [B, V] (fp32, bf16
    or fp16), temperatures [B] fp32, noise [B, V] fp32 (the Exp(1) draws)."""
    lib = lib or load()
    logits = logits.contiguous()
    B, V = logits.shape
    dt = {torch.float32: 2, torch.bfloat16: BF16, torch.float16: F16}[logits.dtype]
    temps = temperatures.to(torch.float32).contiguous()
    noise = noise.to(torch.float32).contiguous()
    out = torch.empty(B, dtype=torch.int32)
    rc = lib.oracle_sample(logits.data_ptr(), V, B, V, dt, temps.data_ptr(), noise.data_ptr(), out.data_ptr())
    if rc:
        raise OracleError(f"oracle_sample returned {rc}")
    return out


def store_kv_fp8(k, v, k_cache, v_cache, slot_mapping, k_scale, v_scale, lib=None) -> None:
    """Quantizing store into uint8 E4M3 caches [N, bs, H_kv, D] (in place): e4m3(x / scale)."""
    lib = lib or load()
    T = slot_mapping.numel()
    n, bs, hkv, d = k_cache.shape
    assert k_cache.dtype == torch.uint8 and v_cache.dtype == torch.uint8
    rc = lib.oracle_store_kv_fp8(k.data_ptr(), v.data_ptr(), k.stride(0), v.stride(0), k_cache.data_ptr(),
                                 v_cache.data_ptr(), slot_mapping.contiguous().data_ptr(), T, hkv, d, n, bs,
                                 _DT[k.dtype], float(k_scale), float(v_scale))
    if rc:
        raise OracleError(f"oracle_store_kv_fp8 returned {rc}")


def decode_fp8(q, k_cache, v_cache, block_tables, context_lens, scale, k_scale, v_scale, lib=None) -> torch.Tensor:
    """Decode over uint8 E4M3 caches, fp32 result [B, H_q, D]."""
    lib = lib or load()
    q = q.contiguous()
    B, hq, d = q.shape
    n, bs, hkv, _ = k_cache.shape
    out = torch.empty(B, hq, d, dtype=torch.float32)
    bt = block_tables.contiguous()
    rc = lib.oracle_decode_fp8(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(), bt.data_ptr(), bt.shape[1],
                               context_lens.contiguous().data_ptr(), B, hq, hkv, d, n, bs, float(scale), float(k_scale),
                               float(v_scale), _DT[q.dtype], out.data_ptr())
    if rc:
        raise OracleError(f"oracle_decode_fp8 returned {rc}")
    return out
