"""pa_decode_static_workspace: decode for callers that cannot allocate.

An engine that handed nearly all free device memory to its KV pool, or a
plugin whose host framework owns every device allocation, cannot cudaMalloc a
per-call workspace; this entry point uses the library's own static device
scratch instead.  The test calls it through the C ABI (ctypes, no binding
code) and checks its output against pa_decode with a caller workspace, bit for
bit (the same kernels and plan), on two calls in a row with different shapes
and dtypes (the second call runs over the scratch the first one left behind).
It checks, in a fresh process, that the set-up call (batch 0) is where the
8 MiB is taken and that later calls take no device memory, and that an
oversized shape is refused before anything runs.

This file is named to be collected last, and it passes alone in a fresh
process as well as after the other tests.
"""

import ctypes
import json
import os
import subprocess
import sys
import textwrap

import pytest
import torch

from tests import inputs
from tests.gpu_cases import assert_bit_equal

pytestmark = pytest.mark.gpu


def _entry(lib):
    f = lib.pa_decode_static_workspace
    p, i32, i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
    f.argtypes = [p, i64, p, p, p, i32, p, i32, i32, i32, i32, i32, i32, ctypes.c_float, p, ctypes.c_int, p, p]
    f.restype = ctypes.c_int
    return f


def _call(pa, f, st, q, kc, vc, bt, cl, out):
    n, bs, hkv, d = kc.shape
    dt = pa.PA_BF16 if q.dtype == torch.bfloat16 else pa.PA_F16
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    return f(P(q), q.stride(0), P(kc), P(vc), P(bt), bt.shape[1], P(cl), q.shape[0], q.shape[1], hkv, d, n, bs,
             ctypes.c_float(st.scale), P(out), dt, None, stream)


def _device_step(pa, st):
    p = st.pool
    kc, vc = p.k_cache.cuda(), p.v_cache.cuda()
    pa.store_kv(st.k_new.cuda(), st.v_new.cuda(), kc, vc, st.slot_mapping.cuda())
    return st.q.cuda(), kc, vc, st.block_tables.cuda(), st.context_lens.cuda()


def test_static_workspace_matches_caller_workspace(pa):
    f = _entry(pa.library())
    steps = [inputs.qwen3_0p6b_decode(),                       # bf16, D 128, several partitions per sequence
             inputs.make_decode([1, 17, 100, 255, 3000, 0], num_q_heads=8, num_kv_heads=2, head_dim=64,
                                block_size=16, dtype=torch.float16, seed=61)]
    for st in steps:
        q, kc, vc, bt, cl = _device_step(pa, st)
        ref = pa.decode(q, kc, vc, bt, cl, st.scale)              # existing entry point, caller workspace
        out = torch.full_like(q, float("nan"))
        rc = _call(pa, f, st, q, kc, vc, bt, cl, out)
        assert rc == 0, pa.library().pa_last_error()
        torch.cuda.synchronize()
        assert_bit_equal(out, ref, "static-workspace decode vs pa_decode")


_FRESH = textwrap.dedent("""
    import ctypes, json, sys, torch
    sys.path.insert(0, sys.argv[1])
    import paged_kv_cache_bs_gb300 as pa
    from tests import inputs
    from tests.test_zz_no_alloc import _entry, _call, _device_step
    f = _entry(pa.library())
    st = inputs.qwen3_0p6b_decode()
    q, kc, vc, bt, cl = _device_step(pa, st)     # every tensor of the test is allocated here
    out = torch.empty_like(q)
    torch.cuda.synchronize()
    free = [torch.cuda.mem_get_info()[0]]
    n, bs, hkv, d = kc.shape
    rc0 = f(None, q.stride(0), None, None, None, bt.shape[1], None, 0, q.shape[1], hkv, d, n, bs,
            ctypes.c_float(st.scale), None, pa.PA_BF16, None, None)                  # the set-up call
    torch.cuda.synchronize()
    free.append(torch.cuda.mem_get_info()[0])
    rcs = []
    for _ in range(2):
        rcs.append(_call(pa, f, st, q, kc, vc, bt, cl, out))
        torch.cuda.synchronize()
        free.append(torch.cuda.mem_get_info()[0])
    print(json.dumps({"rc": [rc0] + rcs, "free": free}))
""")


def test_static_workspace_set_up_takes_the_scratch_and_calls_take_nothing():
    # a fresh process with CUDA's default lazy loading: the library's modules are not loaded yet
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, CUDA_MODULE_LOADING="LAZY")
    r = subprocess.run([sys.executable, "-c", _FRESH, root], capture_output=True, text=True, timeout=600, env=env,
                       cwd=root)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["rc"] == [0, 0, 0]
    f0, f1, f2, f3 = res["free"]
    assert f0 - f1 >= 8 << 20, f"the set-up call took {f0 - f1} bytes, expected the 8 MiB scratch"
    assert f1 == f2 == f3, f"decode calls after the set-up took device memory: free {f1} -> {f2} -> {f3}"


def test_static_workspace_rejects_oversized_shapes(pa):
    lib = pa.library()
    f = _entry(lib)
    lib.pa_decode_workspace_bytes.restype = ctypes.c_size_t
    # batch 512, 32 q heads, contexts up to 256 x 256 tokens: far more than 8 MiB of partials
    need = lib.pa_decode_workspace_bytes(512, 32, 8, 128, 256, 256)
    assert need > (8 << 20)
    dummy = torch.zeros(1, dtype=torch.bfloat16, device="cuda")
    P = ctypes.c_void_p(dummy.data_ptr())
    rc = f(P, 32 * 128, P, P, P, 256, P, 512, 32, 8, 128, 10, 256, ctypes.c_float(0.1), P, pa.PA_BF16, None, None)
    assert rc == -2
    assert b"static scratch" in lib.pa_last_error()
