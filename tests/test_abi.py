"""C-ABI checks that need no GPU: the library loads, exports every function
the headers in ``include/`` declare, and rejects invalid arguments on the host
before making any CUDA call.  Also checks that the CUDA library and the oracle
share no symbols."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
                 if f.endswith(".h"))


@pytest.fixture(scope="module")
def lib():
    import importlib.util
    spec = importlib.util.spec_from_file_location("pa_build", os.path.join(ROOT, "paged_kv_cache_bs_gb300", "build.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.build()
    import paged_kv_cache_bs_gb300 as pa
    return pa.library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names |= set(re.findall(r"\b(pa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def exported_symbols(path):
    out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True, check=True).stdout
    return {line.split()[-1] for line in out.splitlines() if line.strip()}


def test_every_declared_function_is_exported(lib):
    import paged_kv_cache_bs_gb300 as pa
    names = declared_functions()
    assert {"pa_store_kv", "pa_decode", "pa_store_decode", "pa_prefill_paged", "pa_decode_workspace_bytes",
            "pa_last_error", "pa_bm_create", "pa_bm_prefill_inputs", "pa_bm_decode_inputs"} <= set(names)
    syms = exported_symbols(pa.LIB_PATH)
    for n in names:
        assert n in syms, n
        assert getattr(lib, n) is not None
    # nothing but the C ABI is exported
    assert {s for s in syms if s.startswith("pa_")} == set(names)


def test_oracle_and_library_share_nothing(lib, oracle_lib):
    import oracle
    import paged_kv_cache_bs_gb300 as pa
    a, b = exported_symbols(pa.LIB_PATH), exported_symbols(oracle.LIB)
    assert not any(s.startswith("oracle_") for s in a)
    assert not any(s.startswith("pa_") for s in b)
    src = open(os.path.join(ROOT, "oracle", "oracle.c")).read()
    assert "pa_api.h" not in src and "pa_common" not in src
    for f in os.listdir(os.path.join(ROOT, "paged_kv_cache_bs_gb300", "csrc")):
        assert "oracle" not in open(os.path.join(ROOT, "paged_kv_cache_bs_gb300", "csrc", f)).read().lower()


FAKE = ctypes.c_void_p(1 << 20)  # aligned, never dereferenced: validation fails first


def test_store_validation(lib):
    args = dict(k=FAKE, v=FAKE, ks=1024, vs=1024, kc=FAKE, vc=FAKE, sm=FAKE, T=4, hkv=8, d=128, n=10, bs=16, dt=1)

    def call(**kw):
        a = {**args, **kw}
        return lib.pa_store_kv(a["k"], a["v"], a["ks"], a["vs"], a["kc"], a["vc"], a["sm"], a["T"], a["hkv"], a["d"],
                               a["n"], a["bs"], a["dt"], None, None)
    assert call(dt=5) == -2
    assert call(T=-1) == -1
    assert call(k=None) == -1
    assert call(kc=None) == -1
    assert call(ks=1000) == -1
    assert call(hkv=0) == -1
    assert call(k=ctypes.c_void_p((1 << 20) + 1)) == -1  # odd address
    assert b"stride" in ctypes.cast(lib.pa_last_error(), ctypes.c_char_p).value or True
    assert call(T=0, k=None, v=None, sm=None) == 0       # empty step is a no-op


def test_decode_validation(lib):
    base = dict(q=FAKE, qs=2048, kc=FAKE, vc=FAKE, bt=FAKE, mb=16, cl=FAKE, B=64, hq=16, hkv=8, d=128, n=700,
                bs=256, scale=0.088, out=FAKE, ws=FAKE, wsb=1 << 30, dt=1)

    def call(**kw):
        a = {**base, **kw}
        return lib.pa_decode(a["q"], a["qs"], a["kc"], a["vc"], a["bt"], a["mb"], a["cl"], a["B"], a["hq"], a["hkv"],
                             a["d"], a["n"], a["bs"], ctypes.c_float(a["scale"]), a["out"], a["ws"], a["wsb"], a["dt"],
                             None, None)
    assert call(hq=12, hkv=8) == -1          # not a multiple
    assert call(hq=48, hkv=3) == -2          # group of 16 unsupported
    assert call(d=96) == -2
    assert call(bs=12) == -2
    assert call(bs=2048) == -2
    assert call(dt=3) == -2
    assert call(B=-1) == -1
    assert call(q=None) == -1
    assert call(ws=None) == -1
    assert call(qs=100) == -1
    assert call(wsb=16) == -1
    assert call(kc=ctypes.c_void_p((1 << 20) + 8)) == -1   # cache not 16-byte aligned
    assert call(scale=float("nan")) == -1
    assert call(B=0, q=None, out=None, ws=None) == 0


def test_workspace_size_is_host_only_and_sane(lib):
    lib.pa_decode_workspace_bytes.restype = ctypes.c_size_t
    w = lib.pa_decode_workspace_bytes(64, 16, 8, 128, 16, 256)
    assert w > 0 and w % 4 == 0
    # the split-K plan depends on the shape: any valid shape needs a positive, 4-byte multiple
    for shape in ((128, 16, 8, 128, 16, 256), (4, 32, 8, 128, 128, 256), (256, 32, 8, 128, 128, 16)):
        v = lib.pa_decode_workspace_bytes(*shape)
        assert v > 0 and v % 4 == 0
    assert lib.pa_decode_workspace_bytes(-1, 16, 8, 128, 16, 256) == 0
    assert lib.pa_decode_workspace_bytes(4, 32, 8, 128, 128, 12) == 0


def test_prefill_validation(lib):
    def call(**kw):
        a = dict(q=FAKE, k=FAKE, v=FAKE, kc=FAKE, vc=FAKE, cq=FAKE, ck=FAKE, S=8, tq=4096, mq=512, mk=4096, bt=FAKE, mb=16,
                 hq=32, hkv=8, d=128, n=600, bs=256, scale=0.088, out=FAKE, dt=1)
        a.update(kw)
        return lib.pa_prefill_paged(a["q"], a["k"], a["v"], a["kc"], a["vc"], a["cq"], a["ck"], a["S"], a["tq"], a["mq"],
                                    a["mk"], a["bt"], a["mb"], a["hq"], a["hkv"], a["d"], a["n"], a["bs"],
                                    ctypes.c_float(a["scale"]), a["out"], a["dt"], None, None)
    assert call(hq=30) == -1
    assert call(d=80) == -2
    assert call(dt=9) == -2
    assert call(mk=100) == -1                       # max_seqlen_k < max_seqlen_q
    assert call(bt=None, k=None) == -1              # packed keys needed without a block table
    assert call(q=ctypes.c_void_p((1 << 20) + 8)) == -1   # TMA needs 16-byte alignment
    assert call(scale=0.0) == -1 and call(scale=-0.1) == -1
    assert call(S=0) == 0 and call(tq=0) == 0
    # (sequence, q tile, head pair) work items are counted in 32 bits
    assert call(S=65535, tq=1 << 30, mq=1 << 20, mk=1 << 20) == -1


def test_prefill_ex_validation(lib):
    import paged_kv_cache_bs_gb300 as pa
    Opt = pa._PrefillOptions  # the binding's mirror of pa_prefill_options
    f = lib.pa_prefill_paged_ex

    def call(opt, **kw):
        a = dict(S=8, tq=4096, mq=512, mk=4096, kc=FAKE)
        a.update(kw)
        return f(FAKE, FAKE, FAKE, a["kc"], FAKE, FAKE, FAKE, a["S"], a["tq"], a["mq"], a["mk"], FAKE, 16, 32, 8, 128,
                 600, 256, ctypes.c_float(0.088), FAKE, 1, None, opt, None)
    assert call(ctypes.byref(Opt(-1))) == -1
    assert call(ctypes.byref(Opt(65536))) == -1
    assert call(ctypes.byref(Opt(4)), kc=None) == -1          # the usual checks still apply
    assert call(ctypes.byref(Opt(4)), S=0) == 0 and call(None, S=0) == 0


def test_store_decode_validation(lib):
    def call(**kw):
        a = dict(k=FAKE, v=FAKE, ks=1024, vs=1024, sm=FAKE, q=FAKE, qs=2048, kc=FAKE, vc=FAKE, bt=FAKE, mb=16, cl=FAKE,
                 B=64, hq=16, hkv=8, d=128, n=700, bs=256, scale=0.088, out=FAKE, ws=FAKE, wsb=1 << 30, dt=1)
        a.update(kw)
        return lib.pa_store_decode(a["k"], a["v"], a["ks"], a["vs"], a["sm"], a["q"], a["qs"], a["kc"], a["vc"],
                                   a["bt"], a["mb"], a["cl"], a["B"], a["hq"], a["hkv"], a["d"], a["n"], a["bs"],
                                   ctypes.c_float(a["scale"]), a["out"], a["ws"], a["wsb"], a["dt"], None, None)
    assert call(k=None) == -1
    assert call(sm=None) == -1
    assert call(ks=1020) == -1                               # not a multiple of 8
    assert call(vs=512) == -1                                # shorter than H_kv * D
    assert call(v=ctypes.c_void_p((1 << 20) + 8)) == -1      # 16-byte alignment
    assert call(d=96) == -2
    assert call(B=0, k=None, v=None, sm=None, q=None, out=None, ws=None) == 0


def test_sample_validation(lib):
    def call(**kw):
        a = dict(lg=FAKE, rs=152000, B=4, V=151936, dt=1, t=FAKE, n=None, out=FAKE)
        a.update(kw)
        return lib.pa_sample(a["lg"], a["rs"], a["B"], a["V"], a["dt"], a["t"], a["n"], ctypes.c_uint64(0),
                             ctypes.c_uint64(0), a["out"], None, None)
    assert call(dt=7) == -2
    assert call(V=0) == -1
    assert call(rs=1000) == -1                                # shorter than vocab
    assert call(lg=ctypes.c_void_p((1 << 20) + 1)) == -1      # element alignment
    assert call(dt=2, lg=ctypes.c_void_p((1 << 20) + 2)) == -1
    assert call(t=None) == -1
    assert call(B=0, lg=None, t=None, out=None) == 0


def test_fp8_store_validation(lib):
    def call(**kw):
        a = dict(k=FAKE, v=FAKE, ks=1024, vs=1024, kc=FAKE, vc=FAKE, sm=FAKE, T=4, hkv=8, d=128, n=10, bs=16, dt=1,
                 ksc=0.01, vsc=0.01)
        a.update(kw)
        return lib.pa_store_kv_fp8(a["k"], a["v"], a["ks"], a["vs"], a["kc"], a["vc"], a["sm"], a["T"], a["hkv"],
                                   a["d"], a["n"], a["bs"], a["dt"], ctypes.c_float(a["ksc"]),
                                   ctypes.c_float(a["vsc"]), None, None)
    assert call(dt=3) == -2                                   # the 16-bit input rows are fp16 / bf16
    assert call(ksc=0.0) == -1 and call(vsc=-1.0) == -1
    assert call(ksc=float("inf")) == -1 and call(vsc=float("nan")) == -1
    assert call(ks=1028) == -1                                # not a multiple of 8
    assert call(d=60, hkv=1, ks=64, vs=64) == -1              # row of 60 elements
    assert call(k=ctypes.c_void_p((1 << 20) + 8)) == -1       # k needs 16-byte alignment
    assert call(kc=ctypes.c_void_p((1 << 20) + 4)) == -1      # caches need 8-byte alignment
    assert call(T=0, k=None, v=None, sm=None) == 0


def test_fp8_decode_validation(lib):
    def call(**kw):
        a = dict(q=FAKE, qs=2048, kc=FAKE, vc=FAKE, bt=FAKE, mb=16, cl=FAKE, B=64, hq=16, hkv=8, d=128, n=700,
                 bs=256, scale=0.088, ksc=0.01, vsc=0.01, out=FAKE, ws=FAKE, wsb=1 << 30, dt=1)
        a.update(kw)
        return lib.pa_decode_fp8(a["q"], a["qs"], a["kc"], a["vc"], a["bt"], a["mb"], a["cl"], a["B"], a["hq"],
                                 a["hkv"], a["d"], a["n"], a["bs"], ctypes.c_float(a["scale"]),
                                 ctypes.c_float(a["ksc"]), ctypes.c_float(a["vsc"]), a["out"], a["ws"], a["wsb"],
                                 a["dt"], None, None)
    assert call(d=64, qs=1024) == -2                          # head_dim 128 only
    assert call(ksc=0.0) == -1 and call(vsc=float("inf")) == -1
    assert call(dt=3) == -2                                   # q / out are fp16 / bf16
    assert call(wsb=16) == -1
    assert call(kc=ctypes.c_void_p((1 << 20) + 8)) == -1      # TMA: 16-byte aligned pool
    assert call(B=0, q=None, out=None, ws=None) == 0
    lib.pa_decode_fp8_workspace_bytes.restype = ctypes.c_size_t
    assert lib.pa_decode_fp8_workspace_bytes(64, 16, 8, 128, 16, 256) > 0
    assert lib.pa_decode_fp8_workspace_bytes(64, 16, 8, 128, 16, 12) == 0


def test_fp8_store_decode_validation(lib):
    def call(**kw):
        a = dict(k=FAKE, v=FAKE, ks=1024, vs=1024, sm=FAKE, q=FAKE, qs=2048, kc=FAKE, vc=FAKE, bt=FAKE, mb=16, cl=FAKE,
                 B=64, hq=16, hkv=8, d=128, n=700, bs=256, scale=0.088, ksc=0.01, vsc=0.01, out=FAKE, ws=FAKE,
                 wsb=1 << 30, dt=1)
        a.update(kw)
        return lib.pa_store_decode_fp8(a["k"], a["v"], a["ks"], a["vs"], a["sm"], a["q"], a["qs"], a["kc"], a["vc"],
                                       a["bt"], a["mb"], a["cl"], a["B"], a["hq"], a["hkv"], a["d"], a["n"], a["bs"],
                                       ctypes.c_float(a["scale"]), ctypes.c_float(a["ksc"]), ctypes.c_float(a["vsc"]),
                                       a["out"], a["ws"], a["wsb"], a["dt"], None, None)
    assert call(k=None) == -1 and call(sm=None) == -1
    assert call(ks=1020) == -1                                # not a multiple of 8
    assert call(v=ctypes.c_void_p((1 << 20) + 8)) == -1      # 16-byte alignment
    assert call(d=64, qs=1024, ks=512, vs=512) == -2          # head_dim 128 only
    assert call(vsc=0.0) == -1
    assert call(B=0, k=None, v=None, sm=None, q=None, out=None, ws=None) == 0


def test_mixed_step_validation(lib):
    """pa_mixed_step checks all three parts before launching anything."""
    def call(**kw):
        a = dict(k=FAKE, v=FAKE, ks=1024, vs=1024, sm=FAKE, T=4216, pq=FAKE, cuq=FAKE, cuk=FAKE, ns=8, tq=4096,
                 mq=512, mk=4096, pbt=FAKE, pmb=16, pout=FAKE, dq=FAKE, dqs=4096, dbt=FAKE, dmb=16, cl=FAKE, B=120,
                 dout=FAKE, ws=FAKE, wsb=1 << 30, kc=FAKE, vc=FAKE, hq=32, hkv=8, d=128, n=2000, bs=256, scale=0.088,
                 dt=1)
        a.update(kw)
        return lib.pa_mixed_step(a["k"], a["v"], a["ks"], a["vs"], a["sm"], a["T"], a["pq"], a["cuq"], a["cuk"],
                                 a["ns"], a["tq"], a["mq"], a["mk"], a["pbt"], a["pmb"], a["pout"], a["dq"], a["dqs"],
                                 a["dbt"], a["dmb"], a["cl"], a["B"], a["dout"], a["ws"], a["wsb"], a["kc"], a["vc"],
                                 a["hq"], a["hkv"], a["d"], a["n"], a["bs"], ctypes.c_float(a["scale"]), a["dt"], None,
                                 None, None)
    assert call(dt=5) == -2
    assert call(T=-1) == -1
    assert call(sm=None) == -1                                 # the store's slots
    assert call(pbt=None) == -1                                # the prefill reads the pool through its tables
    assert call(mk=100) == -1                                  # max_seqlen_k < max_seqlen_q
    assert call(pout=ctypes.c_void_p((1 << 20) + 8)) == -1    # prefill out 16-byte aligned
    assert call(dqs=100) == -1                                 # decode q rows shorter than H_q * D
    assert call(wsb=16) == -1                                  # decode workspace too small
    assert call(hq=20) == -1                                   # H_q not a multiple of H_kv
    assert call(hq=24) == -2                                   # GQA group of 3


def test_sm_split_validation(lib):
    assert lib.pa_sm_split_create(96, None) == -1
    assert lib.pa_sm_split_info(None, None, None, None, None) == -1
    lib.pa_sm_split_destroy(None)


def test_selftest_wait_timeout_validation(lib):
    assert lib.pa_selftest_wait_timeout(0, FAKE, None) == -1
    assert lib.pa_selftest_wait_timeout(5_000_000_000, FAKE, None) == -1
    assert lib.pa_selftest_wait_timeout(1000, None, None) == -1


def test_headers_compile_as_plain_c(tmp_path):
    """The C ABI headers are plain C99: a C translation unit includes them without warnings."""
    src = tmp_path / "abi.c"
    src.write_text("".join(f'#include "{os.path.basename(h)}"\n' for h in HEADERS) +
                   "int main(void) { return pa_version() > 0 ? 0 : 1; }\n")
    r = subprocess.run(["gcc", "-std=c99", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                        "-c", str(src), "-o", str(tmp_path / "abi.o")], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def test_store_decode_fp8_ex_takes_operands_only(lib):
    import paged_kv_cache_bs_gb300 as pa
    F = FAKE
    for field, val in (("partition", 128), ("stages", 2), ("num_groups", 1), ("prefix_partition", 64)):
        opt = pa._Options()
        setattr(opt, field, val)
        rc = lib.pa_store_decode_fp8_ex(F, F, 1024, 1024, F, F, 2048, F, F, F, 4, F, 2, 16, 8, 128, 64, 256, 0.1,
                                        1.0, 1.0, F, F, 1 << 20, ctypes.byref(opt), 1, None, None)
        assert rc == -1, field
        assert b"operands only" in lib.pa_last_error()
