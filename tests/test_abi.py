"""Host-side checks of the C-ABI library (CPU only: no kernel is launched).

The library must build, load and export every function ``include/sbp.h`` declares;
the workspace query and the argument checks (which run on the host before anything
is enqueued) must behave as the header states.
"""
import ctypes
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def sbp():
    from memory_efficient_exact_gb300 import _build
    _build.build_library()
    from memory_efficient_exact_gb300 import sbp as mod
    return mod


def test_library_exports_every_header_function(sbp):
    names = sbp.header_functions()
    assert {"sbp_lmhead_sft", "sbp_lmhead_grpo", "sbp_lmhead_dpo_pass1", "sbp_lmhead_dpo_pass2",
            "sbp_lmhead_workspace_bytes"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", sbp.LIB_PATH], capture_output=True, text=True).stdout
    exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
    missing = [n for n in names if n not in exported]
    assert not missing, missing
    lib = ctypes.CDLL(sbp.LIB_PATH)
    for n in names:
        getattr(lib, n)


def test_status_strings(sbp):
    assert sbp.status_string(0) == "SBP_OK"
    assert sbp.status_string(4) == "SBP_ERR_LABEL_RANGE"
    assert sbp.status_string(99) == "SBP_ERR_UNKNOWN"


def test_lean_workspace(sbp):
    # two chunk buffers by default for multi-chunk bf16 gradients; the lean size has one
    d, V = 4096, 151936
    full = sbp.workspace_bytes(16384, d, V, 4096, sbp.BF16, sbp.MODE_SFT)
    lean = sbp.workspace_bytes_lean(16384, d, V, 4096, sbp.BF16, sbp.MODE_SFT)
    assert full - lean >= 4096 * V * 2 and lean > 4096 * V * 2
    # one chunk, DPO pass 1 and fp32 have one buffer either way
    assert sbp.workspace_bytes_lean(4096, d, V, 4096, sbp.BF16, sbp.MODE_SFT) == \
        sbp.workspace_bytes(4096, d, V, 4096, sbp.BF16, sbp.MODE_SFT)
    assert sbp.workspace_bytes_lean(16384, d, V, 4096, sbp.BF16, sbp.MODE_DPO1) == \
        sbp.workspace_bytes(16384, d, V, 4096, sbp.BF16, sbp.MODE_DPO1)
    assert sbp.workspace_bytes_lean(256, 64, 1000, 64, sbp.FP32, sbp.MODE_SFT) == \
        sbp.workspace_bytes(256, 64, 1000, 64, sbp.FP32, sbp.MODE_SFT)
    assert sbp.workspace_bytes_lean(16, 0, 10, 4, sbp.BF16, 0) == 0


def test_workspace_bytes(sbp):
    V, d = 151936, 4096
    w1 = sbp.workspace_bytes(16384, d, V, 2048, sbp.BF16, sbp.MODE_SFT)
    w2 = sbp.workspace_bytes(65536, d, V, 2048, sbp.BF16, sbp.MODE_SFT)
    # two chunk buffers of logits (fp16/bf16): chunk c's gradient forms while chunk c+1's
    # forward runs; a single chunk needs only one
    assert w1 > 2 * 2048 * V * 2
    assert w1 < 3 * 2048 * V * 2
    w_one = sbp.workspace_bytes(2048, d, V, 2048, sbp.BF16, sbp.MODE_SFT)
    assert 2048 * V * 2 < w_one < 2 * 2048 * V * 2
    # DPO pass 1 forms no gradient: one buffer
    assert sbp.workspace_bytes(16384, d, V, 2048, sbp.BF16, sbp.MODE_DPO1) < 2 * 2048 * V * 2
    assert w2 - w1 < 64 * 65536                    # T enters only through O(T) scalars
    assert sbp.workspace_bytes(16384, d, V, 4096, sbp.BF16, sbp.MODE_SFT) > w1
    # fp32 path keeps fp32 logits
    assert sbp.workspace_bytes(256, 64, 1000, 64, sbp.FP32, sbp.MODE_SFT) >= 64 * 1000 * 4
    # invalid arguments
    assert sbp.workspace_bytes(16, 0, 10, 4, sbp.BF16, 0) == 0
    assert sbp.workspace_bytes(16, 8, 10, 0, sbp.BF16, 0) == 0
    assert sbp.workspace_bytes(16, 8, 10, 4, 7, 0) == 0
    assert sbp.workspace_bytes(16, 8, 10, 4, sbp.BF16, 9) == 0
    # the chunk never exceeds T
    assert sbp.workspace_bytes(10, 64, 1000, 4096, sbp.FP32, 0) == sbp.workspace_bytes(10, 64, 1000, 10, sbp.FP32, 0)


def _call_sft(lib, **kw):
    a = dict(H=0x1000, W=0x2000, labels=0x3000, T=16, d=64, V=128, chunk=8, ign=-100, dtype=0, loss=0x4000,
             nv=0x5000, lp=None, dH=0x6000, dW=0x7000, acc=0, ws=0x100000, wsb=1 << 30, st=0x8000, stream=None)
    a.update(kw)
    P = ctypes.c_void_p
    return lib.sbp_lmhead_sft(P(a["H"]), P(a["W"]), P(a["labels"]), a["T"], a["d"], a["V"], a["chunk"], a["ign"],
                              a["dtype"], P(a["loss"]), P(a["nv"]), P(a["lp"]), P(a["dH"]), P(a["dW"]), a["acc"],
                              P(a["ws"]), a["wsb"], P(a["st"]), P(a["stream"]))


def test_argument_errors_are_caught_on_the_host(sbp):
    # Every case below fails validation before any CUDA call, so the fake device
    # addresses are never touched.
    lib = sbp._lib
    assert _call_sft(lib, W=None) == sbp.ERR_INVALID_ARG
    assert _call_sft(lib, st=None) == sbp.ERR_INVALID_ARG
    assert _call_sft(lib, dW=None) == sbp.ERR_INVALID_ARG
    assert _call_sft(lib, loss=None) == sbp.ERR_INVALID_ARG
    assert _call_sft(lib, d=-1) == sbp.ERR_INVALID_ARG
    assert _call_sft(lib, chunk=0) == sbp.ERR_INVALID_ARG
    assert _call_sft(lib, dtype=5) == sbp.ERR_INVALID_ARG
    assert _call_sft(lib, d=60) == sbp.ERR_UNSUPPORTED        # bf16 rows must be 16-byte multiples
    assert _call_sft(lib, V=100) == sbp.ERR_UNSUPPORTED
    assert _call_sft(lib, H=0x1008) == sbp.ERR_ALIGNMENT
    assert _call_sft(lib, ws=0x100010) == sbp.ERR_WORKSPACE    # not 256-byte aligned
    assert _call_sft(lib, wsb=16) == sbp.ERR_WORKSPACE          # too small
    P = ctypes.c_void_p
    # GRPO without advantages, DPO pass 2 with an odd number of sequences
    r = lib.sbp_lmhead_grpo(P(0x1000), P(0x2000), P(0x3000), None, P(0x9000), 0.8, 1.2, 16, 64, 128, 8, -100, 0,
                            P(0x4000), None, None, P(0x6000), P(0x7000), 0, P(0x100000), 1 << 30, P(0x8000), None)
    assert r == sbp.ERR_INVALID_ARG
    r = lib.sbp_lmhead_dpo_pass2(P(0x1000), P(0x2000), P(0x3000), P(0x9000), 3, P(0xa000), P(0xb000), 0.1,
                                 16, 64, 128, 8, -100, 0, P(0x4000), None, P(0x6000), P(0x7000), 0,
                                 P(0x100000), 1 << 30, P(0x8000), None)
    assert r == sbp.ERR_INVALID_ARG


def test_host_stream_workspace(sbp):
    # the host-buffer call needs the SFT workspace plus three H-row slots, two dH-row
    # slots (chunk x d elements each) and the labels
    T, d, V, C = 16384, 4096, 151936, 4096
    base = sbp.workspace_bytes(T, d, V, C, sbp.BF16, sbp.MODE_SFT)
    host = sbp.host_workspace_bytes(T, d, V, C, sbp.BF16)
    assert 5 * C * d * 2 + 4 * T <= host - base <= 5 * C * d * 2 + 4 * T + 4 * 256
    # fp32 slots hold fp32 rows; the chunk never exceeds T
    b32 = sbp.workspace_bytes(100, 64, 1000, 4096, sbp.FP32, sbp.MODE_SFT)
    h32 = sbp.host_workspace_bytes(100, 64, 1000, 4096, sbp.FP32)
    assert 5 * 100 * 64 * 4 + 400 <= h32 - b32 <= 5 * 100 * 64 * 4 + 400 + 4 * 256
    assert sbp.host_workspace_bytes(16, 0, 10, 4, sbp.BF16) == 0


def test_host_stream_argument_errors(sbp):
    # fails validation before any CUDA call: the fake addresses are never touched
    lib = sbp._lib
    P = ctypes.c_void_p

    def call(**kw):
        a = dict(H=0x1000, W=0x2000, y=0x3000, T=16, d=64, V=128, chunk=8, dtype=0, loss=0x4000, nv=None,
                 dH=0x6000, dW=0x7000, ws=0x100000, wsb=1 << 30, st=0x8000)
        a.update(kw)
        return lib.sbp_lmhead_sft_host(P(a["H"]), P(a["W"]), P(a["y"]), a["T"], a["d"], a["V"], a["chunk"], -100,
                                       a["dtype"], P(a["loss"]), P(a["nv"]), P(a["dH"]), P(a["dW"]), 0, P(a["ws"]),
                                       a["wsb"], P(a["st"]), None)

    assert call(loss=None) == sbp.ERR_INVALID_ARG
    assert call(H=None) == sbp.ERR_INVALID_ARG
    assert call(y=None) == sbp.ERR_INVALID_ARG
    assert call(dH=None) == sbp.ERR_INVALID_ARG
    assert call(W=None) == sbp.ERR_INVALID_ARG
    assert call(dW=None) == sbp.ERR_INVALID_ARG
    assert call(st=None) == sbp.ERR_INVALID_ARG
    assert call(d=60) == sbp.ERR_UNSUPPORTED
    assert call(W=0x2008) == sbp.ERR_ALIGNMENT
    # the plain SFT workspace lacks the row slots
    assert call(wsb=sbp.workspace_bytes(16, 64, 128, 8, sbp.BF16, sbp.MODE_SFT)) == sbp.ERR_WORKSPACE


def test_checked_and_nvtx_variants(sbp):
    # the checked build (guard zones after every workspace region) and the NVTX build of the
    # same sources: both export every header function; the checked build's workspace is
    # larger by 256 bytes per region, the others' layouts are the release one
    from memory_efficient_exact_gb300 import _build
    names = sbp.header_functions()
    libs = {}
    for v in ("checked", "nvtx"):
        path = _build.build_library(variant=v)
        out = subprocess.run(["nm", "-D", "--defined-only", path], capture_output=True, text=True).stdout
        exported = {l.split()[-1] for l in out.splitlines() if " T " in l}
        assert not [n for n in names if n not in exported], v
        lib = ctypes.CDLL(path)
        lib.sbp_lmhead_workspace_bytes.restype = ctypes.c_size_t
        lib.sbp_lmhead_workspace_bytes.argtypes = [ctypes.c_int64] * 4 + [ctypes.c_int] * 2
        lib.sbp_status_string.restype = ctypes.c_char_p
        lib.sbp_status_string.argtypes = [ctypes.c_int]
        libs[v] = lib
    args = (16384, 4096, 151936, 4096, sbp.BF16, sbp.MODE_SFT)
    base = sbp.workspace_bytes(*args)
    assert libs["nvtx"].sbp_lmhead_workspace_bytes(*args) == base
    extra = libs["checked"].sbp_lmhead_workspace_bytes(*args) - base
    assert extra > 0 and extra % 256 == 0 and extra <= 24 * 256
    assert libs["checked"].sbp_status_string(sbp.ERR_WORKSPACE_OVERRUN) == b"SBP_ERR_WORKSPACE_OVERRUN"
    assert sbp.status_string(sbp.ERR_WORKSPACE_OVERRUN) == "SBP_ERR_WORKSPACE_OVERRUN"


def test_product_path_never_imports_the_oracle():
    pkg = os.path.join(ROOT, "memory_efficient_exact_gb300")
    for dp, _, fs in os.walk(pkg):
        for f in fs:
            if f.endswith((".py", ".cu", ".h", ".cuh")):
                src = open(os.path.join(dp, f)).read()
                assert "import oracle" not in src and "from oracle" not in src, f


def test_binding_fails_loudly_without_its_library(tmp_path):
    # an unknown variant, and a package copy whose library was never built, both raise on
    # import: there is no other implementation to fall back to
    env = dict(os.environ, SBP_LIBRARY_VARIANT="bogus")
    code = f"import sys; sys.path.insert(0, {ROOT!r}); import memory_efficient_exact_gb300.sbp"
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True)
    assert r.returncode != 0 and "SBP_LIBRARY_VARIANT" in r.stderr
    import shutil
    pkg = tmp_path / "memory_efficient_exact_gb300"
    pkg.mkdir()
    for f in ("__init__.py", "sbp.py"):
        src = os.path.join(ROOT, "memory_efficient_exact_gb300", f)
        if os.path.exists(src):
            shutil.copy(src, pkg / f)
    env = dict(os.environ)
    env.pop("SBP_LIBRARY_VARIANT", None)
    code = f"import sys; sys.path.insert(0, {str(tmp_path)!r}); import memory_efficient_exact_gb300.sbp"
    r = subprocess.run([sys.executable, "-c", code], cwd=str(tmp_path), env=env, capture_output=True, text=True)
    assert r.returncode != 0 and "is missing" in r.stderr


def test_header_is_plain_c(sbp, tmp_path):
    # the boundary is a C ABI: the header compiles as C99 (and as C++) on its own, and every
    # function it declares can be referenced from C
    import shutil
    names = sbp.header_functions()
    src = tmp_path / "uses_every_function.c"
    body = "\n".join(f"    (any_fn){n}," for n in names)
    src.write_text('#include "sbp.h"\n#include <stddef.h>\n'
                   "typedef void (*any_fn)(void);\n"
                   f"static const any_fn table[] = {{\n{body}\n}};\n"
                   "int main(void) { return table[0] == NULL; }\n")
    inc = os.path.join(ROOT, "include")
    for cc, extra in (("gcc", ["-std=c99", "-x", "c"]), ("g++", ["-std=c++17", "-x", "c++"])):
        if not shutil.which(cc):
            pytest.skip(f"{cc} not available")
        r = subprocess.run([cc, *extra, "-Wall", "-Wextra", "-Werror", "-pedantic", "-I", inc, "-c", str(src),
                            "-o", str(tmp_path / f"t_{cc}.o")], capture_output=True, text=True)
        assert r.returncode == 0, r.stderr
