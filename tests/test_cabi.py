"""C-ABI checks that need no GPU: the library loads, exports every entry
point the public header declares, and rejects malformed calls on the host
before touching CUDA."""
from __future__ import annotations

import ctypes
import glob
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = sorted(glob.glob(os.path.join(ROOT, "include", "*.h")))

FAKE = 0x10000  # aligned, never dereferenced: validation fails before any CUDA call


def declared_functions():
    text = "\n".join(open(h).read() for h in HEADERS)
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"^\s*[A-Za-z_][\w\s\*]*?\b(pa_\w+)\s*\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("pa_write_kv", "pa_attention", "pa_attention_workspace_size",
                     "pa_status_string", "pa_get_device_error"):
        assert required in names


def test_library_exports_every_declared_symbol(pa_lib):
    for name in declared_functions():
        assert hasattr(pa_lib, name), f"{name} declared in include/ but not exported"


def test_library_does_not_contain_the_oracle():
    from paged_kv_cache_42_gb300 import build
    out = subprocess.run(["nm", "-D", "--defined-only", build.LIB_PATH], capture_output=True,
                         text=True).stdout
    assert "oracle" not in out
    assert "pa_attention" in out


def test_status_strings(pa_lib):
    for code in (0, -1, -2, -3, -4, -5, -6):
        assert pa_lib.pa_status_string(code)
    assert b"unknown" in pa_lib.pa_status_string(42)


def test_version(pa_lib):
    assert pa_lib.pa_version() >= 100


def test_set_option_validates_values(pa_lib):
    # PA_OPT_DECODE_TM_CTAS_PER_SM takes 1 or 2 only; a valid value is kept
    # until set again (restored here to the default, 2)
    for v in (0, 3, -1):
        assert pa_lib.pa_set_option(7, v) == -1  # PA_ERR_INVALID_ARG
    assert pa_lib.pa_set_option(7, 1) == 0
    assert pa_lib.pa_set_option(7, 2) == 0
    # PA_OPT_MIXED_PREFILL_CTAS: 0 (the planner's choice) or a positive share
    assert pa_lib.pa_set_option(8, -1) == -1
    assert pa_lib.pa_set_option(8, 12) == 0
    assert pa_lib.pa_set_option(8, 0) == 0
    assert pa_lib.pa_set_option(99, 1) == -1  # no such option


def write(pa_lib, **kw):
    a = dict(k=FAKE, v=FAKE, slot=FAKE, kc=FAKE, vc=FAKE, T=4, hkv=2, d=64, bs=16, nb=8)
    a.update(kw)
    return pa_lib.pa_write_kv(a["k"], a["v"], a["slot"], a["kc"], a["vc"], a["T"], a["hkv"],
                              a["d"], a["bs"], a["nb"], None)


def test_write_kv_validation(pa_lib):
    assert write(pa_lib, k=None) == -1
    assert write(pa_lib, slot=None) == -1
    assert write(pa_lib, T=-1) == -1
    assert write(pa_lib, hkv=0) == -1
    assert write(pa_lib, bs=32) == -2
    assert write(pa_lib, d=60) == -2
    assert write(pa_lib, k=FAKE + 8) == -1      # misaligned
    assert write(pa_lib, T=0, k=None) == 0      # empty batch: nothing to do


def attn(pa_lib, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, sl=FAKE, qsl=FAKE, scale=0.125, out=FAKE, R=4,
             T=4, hq=4, hkv=2, d=64, bs=16, nb=32, mb=4, mq=1, ms=56, ws=FAKE, wsb=None)
    a.update(kw)
    if a["wsb"] is None:
        a["wsb"] = pa_lib.pa_attention_workspace_size(a["R"], a["T"], a["hq"], a["hkv"], a["d"])
    return pa_lib.pa_attention(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["qsl"],
                               ctypes.c_float(a["scale"]), a["out"], a["R"], a["T"], a["hq"],
                               a["hkv"], a["d"], a["bs"], a["nb"], a["mb"], a["mq"], a["ms"],
                               a["ws"], a["wsb"], None)


def test_attention_validation(pa_lib):
    assert attn(pa_lib, q=None) == -1
    assert attn(pa_lib, out=None) == -1
    assert attn(pa_lib, R=-1) == -1
    assert attn(pa_lib, hq=6, hkv=4) == -1       # not a multiple
    assert attn(pa_lib, d=96) == -2
    assert attn(pa_lib, bs=32) == -2
    assert attn(pa_lib, hq=32, hkv=2) == -2      # group 16 unsupported
    assert attn(pa_lib, scale=float("nan")) == -1
    assert attn(pa_lib, ws=None) == -3
    assert attn(pa_lib, wsb=16) == -3
    assert attn(pa_lib, ws=FAKE + 16) == -3      # workspace must be 256-byte aligned
    assert attn(pa_lib, q=FAKE + 2) == -1
    assert attn(pa_lib, R=0) == 0                # empty batch
    assert attn(pa_lib, T=2**20, hkv=2, ms=2**20) == -2  # flattened work overflows int32


def test_workspace_size(pa_lib):
    f = pa_lib.pa_attention_workspace_size
    assert f(-1, 4, 4, 2, 64) == 0
    assert f(4, 4, 6, 4, 64) == 0
    a = f(4, 4, 4, 2, 64)
    b = f(4, 400, 4, 2, 64)
    c = f(4, 400, 32, 8, 128)
    assert 0 < a < b < c
    assert a % 256 == 0


@pytest.mark.skipif(__import__("tests.conftest", fromlist=["x"]).cuda_available(),
                    reason="checks the no-GPU error path")
def test_device_calls_fail_cleanly_without_gpu(pa_lib):
    code = ctypes.c_int(0)
    det = ctypes.c_longlong(0)
    assert pa_lib.pa_get_device_error(ctypes.byref(code), ctypes.byref(det), 0) == -4
    assert pa_lib.pa_init() == -4


def test_mapped_pointer_rejects_null_arguments(pa_lib):
    """pa_mapped_pointer checks its arguments before any CUDA call."""
    f = pa_lib.pa_mapped_pointer
    f.argtypes = [ctypes.c_void_p, ctypes.POINTER(ctypes.c_void_p)]
    f.restype = ctypes.c_int
    out = ctypes.c_void_p(0)
    assert f(None, ctypes.byref(out)) == -1
    assert f(ctypes.c_void_p(FAKE), None) == -1
    assert out.value is None


def noalloc(pa_lib, **kw):
    a = dict(q=FAKE, kc=FAKE, vc=FAKE, bt=FAKE, sl=FAKE, qsl=FAKE, scale=0.125, out=FAKE, R=4,
             T=4, hq=4, hkv=2, d=64, bs=16, nb=32, mb=4, mq=1, ms=56)
    a.update(kw)
    return pa_lib.pa_attention_noalloc(a["q"], a["kc"], a["vc"], a["bt"], a["sl"], a["qsl"],
                                       ctypes.c_float(a["scale"]), a["out"], a["R"], a["T"],
                                       a["hq"], a["hkv"], a["d"], a["bs"], a["nb"], a["mb"],
                                       a["mq"], a["ms"], None)


def test_noalloc_reports_argument_errors_before_the_size_check(pa_lib):
    """A batch too large for the fixed scratch still gets pa_attention's own
    error code when its arguments are wrong (checked on the host, no GPU)."""
    big = dict(R=1 << 19, T=1 << 19, hq=32, hkv=8, d=128, ms=16)
    assert noalloc(pa_lib, **big) == -3                # well-formed but too large
    assert noalloc(pa_lib, **dict(big, d=96)) == -2    # unsupported head_dim
    assert noalloc(pa_lib, **dict(big, q=None)) == -1  # null pointer
    assert noalloc(pa_lib, **dict(big, bs=32)) == -2   # unsupported block size
    assert noalloc(pa_lib, R=0) == 0                   # empty batch: nothing to do
