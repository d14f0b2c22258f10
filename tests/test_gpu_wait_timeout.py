"""The bounded-wait give-up path of the CUDA-core split-KV kernel.

Every wait in the kernels is bounded: a wait that runs out sets
PA_DEVERR_WAIT_TIMEOUT on the device error word and the kernel returns, so a
copy that never completes cannot hang the GPU. To make a wait run out without
a fault, this test builds the library with two test definitions: a 20 ms wait
limit, and a split-KV stage barrier that expects 16 bytes more than the copies
bring (every copy issued still lands, so none is in flight when the CTA
returns). One decode step runs through that build in a child process, which
reports the error word and whether the CUDA context still works.
"""
from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

pytestmark = [pytest.mark.gpu, pytest.mark.slow]

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_split_kv_wait_gives_up_and_reports_without_faulting():
    from paged_kv_cache_42_gb300 import build
    lib = build.build_variant("pagedattn_waittest",
                              ["PA_WAIT_LIMIT_NS=20000000ull", "PA_TEST_EXTRA_TX=16"])
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "wait_timeout_child.py"), lib],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    res = json.loads(r.stdout.strip().splitlines()[-1])
    assert res["code"] == 5, res          # PA_DEVERR_WAIT_TIMEOUT
    assert res["usable"], res             # the context survived
