"""The bench's algorithmic byte counts, checked on CPU against the per-request
definition the roofline uses: for each request, its K and V rows
(L x Hkv x D x 2 tensors x bytes per cached element), its queries in and
outputs out (2 x qlen x Hq x D x 2 B) and its block-table entries
(ceil(L / 16) x 4 B), plus the per-request lengths (8 B) and one offset."""
from __future__ import annotations

import functools
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from paged_kv_cache_42_gb300 import workloads as wl  # noqa: E402


@functools.lru_cache(maxsize=None)
def config(i):
    return wl.make_config(i)


def per_request_bytes(w, elem_bytes):
    kv = qo = meta = 0
    for r in range(w.num_reqs):
        L = int(w.seq_lens[r])
        ql = int(w.query_start_loc[r + 1] - w.query_start_loc[r])
        kv += L * w.num_kv_heads * w.head_dim * 2 * elem_bytes
        qo += 2 * ql * w.num_q_heads * w.head_dim * 2
        meta += -(-L // 16) * 4 + 8
    return kv, kv + qo + meta + 4


@pytest.mark.parametrize("cfg", [1, 2, 5])
@pytest.mark.parametrize("fp8", [False, True])
def test_step_bytes_follow_the_definition(cfg, fp8):
    w = config(cfg)
    sb = bench.step_bytes(w, fp8=fp8)
    kv, attn = per_request_bytes(w, 1 if fp8 else 2)
    assert sb["kv"] == kv and sb["attention"] == attn
    # the KV write: new K and V read as bf16, written as cached elements,
    # plus one 8-byte slot per token
    T = w.num_tokens
    assert sb["write"] == T * w.num_kv_heads * w.head_dim * 2 * (2 + (1 if fp8 else 2)) + T * 8
    assert sb["step"] == sb["attention"] + sb["write"]


def test_llama8b_launch_bytes():
    # the per-launch figures the roofline divides, as recorded with the ncu
    # traffic of the same launches
    w = config(2)
    assert bench.step_bytes(w)["attention"] == 556_685_036
    assert bench.step_bytes(w, fp8=True)["attention"] == 278_884_076
