"""Attention output stored straight into pinned host memory.

`out` may be pinned host memory reached through pa_mapped_pointer; the
kernels then store the result across the host link. The result must be bit
for bit the one the same call writes to device memory, on every path that
writes output: split-KV segments, the merge pass, tensor-core chunks, the
cascade and the E4M3 cache.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from paged_kv_cache_42_gb300 import binding  # noqa: E402
from paged_kv_cache_42_gb300 import workloads as wl  # noqa: E402
from tests import gpu_util as gu  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_42_gb300 import build
    build.build()
    binding.init()
    binding.get_device_error(clear=True)
    yield


def _host_out(like: torch.Tensor) -> torch.Tensor:
    return torch.full(tuple(like.shape), float("nan"), dtype=torch.bfloat16).pin_memory()


def _same(a: torch.Tensor, b: torch.Tensor) -> bool:
    return torch.equal(a.cpu().view(torch.int16), b.cpu().view(torch.int16))


@pytest.mark.parametrize("ctx,ql,hq,hkv", [
    ([500, 1200, 3000, 77], [1, 1, 1, 1], 32, 8),        # decode only: self-planned, merges
    ([0, 700, 33, 1500, 90], [100, 1, 1, 37, 1], 32, 8),  # chunks on the tensor cores too
    ([2000, 4000], [1, 1], 64, 8),                        # group 8
])
def test_host_out_matches_device_out(ctx, ql, hq, hkv):
    w = wl.make_workload(ctx, ql, num_q_heads=hq, num_kv_heads=hkv, head_dim=128, seed=1301,
                         pool_factor=1.2)
    b = gu.DeviceBatch(w)
    dev = b.step().clone()
    h = _host_out(b.q)
    binding.attention(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qsl, w.scale,
                      max_query_len=w.max_query_len, max_seq_len=w.max_seq_len, out=h)
    torch.cuda.synchronize()
    gu.check_no_device_error()
    assert _same(h, dev)
    gu.assert_close(gu.to_f64(h), gu.oracle_reference(w), "host out vs oracle")


def test_host_out_cascade_and_fp8():
    w = wl.make_workload([1100, 1200, 1300, 1030], [1, 1, 1, 1], num_q_heads=32, num_kv_heads=8,
                         head_dim=128, seed=1302, shared_prefix_blocks=64)
    b = gu.DeviceBatch(w)
    b.write()
    ws = torch.empty(binding.cascade_workspace_size(w.num_reqs, w.num_tokens, w.num_q_heads,
                                                    w.num_kv_heads, w.head_dim),
                     dtype=torch.uint8, device="cuda")
    args = (b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qsl, w.scale)
    kw = dict(common_prefix_len=1024, max_query_len=w.max_query_len, max_seq_len=w.max_seq_len,
              workspace=ws)
    dev = binding.attention_cascade(*args, **kw).clone()
    h = _host_out(b.q)
    binding.attention_cascade(*args, out=h, **kw)
    torch.cuda.synchronize()
    assert _same(h, dev)

    ks, vs = 0.0113, 0.0127
    kc = torch.from_numpy(oracle.e4m3_quantize(w.k_cache, ks)).cuda()
    vc = torch.from_numpy(oracle.e4m3_quantize(w.v_cache, vs)).cuda()
    binding.write_kv_fp8(b.k, b.v, b.slot_mapping, kc, vc, ks, vs)
    a8 = (b.q, kc, vc, b.block_tables, b.seq_lens, b.qsl, w.scale, ks, vs)
    kw8 = dict(max_query_len=w.max_query_len, max_seq_len=w.max_seq_len)
    dev8 = binding.attention_fp8(*a8, **kw8).clone()
    h8 = _host_out(b.q)
    binding.attention_fp8(*a8, out=h8, **kw8)
    torch.cuda.synchronize()
    gu.check_no_device_error()
    assert _same(h8, dev8)


def test_mapped_pointer_rejects_unpinned_memory():
    t = torch.zeros(64, dtype=torch.bfloat16)  # pageable
    p = ctypes.c_void_p()
    assert binding.lib().pa_mapped_pointer(t.data_ptr(), ctypes.byref(p)) == -1
    assert binding.lib().pa_mapped_pointer(None, ctypes.byref(p)) == -1
    pinned = torch.zeros(64, dtype=torch.bfloat16).pin_memory()
    assert binding.mapped_pointer(pinned) != 0
    w = wl.make_workload([10], [1], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=1303)
    b = gu.DeviceBatch(w)
    with pytest.raises(ValueError):
        binding.attention(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qsl, w.scale,
                          max_query_len=1, max_seq_len=w.max_seq_len,
                          out=torch.empty(tuple(b.q.shape), dtype=torch.bfloat16))
