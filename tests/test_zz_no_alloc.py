"""pa_attention_noalloc: the allocation-free variant of pa_attention.

Some callers cannot allocate device memory (code inside an allocator's own
callbacks, or under a host framework that owns all device memory), so they
cannot provide pa_attention's workspace. pa_attention_noalloc runs the same
kernels with a fixed scratch array compiled into the library. These tests
call it through the C ABI and check its output against pa_attention's on two
calls in a row (two different batches, so the second call runs on scratch
left over from the first): within the attention tolerances and bit for bit,
since both run the same kernels on the same workspace layout. An oversized
batch is refused.

This file is named to be collected last.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

from paged_kv_cache_42_gb300 import binding  # noqa: E402
from paged_kv_cache_42_gb300 import build  # noqa: E402
from paged_kv_cache_42_gb300 import workloads as wl  # noqa: E402
from tests import gpu_util as gu  # noqa: E402

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    binding.init()
    binding.get_device_error(clear=True)
    yield


def _batches():
    a = wl.make_workload([0, 1023, 2047, 40, 700], [33, 1, 1, 9, 1], num_q_heads=32,
                         num_kv_heads=8, head_dim=128, seed=901)
    b = wl.make_workload([8, 55, 16, 32], [1, 1, 1, 1], num_q_heads=4, num_kv_heads=2,
                         head_dim=64, seed=902)
    return a, b


def test_noalloc_matches_pa_attention_on_two_calls():
    for w in _batches():
        assert binding.workspace_size(w.num_reqs, w.num_tokens, w.num_q_heads, w.num_kv_heads,
                                      w.head_dim) <= binding.noalloc_scratch_bytes()
        dev = gu.DeviceBatch(w)
        dev.write()
        ref = dev.attend().clone()  # pa_attention with a caller-provided workspace
        out = torch.full_like(dev.q, float("nan"))
        binding.attention_noalloc(dev.q, dev.k_cache, dev.v_cache, dev.block_tables,
                                  dev.seq_lens, dev.qsl, w.scale, max_query_len=w.max_query_len,
                                  max_seq_len=w.max_seq_len, out=out)
        torch.cuda.synchronize()
        gu.check_no_device_error()
        got = gu.to_f64(out)
        assert np.isfinite(got).all()
        err = np.abs(got - gu.to_f64(ref))
        assert err.max() <= gu.MAX_ABS and err.mean() <= gu.MEAN_ABS
        # the same kernels on the same workspace layout: the same bits, so a
        # fault in how the shared scratch is reused cannot hide in the tolerance
        assert torch.equal(out.view(torch.int16), ref.view(torch.int16))


def test_noalloc_refuses_a_batch_larger_than_its_scratch():
    cap = binding.noalloc_scratch_bytes()
    T = 1
    while binding.workspace_size(T, T, 32, 8, 128) <= cap:
        T *= 2
    q = torch.zeros((T, 32, 128), dtype=torch.bfloat16, device="cuda")
    kc = torch.zeros((1, 8, 16, 128), dtype=torch.bfloat16, device="cuda")
    bt = torch.zeros((T, 1), dtype=torch.int32, device="cuda")
    sl = torch.ones(T, dtype=torch.int32, device="cuda")
    qsl = torch.arange(T + 1, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.PagedAttentionError) as ei:
        binding.attention_noalloc(q, kc, kc, bt, sl, qsl, 0.1, max_query_len=1, max_seq_len=1,
                                  out=torch.empty_like(q))
    assert ei.value.status == -3
