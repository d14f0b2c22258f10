"""The split-KV merge pass at its edges.

A (token, kv head) whose key blocks span many split-KV workers leaves one
partial per worker; the merge pass combines them after the split-KV grid.
These cases push the partial count per merge to its extremes and check the
result against the float64 oracle, the self-planned path against the
planned one bit for bit, and repeated calls for identical bits.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

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
    binding.set_option("decode_self_plan", 1)


def _attend(b: gu.DeviceBatch):
    w = b.w
    out = binding.attention(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qsl,
                            w.scale, max_query_len=w.max_query_len, max_seq_len=w.max_seq_len)
    torch.cuda.synchronize()
    gu.check_no_device_error()
    return out


@pytest.mark.parametrize("ctx,hq,hkv,d", [
    ([40000], 32, 8, 128),  # one request: each kv head's blocks span ~150 workers
    ([60000], 8, 8, 64),    # MHA, D 64
    ([30000], 64, 8, 128),  # group 8
])
def test_one_long_request(ctx, hq, hkv, d):
    w = wl.make_workload(ctx, [1] * len(ctx), num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                         seed=1401, pool_factor=1.1)
    b = gu.DeviceBatch(w)
    b.write()
    got = _attend(b)
    gu.assert_close(gu.to_f64(got), gu.oracle_reference(w), "one long request")
    # planned (not self-planned) launch: the same slices, the same bits
    binding.set_option("decode_self_plan", 0)
    try:
        planned = _attend(b)
    finally:
        binding.set_option("decode_self_plan", 1)
    assert torch.equal(got.view(torch.int16), planned.view(torch.int16))
    again = _attend(b)
    assert torch.equal(got.view(torch.int16), again.view(torch.int16))


def test_long_and_short_requests_together():
    """A long request beside many one-block ones: merges of ~100 partials and
    slices holding dozens of whole (token, kv head) segments in one launch."""
    ctx = [50000] + [int(x) for x in np.random.default_rng(5).integers(0, 15, 200)]
    w = wl.make_workload(ctx, [1] * len(ctx), num_q_heads=32, num_kv_heads=8, head_dim=128,
                         seed=1402, pool_factor=1.1)
    b = gu.DeviceBatch(w)
    b.write()
    got = _attend(b)
    reqs = [0, 1, 2, 100, 199, 200]
    rows = gu.rows_of(w, reqs)
    gu.assert_close(gu.to_f64(got)[rows], gu.oracle_reference(w, reqs=reqs)[rows],
                    "long beside short")
