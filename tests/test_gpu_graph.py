"""The library's calls are CUDA-graph capturable: no host synchronisation,
no allocation and no host-read device state on the hot path. A step
(write + attention) captured once and replayed must give exactly what the
same calls give eagerly, including after new inputs are copied into the
captured tensors."""
from __future__ import annotations

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


def _capture(fn):
    """Warm up on a side stream (first-use set-up happens outside the
    capture), then capture fn into a graph."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def _check_replays(make_batch, step, n_new_q=2):
    eager, graphed = make_batch(), make_batch()
    g = _capture(lambda: step(graphed))
    for rep in range(n_new_q + 1):
        if rep:
            q = gu.bf16_tensor(wl.to_bf16_bits(
                np.random.default_rng(rep).standard_normal(tuple(eager.q.shape)).astype(np.float32)))
            eager.q.copy_(q)
            graphed.q.copy_(q)
        want = step(eager).clone()
        g.replay()
        torch.cuda.synchronize()
        gu.check_no_device_error()
        assert np.array_equal(gu.to_bits(graphed.out), gu.to_bits(want)), f"replay {rep}"


def test_mixed_batch_step_in_a_graph():
    """Planner, tensor-core chunks and split-KV decode in one captured step."""
    w = wl.make_workload([0, 700, 33, 1500, 90], [100, 1, 1, 37, 1], num_q_heads=32,
                         num_kv_heads=8, head_dim=128, seed=1201, pool_factor=1.2)

    def step(b):
        return b.step()

    _check_replays(lambda: gu.DeviceBatch(w), step)
    # and the replayed result is the right one
    b = gu.DeviceBatch(w)
    g = _capture(lambda: b.step())
    g.replay()
    torch.cuda.synchronize()
    gu.assert_close(gu.to_f64(b.out), gu.oracle_reference(w), "graph replay vs oracle")


def test_cascade_step_in_a_graph():
    w = wl.make_workload([1100, 1200, 1300, 1030], [1, 1, 1, 1], num_q_heads=32, num_kv_heads=8,
                         head_dim=128, seed=1202, shared_prefix_blocks=64)

    def step(b):
        b.write()
        return binding.attention_cascade(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens,
                                         b.qsl, w.scale, common_prefix_len=1024,
                                         max_query_len=w.max_query_len,
                                         max_seq_len=w.max_seq_len, out=b.out,
                                         workspace=b.cascade_ws)

    def make():
        b = gu.DeviceBatch(w)
        b.cascade_ws = torch.empty(binding.cascade_workspace_size(
            w.num_reqs, w.num_tokens, w.num_q_heads, w.num_kv_heads, w.head_dim),
            dtype=torch.uint8, device="cuda")
        return b

    _check_replays(make, step)


def test_fp8_step_in_a_graph():
    w = wl.make_workload([300, 0, 77], [1, 48, 1], num_q_heads=16, num_kv_heads=4, head_dim=128,
                         seed=1203, pool_factor=1.3)
    ks, vs = 0.0113, 0.0127
    kc8 = oracle.e4m3_quantize(w.k_cache, ks)
    vc8 = oracle.e4m3_quantize(w.v_cache, vs)

    class B:
        def __init__(self):
            d = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
            self.q, self.k, self.v = gu.bf16_tensor(w.q), gu.bf16_tensor(w.k_new), gu.bf16_tensor(w.v_new)
            self.kc, self.vc = d(kc8), d(vc8)
            self.bt, self.sl, self.qsl, self.sm = (d(w.block_tables), d(w.seq_lens),
                                                   d(w.query_start_loc), d(w.slot_mapping))
            self.out = torch.empty_like(self.q)
            self.ws = torch.empty(binding.workspace_size(w.num_reqs, w.num_tokens, w.num_q_heads,
                                                         w.num_kv_heads, w.head_dim),
                                  dtype=torch.uint8, device="cuda")

    def step(b):
        binding.write_kv_fp8(b.k, b.v, b.sm, b.kc, b.vc, ks, vs)
        return binding.attention_fp8(b.q, b.kc, b.vc, b.bt, b.sl, b.qsl, w.scale, ks, vs,
                                     max_query_len=w.max_query_len, max_seq_len=w.max_seq_len,
                                     out=b.out, workspace=b.ws)

    _check_replays(B, step)
