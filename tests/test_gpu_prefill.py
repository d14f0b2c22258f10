"""GPU parity for prefill chunks (the tensor-core path: requests with at
least 16 new tokens) against the CPU oracle."""
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


def _check(w, what):
    b = gu.DeviceBatch(w)
    out = b.step()
    torch.cuda.synchronize()
    gu.check_no_device_error()
    ref = gu.oracle_reference(w)
    return gu.assert_close(gu.to_f64(out), ref, what)


CASES = [
    # (ctx_lens, q_lens, Hq, Hkv, D): chunk shapes around the 128-row / 128-key tiles
    ([0], [16], 4, 1, 64),                      # threshold length, one tile
    ([0], [128], 8, 8, 128),                    # G=1: 128 tokens per tile
    ([100], [200], 16, 8, 128),                 # G=2, tail tile, unaligned context
    ([0, 1024, 2048], [512, 512, 512], 32, 8, 128),  # the mixed-batch chunks
    ([5], [300], 32, 4, 128),                   # G=8: 16 tokens per tile
    ([777], [45], 8, 2, 64),                    # D=64, G=4, partial last block
    ([0, 17], [31, 16], 8, 8, 64),              # several requests, G=1, D=64
    ([3000], [20], 64, 8, 128),                 # long context, G=8, one tile of rows
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_prefill_chunk_cases(i):
    ctx, ql, hq, hkv, d = CASES[i]
    w = wl.make_workload(ctx, ql, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=700 + i,
                         pool_factor=1.3)
    _check(w, f"prefill case {i}")


def test_prefill_running_max_jumps():
    # Scores grow by ~4 (log2 units) every 128 keys, so the running max moves
    # by more than 2^8 and O is rescaled through TMEM.
    L0, ql = 900, 40
    w = wl.make_workload([L0], [ql], num_q_heads=4, num_kv_heads=1, head_dim=128, seed=790)
    one = wl.to_bf16_bits(np.float32(1.0))
    w.q[...] = one
    for p in range(L0):
        val = wl.to_bf16_bits(np.float32(0.25 * (p // 128)))
        w.k_cache[w.block_tables[0, p // 16], 0, p % 16, :] = val
    w.k_new[...] = wl.to_bf16_bits(np.float32(0.25 * (L0 // 128)))
    _check(w, "rescale path")


def test_prefill_and_decode_in_one_batch():
    w = wl.make_workload([300, 0, 1500, 64, 2000], [1, 200, 1, 17, 1], num_q_heads=32,
                         num_kv_heads=8, head_dim=128, seed=791)
    _check(w, "mixed")
