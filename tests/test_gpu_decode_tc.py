"""GPU parity of the tensor-core split-KV decode (tcgen05) against the CPU
oracle, and of the split-KV merge under any split count.

The tensor-core kernel takes the split-KV work at head_dim 128 over a bf16
cache: by default for GQA groups of 4 and 8, with ``decode_tc`` set to 2 for
every group. Both kernels must match the float64 oracle within the attention
tolerances; they are not bit-identical to each other (the tensor-core P.V
product takes P rounded to bf16).
"""
from __future__ import annotations

import contextlib

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
    binding.set_option("decode_tc", 1)
    binding.set_option("decode_max_workers", 0)
    binding.set_option("decode_self_plan", 1)


@contextlib.contextmanager
def options(**kw):
    try:
        for k, v in kw.items():
            binding.set_option(k, v)
        yield
    finally:
        binding.set_option("decode_tc", 1)
        binding.set_option("decode_max_workers", 0)
        binding.set_option("decode_self_plan", 1)


def _run(w, reqs=None, **opts):
    with options(**opts):
        b = gu.DeviceBatch(w)
        out = b.step()
        torch.cuda.synchronize()
    gu.check_no_device_error()
    return b, gu.to_f64(out)


def _compare(w, what, reqs=None, **opts):
    _, got = _run(w, **opts)
    ref = gu.oracle_reference(w, reqs=reqs)
    if reqs is not None:
        rows = gu.rows_of(w, reqs)
        got, ref = got[rows], ref[rows]
    return gu.assert_close(got, ref, what)


CASES = [
    # (ctx_lens, q_lens, Hq, Hkv): head_dim 128 throughout
    ([0, 14, 15, 16, 31, 63, 64, 127, 128, 129], [1] * 10, 64, 8),  # seq_len edges, G=8
    ([2000, 3, 511, 512, 4095], [1] * 5, 64, 8),                      # G=8 long and short
    ([8, 55, 16, 32, 200, 1000], [1] * 6, 8, 8),                      # G=1
    ([300, 0, 5000, 17], [1, 1, 1, 1], 16, 8),                        # G=2
    ([1000, 1, 130, 4000], [1, 1, 1, 1], 32, 8),                      # G=4
    ([0, 0, 10, 100, 250], [1, 2, 15, 7, 3], 8, 1),                   # MQA-like G=8, short spans
    ([0, 30, 47, 700], [17, 33, 64, 1], 32, 4),                       # prefill chunks beside decodes
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_tensor_core_decode_cases(i):
    ctx, ql, hq, hkv = CASES[i]
    w = wl.make_workload(ctx, ql, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                         seed=1100 + i, pool_factor=1.25)
    _compare(w, f"tc case {i}", decode_tc=2)


def test_tensor_core_decode_random_batches():
    rng = np.random.default_rng(1150)
    for it in range(5):
        R = int(rng.integers(1, 60))
        ctx = rng.integers(0, 2500, size=R)
        ql = np.where(rng.random(R) < 0.85, 1, rng.integers(0, 12, size=R))
        g = int(rng.choice([1, 2, 4, 8]))
        hkv = int(rng.choice([1, 2, 8]))
        ctx = np.maximum(ctx, np.where(ql == 0, 1, 0))
        w = wl.make_workload(ctx, ql, num_q_heads=g * hkv, num_kv_heads=hkv, head_dim=128,
                             seed=1160 + it, pool_factor=1.2)
        _compare(w, f"tc random batch {it}", decode_tc=2)


def test_long_context_every_row():
    # 8 x 32768 tokens, 64 query heads over 8 KV heads: the default routing
    # takes the tensor-core kernel; every row is checked
    w = wl.make_config(5)
    _compare(w, "long context, all rows")


@pytest.mark.parametrize("idx", [2, 4, 5])
def test_full_configs_every_row_on_the_cuda_core_path(idx):
    # the default routing takes these (G = 4 and 8) to the tensor-core kernel;
    # the CUDA-core kernel must still match the oracle on them
    w = wl.make_config(idx)
    _compare(w, f"config {idx} (CUDA-core split-KV), all rows", decode_tc=0)


def test_tensor_core_decode_running_max_jumps():
    # Scores grow by ~4 (log2 units) every 128 keys: the reference max moves
    # by more than 2^8 after the first tile and O is rescaled through TMEM.
    L0 = 1500
    w = wl.make_workload([L0 - 1, 40], [1, 1], num_q_heads=8, num_kv_heads=1, head_dim=128,
                         seed=1190)
    one = wl.to_bf16_bits(np.float32(1.0))
    w.q[...] = one
    for p in range(L0 - 1):
        val = wl.to_bf16_bits(np.float32(0.25 * (p // 128)))
        w.k_cache[w.block_tables[0, p // 16], 0, p % 16, :] = val
    w.k_new[0] = wl.to_bf16_bits(np.float32(0.25 * ((L0 - 1) // 128)))
    _compare(w, "tc rescale path", decode_tc=2)
    # and split over several workers, each with its own reference max
    _compare(w, "tc rescale path, 5 workers", decode_tc=2, decode_max_workers=5)


def test_self_planned_is_bit_identical_to_planner_path():
    rng = np.random.default_rng(1195)
    w = wl.make_workload(rng.integers(0, 3000, size=200), (rng.random(200) < 0.9).astype(int),
                         num_q_heads=64, num_kv_heads=8, head_dim=128, seed=1196)
    b = gu.DeviceBatch(w)
    b.write()
    with options(decode_self_plan=1):
        own = gu.to_bits(b.attend(out=torch.empty_like(b.q)))
    with options(decode_self_plan=0):
        planned = gu.to_bits(b.attend(out=torch.empty_like(b.q)))
    torch.cuda.synchronize()
    gu.check_no_device_error()
    assert np.array_equal(own, planned)


def test_deterministic_and_block_permutation_invariant():
    w = wl.make_workload(np.arange(30) * 211, [1] * 30, num_q_heads=64, num_kv_heads=8,
                         head_dim=128, seed=1197, pool_factor=1.3)
    b = gu.DeviceBatch(w)
    o1 = b.step().clone()
    o2 = b.attend().clone()
    o3 = gu.DeviceBatch(wl.permute_physical_blocks(w, seed=5)).step()
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))
    assert torch.equal(o1.view(torch.int16), o3.view(torch.int16))


@pytest.mark.parametrize("tc", [0, 2])
def test_split_count_does_not_change_the_result(tc):
    # One long request over one KV head: its 16-key blocks are the whole
    # flattened work, so capping the workers at n splits it into exactly n
    # parts (or 1 part: no merge at all), merged by log-sum-exp.
    w = wl.make_workload([8191], [1], num_q_heads=8, num_kv_heads=1, head_dim=128, seed=1198)
    ref = gu.oracle_reference(w)
    outs = {}
    for n in (1, 2, 7, 0):  # 0: every worker the launch has
        _, got = _run(w, decode_tc=tc, decode_max_workers=n)
        gu.assert_close(got, ref, f"{n} splits")
        outs[n] = got
    for n in (1, 2, 7):
        assert np.abs(outs[n] - outs[0]).max() <= gu.MAX_ABS


def test_bad_block_id_is_reported_on_the_tensor_core_path():
    w = wl.make_workload([400, 200], [1, 1], num_q_heads=64, num_kv_heads=8, head_dim=128,
                         seed=1199)
    b = gu.DeviceBatch(w)
    b.write()
    bt = w.block_tables.copy()
    bt[1, 3] = w.num_blocks + 9
    b.block_tables = torch.from_numpy(bt).cuda()
    b.attend()
    torch.cuda.synchronize()
    code, _ = binding.get_device_error(clear=True)
    assert code == 2
