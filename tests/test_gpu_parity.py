"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

KV scatter: bit-exact. Attention: bf16 output within max abs 2e-2 and mean
abs 2e-3 of the float64 oracle. Every unused cache slot holds a NaN sentinel,
so any read outside a request's own valid keys turns up as a non-finite
output.
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


# ---------------------------------------------------------------------------
# KV write
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("case", ["config1", "mixed-small", "d128-chunks"])
def test_write_kv_bit_exact_and_sentinels(case):
    if case == "config1":
        w = wl.make_config(1)
    elif case == "mixed-small":
        w = wl.make_workload([5, 40, 0, 17], [1, 1, 33, 9], num_q_heads=8, num_kv_heads=2,
                             head_dim=64, seed=101, pool_factor=1.6)
    else:
        w = wl.make_workload([0, 100, 7], [64, 1, 40], num_q_heads=32, num_kv_heads=8,
                             head_dim=128, seed=102, pool_factor=1.3)
    b = gu.DeviceBatch(w)
    b.write()
    torch.cuda.synchronize()
    gu.check_no_device_error()
    kc = w.k_cache.copy()
    vc = w.v_cache.copy()
    import oracle
    oracle.write_kv(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    assert np.array_equal(gu.to_bits(b.k_cache), kc)
    assert np.array_equal(gu.to_bits(b.v_cache), vc)


def test_write_kv_padding_and_bad_slot():
    w = wl.make_workload([3, 9], [2, 3], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=103,
                         pool_factor=2.0)
    b = gu.DeviceBatch(w)
    sm = w.slot_mapping.copy()
    sm[1] = -1                      # padding token: skipped
    sm[3] = w.num_blocks * 16 + 5   # outside the pool: skipped + device error
    b.slot_mapping = torch.from_numpy(sm).cuda()
    before_k = gu.to_bits(b.k_cache)
    b.write()
    torch.cuda.synchronize()
    code, detail = binding.get_device_error(clear=True)
    assert code == 1 and detail == 3
    after_k = gu.to_bits(b.k_cache)
    expect = before_k.copy()
    for t, s in enumerate(sm):
        if 0 <= s < w.num_blocks * 16:
            expect[s // 16, :, s % 16, :] = w.k_new[t]
    assert np.array_equal(after_k, expect)


# ---------------------------------------------------------------------------
# attention: small cases in full, against the oracle
# ---------------------------------------------------------------------------
def _run_and_compare(w, what, reqs=None):
    b = gu.DeviceBatch(w)
    out = b.step()
    torch.cuda.synchronize()
    gu.check_no_device_error()
    ref = gu.oracle_reference(w, reqs=reqs)
    got = gu.to_f64(out)
    if reqs is not None:
        rows = gu.rows_of(w, reqs)
        got, ref = got[rows], ref[rows]
    return gu.assert_close(got, ref, what), b


def test_config1_tiny_decode():
    _run_and_compare(wl.make_config(1), "config 1")


SWEEP = [
    # (ctx_lens, q_lens, Hq, Hkv, D)
    ([0, 14, 15, 16, 31, 63, 64], [1] * 7, 8, 2, 128),            # seq_len 1, 15, 16, 17, ...
    ([8, 55, 16, 32, 200, 1000], [1] * 6, 4, 4, 64),              # MHA
    ([0, 0, 10, 100], [1, 2, 15, 16], 8, 1, 64),                  # MQA (G=8), short spans
    ([0, 30, 47], [17, 33, 64], 32, 8, 128),                      # chunks crossing blocks
    ([2000, 3, 511, 512], [1, 1, 1, 1], 64, 8, 128),              # G=8 decodes
    ([0, 16, 1], [5, 1, 40], 2, 1, 128),                          # G=2
    ([300, 0, 5000], [1, 130, 1], 16, 8, 64),                     # G=2, D=64, long
    ([4095, 17], [1, 3], 32, 32, 128),                            # G=1, D=128
]


@pytest.mark.parametrize("i", range(len(SWEEP)))
def test_attention_sweep(i):
    ctx, ql, hq, hkv, d = SWEEP[i]
    w = wl.make_workload(ctx, ql, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=200 + i,
                         pool_factor=1.25)
    _run_and_compare(w, f"sweep {i}")


def test_random_mixed_batches():
    rng = np.random.default_rng(7)
    for it in range(6):
        R = int(rng.integers(1, 40))
        ctx = rng.integers(0, 700, size=R)
        ql = np.where(rng.random(R) < 0.7, 1, rng.integers(0, 70, size=R))
        g = int(rng.choice([1, 2, 4, 8]))
        hkv = int(rng.choice([1, 2, 8]))
        d = int(rng.choice([64, 128]))
        ctx = np.maximum(ctx, np.where(ql == 0, 1, 0))  # a request with no new token still has keys
        w = wl.make_workload(ctx, ql, num_q_heads=g * hkv, num_kv_heads=hkv, head_dim=d,
                             seed=300 + it, pool_factor=1.2)
        _run_and_compare(w, f"random batch {it}")


def test_query_span_of_zero_leaves_rows_untouched():
    w = wl.make_workload([20, 5, 9], [1, 0, 1], num_q_heads=4, num_kv_heads=2, head_dim=64,
                         seed=401)
    b = gu.DeviceBatch(w)
    out = b.step()
    torch.cuda.synchronize()
    ref = gu.oracle_reference(w)
    gu.assert_close(gu.to_f64(out), ref, "qlen 0")


# ---------------------------------------------------------------------------
# full-size configs, in the launch configuration bench.py times: every row of
# every request against the oracle (a second or two of oracle time each)
# ---------------------------------------------------------------------------
@pytest.mark.slow
@pytest.mark.parametrize("idx", [2, 3, 4, 5])
def test_full_config_every_row(idx):
    w = wl.make_config(idx)
    _run_and_compare(w, f"config {idx}, all rows")


# ---------------------------------------------------------------------------
# invariances of the GPU path
# ---------------------------------------------------------------------------
def test_block_permutation_invariance_bit_exact():
    w = wl.make_workload([30, 0, 700, 64], [1, 12, 1, 40], num_q_heads=32, num_kv_heads=8,
                         head_dim=128, seed=501, pool_factor=1.5)
    a = gu.DeviceBatch(w).step()
    b = gu.DeviceBatch(wl.permute_physical_blocks(w, seed=77)).step()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_deterministic():
    w = wl.make_workload(np.arange(40) * 37, [1] * 40, num_q_heads=32, num_kv_heads=8,
                         head_dim=128, seed=502)
    b = gu.DeviceBatch(w)
    o1 = b.step().clone()
    o2 = b.attend().clone()
    torch.cuda.synchronize()
    assert torch.equal(o1.view(torch.int16), o2.view(torch.int16))


def test_shared_prefix_equals_private_copies():
    w = wl.make_workload([1100, 1030, 1500, 1024], [1, 1, 1, 1], num_q_heads=32, num_kv_heads=8,
                         head_dim=128, seed=503, shared_prefix_blocks=64)
    a = gu.DeviceBatch(w).step()
    b = gu.DeviceBatch(wl.unshare_prefix(w, seed=9)).step()
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_mixed_batch_matches_parts():
    w = wl.make_workload([15, 16, 900, 0, 31], [1, 1, 1, 20, 9], num_q_heads=32,
                         num_kv_heads=8, head_dim=128, seed=504)
    whole = gu.to_f64(gu.DeviceBatch(w).step())
    dec = gu.to_f64(gu.DeviceBatch(wl.subset_requests(w, [0, 1, 2])).step())
    pre = gu.to_f64(gu.DeviceBatch(wl.subset_requests(w, [3, 4])).step())
    parts = np.concatenate([dec, pre])
    assert np.abs(whole - parts).max() <= gu.MAX_ABS


# ---------------------------------------------------------------------------
# data-dependent errors: reported on the device error word, nothing faults
# ---------------------------------------------------------------------------
def test_bad_block_id_is_reported():
    w = wl.make_workload([40, 20], [1, 1], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=601)
    b = gu.DeviceBatch(w)
    b.write()
    bt = w.block_tables.copy()
    bt[1, 0] = w.num_blocks + 5
    b.block_tables = torch.from_numpy(bt).cuda()
    b.attend()
    torch.cuda.synchronize()
    code, _ = binding.get_device_error(clear=True)
    assert code == 2


def test_inconsistent_lengths_are_reported():
    w = wl.make_workload([40, 20], [1, 3], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=602)
    b = gu.DeviceBatch(w)
    b.write()
    sl = w.seq_lens.copy()
    sl[1] = 2  # shorter than its 3-token query span
    b.seq_lens = torch.from_numpy(sl).cuda()
    out = b.attend()
    torch.cuda.synchronize()
    code, detail = binding.get_device_error(clear=True)
    assert code == 3 and detail == 1
    assert torch.isnan(out[1:].float()).all()  # rows of the bad request untouched
    ref = gu.oracle_reference(wl.subset_requests(w, [0]))
    gu.assert_close(gu.to_f64(out[:1]), ref, "good request next to a bad one")


def test_batch_larger_than_planner_shared_memory():
    # more than 4096 new tokens: the planner's scratch lives in the workspace
    # and each split-KV worker searches for its first unit itself
    rng = np.random.default_rng(11)
    R = 4400
    ctx = rng.integers(0, 300, size=R)
    w = wl.make_workload(ctx, [1] * (R - 2) + [40, 17], num_q_heads=8, num_kv_heads=2,
                         head_dim=64, seed=612, pool_factor=1.1)
    assert w.num_tokens > 4096
    _run_and_compare(w, "T > 4096", reqs=[0, 1, 2047, 4096, R - 3, R - 2, R - 1])


# ---------------------------------------------------------------------------
# self-planned decode-only batches against the planner path
# ---------------------------------------------------------------------------
def _decode_batches():
    rng = np.random.default_rng(77)
    yield "config 1", wl.make_config(1)
    yield "config 2", wl.make_config(2)
    yield "config 4", wl.make_config(4)
    ctx = rng.integers(0, 3000, size=300)
    ql = (rng.random(300) < 0.9).astype(np.int64)  # some requests have no new token
    yield "300 requests, some idle", wl.make_workload(ctx, ql, num_q_heads=32, num_kv_heads=8,
                                                     head_dim=128, seed=801, pool_factor=1.05)
    yield "G 8, D 64", wl.make_workload(rng.integers(0, 900, size=40), [1] * 40, num_q_heads=16,
                                        num_kv_heads=2, head_dim=64, seed=802)


@pytest.mark.parametrize("which", range(5))
def test_self_planned_decode_is_bit_identical_to_planner_path(which):
    name, w = list(_decode_batches())[which]
    b = gu.DeviceBatch(w)
    b.write()
    try:
        binding.set_option("decode_self_plan", 1)
        own = gu.to_bits(b.attend(out=torch.empty_like(b.q)))
        binding.set_option("decode_self_plan", 0)
        planned = gu.to_bits(b.attend(out=torch.empty_like(b.q)))
    finally:
        binding.set_option("decode_self_plan", 1)
    torch.cuda.synchronize()
    gu.check_no_device_error()
    assert np.array_equal(own, planned), name
    if w.num_tokens <= 400:
        got = gu.to_f64(b.attend())
        gu.assert_close(got[gu.rows_of(w, range(w.num_reqs))],
                        gu.oracle_reference(w)[gu.rows_of(w, range(w.num_reqs))], name)


def test_self_planned_decode_reports_bad_requests():
    w = wl.make_workload([40, 20, 70], [1, 1, 1], num_q_heads=8, num_kv_heads=2, head_dim=128,
                         seed=803)
    b = gu.DeviceBatch(w)
    b.write()
    sl = w.seq_lens.copy()
    sl[1] = w.max_seq_len + 5  # longer than the bound the call was given
    b.seq_lens = torch.from_numpy(sl).cuda()
    out = b.attend()
    torch.cuda.synchronize()
    code, detail = binding.get_device_error(clear=True)
    assert code == 3 and detail == 1
    assert torch.isnan(out[1].float()).all()
    ref = gu.oracle_reference(wl.subset_requests(w, [0, 2]))
    gu.assert_close(gu.to_f64(out[[0, 2]]), ref, "good requests next to a bad one")
