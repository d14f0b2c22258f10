"""GPU parity of the overlapped mixed batch: prefill chunks on a few SMs beside
the split-KV work.

With the option on (the default), the planner may give the tensor-core
prefill-chunk kernel P SMs and the split-KV kernel the other S - P, both
running at once. The chunks' rows are computed by the same items either way
(bit-identical); the split-KV rows are sliced over fewer workers, so they are
compared with the oracle and with the serial path within the attention
tolerances. The planner's choice is read from the workspace header (its
fourth and fifth ints: prefill CTAs, split-KV workers) to show which path
each case took.
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
    binding.set_option("mixed_overlap", 1)
    binding.set_option("mixed_prefill_ctas", 0)


@contextlib.contextmanager
def overlap(on: bool):
    binding.set_option("mixed_overlap", 1 if on else 0)
    try:
        yield
    finally:
        binding.set_option("mixed_overlap", 1)


def _num_sms():
    return torch.cuda.get_device_properties(0).multi_processor_count


def _run(w, on: bool):
    """(output as float64, prefill CTAs, split-KV workers) of one step."""
    with overlap(on):
        b = gu.DeviceBatch(w)
        out = b.step()
        torch.cuda.synchronize()
    gu.check_no_device_error()
    hdr = b.workspace[:32].view(torch.int32).cpu().numpy()
    return gu.to_f64(out), int(hdr[3]), int(hdr[4])


def _chunk_and_decode_rows(w):
    ql = np.diff(w.query_start_loc)
    chunks = [r for r in range(w.num_reqs) if ql[r] >= 16]
    decodes = [r for r in range(w.num_reqs) if 0 < ql[r] < 16]
    return chunks, decodes


def test_mixed_config_overlapped_against_serial_and_oracle():
    # 512 decodes (L ~ U[128, 2048]) beside three 512-token chunks on contexts
    # 0, 1024 and 2048: the planner overlaps them
    w = wl.make_config(3)
    got, ctas, workers = _run(w, True)
    ser, ctas0, workers0 = _run(w, False)
    S = _num_sms()
    assert 0 < ctas < S and workers == S - ctas, (ctas, workers)
    assert ctas0 == S and workers0 == S
    chunks, decodes = _chunk_and_decode_rows(w)
    crow, drow = gu.rows_of(w, chunks), gu.rows_of(w, decodes)
    # the chunk rows: the same items on either path
    assert np.array_equal(got[crow], ser[crow])
    # the split-KV rows: another slicing, the same attention
    assert np.abs(got[drow] - ser[drow]).max() <= gu.MAX_ABS
    reqs = chunks + decodes[:40] + decodes[-40:]
    rows = gu.rows_of(w, reqs)
    gu.assert_close(got[rows], gu.oracle_reference(w, reqs=reqs)[rows], "overlapped config 3")


def test_chunk_heavy_batch_stays_serial():
    # three long chunks and a few short decodes: the split-KV work is too
    # small to hide the chunks under, so the planner runs them in turn
    w = wl.make_workload([4096, 3000, 2048, 40, 300, 17], [512, 512, 512, 1, 1, 1],
                         num_q_heads=32, num_kv_heads=8, head_dim=128, seed=2101)
    got, ctas, workers = _run(w, True)
    assert ctas == _num_sms()
    gu.assert_close(got, gu.oracle_reference(w), "chunk-heavy batch")


@pytest.mark.parametrize("g", [4, 8])
def test_decode_heavy_batches_with_small_chunks(g):
    # many long decodes beside one or two short chunks: the chunks get one or
    # a few SMs (a single CTA then takes every item)
    rng = np.random.default_rng(2110 + g)
    R = 300
    ctx = rng.integers(1000, 3000, size=R)
    ql = np.ones(R, np.int64)
    ctx[5], ql[5] = 500, 64
    ctx[200], ql[200] = 0, 17
    w = wl.make_workload(ctx, ql, num_q_heads=8 * g, num_kv_heads=8, head_dim=128,
                         seed=2120 + g, pool_factor=1.1)
    got, ctas, workers = _run(w, True)
    S = _num_sms()
    assert 0 < ctas < S and workers == S - ctas, (ctas, workers)
    chunks, decodes = _chunk_and_decode_rows(w)
    reqs = chunks + decodes[:30] + decodes[-30:]
    rows = gu.rows_of(w, reqs)
    gu.assert_close(got[rows], gu.oracle_reference(w, reqs=reqs)[rows], f"G={g} small chunks")
    ser, _, _ = _run(w, False)
    crow = gu.rows_of(w, chunks)
    assert np.array_equal(got[crow], ser[crow])


def test_overlapped_step_is_deterministic_and_split_count_capped():
    w = wl.make_config(3)
    a, _, _ = _run(w, True)
    b, _, _ = _run(w, True)
    assert np.array_equal(a, b)
    # a worker cap below the planner's split still bounds the slicing
    binding.set_option("decode_max_workers", 7)
    try:
        c, ctas, workers = _run(w, True)
    finally:
        binding.set_option("decode_max_workers", 0)
    assert workers == 7
    chunks, decodes = _chunk_and_decode_rows(w)
    reqs = chunks + decodes[:20]
    rows = gu.rows_of(w, reqs)
    gu.assert_close(c[rows], gu.oracle_reference(w, reqs=reqs)[rows], "overlap, 7 workers")


@pytest.mark.parametrize("n", [1, 12, 40, 10000])
def test_forced_prefill_share(n):
    # PA_OPT_MIXED_PREFILL_CTAS: the chunks take min(n, SMs / 2) SMs whatever
    # the cost model says, even on the chunk-heavy batch it keeps serial
    S = _num_sms()
    for w in (wl.make_config(3),
              wl.make_workload([4096, 3000, 40, 300], [512, 512, 1, 1], num_q_heads=32,
                               num_kv_heads=8, head_dim=128, seed=2130)):
        ser, _, _ = _run(w, False)
        binding.set_option("mixed_prefill_ctas", n)
        try:
            got, ctas, workers = _run(w, True)
        finally:
            binding.set_option("mixed_prefill_ctas", 0)
        assert ctas == min(n, S // 2) and workers == S - ctas, (n, ctas, workers)
        chunks, decodes = _chunk_and_decode_rows(w)
        crow = gu.rows_of(w, chunks)
        assert np.array_equal(got[crow], ser[crow])  # the same items on either path
        reqs = chunks + decodes[:20] + decodes[-20:]
        rows = gu.rows_of(w, reqs)
        gu.assert_close(got[rows], gu.oracle_reference(w, reqs=reqs)[rows],
                        f"{n} prefill CTAs")


def test_bad_prefill_share_rejected():
    with pytest.raises(RuntimeError):
        binding.set_option("mixed_prefill_ctas", -1)
