"""Cascade attention (pa_attention_cascade) against the CPU oracle.

Cascade attention computes the common prefix once for the whole batch and
merges it with each request's own suffix by log-sum-exp renormalisation
("vLLM: An Exhaustive Technical Study for Kernel Engineers", 2.3). It reaches
the plain result up to rounding, so the oracle is the plain definition (the
same float64 attention oracle as for pa_attention), with the same tolerances.
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


def cascade(b: gu.DeviceBatch, prefix_len: int, out=None):
    w = b.w
    return binding.attention_cascade(
        b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qsl, w.scale,
        common_prefix_len=prefix_len, max_query_len=w.max_query_len, max_seq_len=w.max_seq_len,
        out=b.out if out is None else out)


def run_case(w: wl.Workload, prefix_len: int, what: str, reqs=None):
    b = gu.DeviceBatch(w)
    b.write()
    out = cascade(b, prefix_len)
    torch.cuda.synchronize()
    gu.check_no_device_error()
    ref = gu.oracle_reference(w, reqs=reqs)
    got = gu.to_f64(out)
    if reqs is not None:
        rows = gu.rows_of(w, reqs)
        got, ref = got[rows], ref[rows]
    gu.assert_close(got, ref, what)
    return b, out


def test_prefix_share_config_full():
    """128 decodes sharing a 1024-token prefix (the prefix-sharing benchmark
    shape), every request against the oracle."""
    w = wl.make_config(4)
    run_case(w, w.shared_prefix_blocks * 16, "prefix-share cascade")


def test_cascade_matches_plain_attention_on_gpu():
    w = wl.make_config(4)
    b = gu.DeviceBatch(w)
    b.write()
    plain = b.attend(out=torch.empty_like(b.q)).float()
    casc = cascade(b, w.shared_prefix_blocks * 16, out=torch.empty_like(b.q)).float()
    torch.cuda.synchronize()
    gu.check_no_device_error()
    assert (plain - casc).abs().max().item() <= gu.MAX_ABS


@pytest.mark.parametrize("overlap", [0, 1])
def test_prefix_pass_beside_suffix_pass(overlap):
    # the prefix pass on a few SMs beside the suffix pass (every (token, kv
    # head) folded by the merge pass), or first (folded by the suffix pass):
    # both match the oracle, and each other
    w = wl.make_config(4)
    binding.set_option("cascade_overlap", overlap)
    try:
        b, out = run_case(w, w.shared_prefix_blocks * 16, f"prefix-share cascade, overlap {overlap}")
        binding.set_option("cascade_overlap", 1 - overlap)
        other = cascade(b, w.shared_prefix_blocks * 16, out=torch.empty_like(b.q)).float()
        torch.cuda.synchronize()
        gu.check_no_device_error()
        assert (out.float() - other).abs().max().item() <= gu.MAX_ABS
    finally:
        binding.set_option("cascade_overlap", 1)


CASES = [
    # (ctx_lens, q_lens, Hq, Hkv, D, shared prefix blocks)
    ([40, 17, 90], [1, 1, 1], 8, 2, 128, 1),                   # 16-key prefix, one partial tile
    ([300, 129, 800, 144], [1, 1, 1, 1], 32, 8, 128, 8),       # 128-key prefix: one key tile
    ([160, 400, 170], [1, 3, 1], 16, 4, 128, 9),               # 144 keys: a ragged key tile
    ([2100, 2500, 3000], [1, 1, 1], 32, 8, 128, 128),          # 2048-key prefix, many chunks
    ([520, 700], [40, 1], 8, 8, 64, 32),                       # MHA, D 64, a chunk on top
    ([100, 130, 260, 99], [1, 2, 1, 1], 16, 2, 64, 6),         # G 8
    ([80, 81, 82, 83, 84], [1] * 5, 4, 2, 64, 5),              # G 2, prefix = nearly all keys
]


@pytest.mark.parametrize("i", range(len(CASES)))
def test_cascade_cases(i):
    ctx, ql, hq, hkv, d, pb = CASES[i]
    w = wl.make_workload(ctx, ql, num_q_heads=hq, num_kv_heads=hkv, head_dim=d,
                         seed=700 + i, shared_prefix_blocks=pb, pool_factor=1.3)
    run_case(w, pb * 16, f"cascade case {i}")


def test_cascade_many_tokens_one_chunk():
    """Enough tokens that the prefix pass needs a single key chunk (row-tile
    pairs alone fill the GPU), with a ragged last pair."""
    rng = np.random.default_rng(5)
    R = 1000
    ctx = 512 + rng.integers(0, 600, size=R)
    w = wl.make_workload(ctx, [1] * R, num_q_heads=32, num_kv_heads=8, head_dim=128, seed=731,
                         shared_prefix_blocks=32, pool_factor=1.1)
    run_case(w, 512, "1000 tokens", reqs=[0, 1, 499, 998, 999])


def test_cascade_prefix_shorter_than_sharing():
    """The common prefix handed to the call may be shorter than what the
    requests really share: the rest is just part of each suffix."""
    w = wl.make_workload([600, 700, 800], [1, 1, 1], num_q_heads=32, num_kv_heads=8,
                         head_dim=128, seed=741, shared_prefix_blocks=30)
    run_case(w, 16 * 7, "prefix 7 of 30 shared blocks")


def test_cascade_deterministic():
    w = wl.make_config(4)
    b = gu.DeviceBatch(w)
    b.write()
    o1 = gu.to_bits(cascade(b, 1024, out=torch.empty_like(b.q)))
    o2 = gu.to_bits(cascade(b, 1024, out=torch.empty_like(b.q)))
    assert np.array_equal(o1, o2)


def test_short_context_is_reported_and_skipped():
    w = wl.make_workload([300, 300, 300], [1, 1, 1], num_q_heads=8, num_kv_heads=2,
                         head_dim=128, seed=751, shared_prefix_blocks=4)
    b = gu.DeviceBatch(w)
    b.write()
    sl = w.seq_lens.copy()
    sl[2] = 60  # context 59 < the 64-token prefix
    b.seq_lens = torch.from_numpy(sl).cuda()
    out = cascade(b, 64)
    torch.cuda.synchronize()
    code, detail = binding.get_device_error(clear=True)
    assert code == 3 and detail == 2
    assert torch.isnan(out[2:].float()).all()  # the bad request's row untouched
    ref = gu.oracle_reference(wl.subset_requests(w, [0, 1]))
    gu.assert_close(gu.to_f64(out[:2]), ref, "good requests next to a bad one")


def test_foreign_prefix_block_is_reported():
    w = wl.make_workload([300, 300], [1, 1], num_q_heads=8, num_kv_heads=2, head_dim=128,
                         seed=761, shared_prefix_blocks=4)
    b = gu.DeviceBatch(w)
    b.write()
    bt = w.block_tables.copy()
    bt[1, 2] = bt[1, 10]  # request 1's third prefix block is not request 0's
    b.block_tables = torch.from_numpy(bt).cuda()
    cascade(b, 64)
    torch.cuda.synchronize()
    code, detail = binding.get_device_error(clear=True)
    assert code == 6 and detail == 1


def test_host_rejections():
    w = wl.make_workload([300, 300], [1, 1], num_q_heads=8, num_kv_heads=2, head_dim=128,
                         seed=771, shared_prefix_blocks=4)
    b = gu.DeviceBatch(w)
    for bad in (0, 40, -16, w.max_seq_len + 16):
        with pytest.raises(binding.PagedAttentionError) as e:
            cascade(b, bad)
        assert e.value.status == -1
    small = torch.empty(binding.workspace_size(2, 2, 8, 2, 128), dtype=torch.uint8,
                        device="cuda")
    with pytest.raises(binding.PagedAttentionError) as e:
        binding.attention_cascade(b.q, b.k_cache, b.v_cache, b.block_tables, b.seq_lens, b.qsl,
                                  w.scale, common_prefix_len=64, max_query_len=1,
                                  max_seq_len=w.max_seq_len, workspace=small)
    assert e.value.status == -3
