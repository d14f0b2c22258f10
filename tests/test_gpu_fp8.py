"""FP8 (E4M3) KV cache on the GPU against the oracle.

The quantising write must match the oracle bit for bit (the code is decided
from the same binary32 quotient on both sides). Attention over an E4M3 cache
is compared with the float64 oracle on the same codes and scales, with the
same tolerances as the bf16 path: both sides see identical dequantised keys
and values, so only fp32 rounding and the bf16 output differ. Unused cache
slots hold the E4M3 NaN code, so a read outside a request's keys shows up as
a non-finite output.
"""
from __future__ import annotations

import numpy as np
import pytest

torch = pytest.importorskip("torch")

import oracle  # noqa: E402
from paged_kv_cache_42_gb300 import binding  # noqa: E402
from paged_kv_cache_42_gb300 import workloads as wl  # noqa: E402
from tests import gpu_util as gu  # noqa: E402

pytestmark = pytest.mark.gpu

E4M3_NAN = 0x7F


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from paged_kv_cache_42_gb300 import build
    build.build()
    binding.init()
    binding.get_device_error(clear=True)
    yield


class Fp8Batch:
    """A workload whose cached context is stored as E4M3 codes."""

    def __init__(self, w: wl.Workload, k_scale: float, v_scale: float):
        self.w, self.ks, self.vs = w, float(k_scale), float(v_scale)
        # context codes from the oracle's quantiser (NaN sentinels stay NaN codes)
        self.kc_cpu = oracle.e4m3_quantize(w.k_cache, self.ks)
        self.vc_cpu = oracle.e4m3_quantize(w.v_cache, self.vs)
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        self.kc = dev(self.kc_cpu)
        self.vc = dev(self.vc_cpu)
        self.q = gu.bf16_tensor(w.q)
        self.k = gu.bf16_tensor(w.k_new)
        self.v = gu.bf16_tensor(w.v_new)
        self.bt = dev(w.block_tables)
        self.sl = dev(w.seq_lens)
        self.qsl = dev(w.query_start_loc)
        self.sm = dev(w.slot_mapping)
        self.out = torch.full_like(self.q, float("nan"))

    def write(self):
        binding.write_kv_fp8(self.k, self.v, self.sm, self.kc, self.vc, self.ks, self.vs)

    def attend(self):
        w = self.w
        return binding.attention_fp8(self.q, self.kc, self.vc, self.bt, self.sl, self.qsl,
                                     w.scale, self.ks, self.vs, max_query_len=w.max_query_len,
                                     max_seq_len=w.max_seq_len, out=self.out)

    def oracle_after_write(self, reqs=None):
        kc, vc = self.kc_cpu.copy(), self.vc_cpu.copy()
        oracle.write_kv_fp8(self.w.k_new, self.w.v_new, self.w.slot_mapping, kc, vc, self.ks,
                            self.vs)
        ref = oracle.attention_fp8(self.w.q, kc, vc, self.ks, self.vs, self.w.block_tables,
                                   self.w.seq_lens, self.w.query_start_loc, self.w.scale,
                                   reqs=reqs)
        return kc, vc, ref


def run(w, ks, vs, what, reqs=None):
    b = Fp8Batch(w, ks, vs)
    b.write()
    out = b.attend()
    torch.cuda.synchronize()
    gu.check_no_device_error()
    kc, vc, ref = b.oracle_after_write(reqs)
    assert np.array_equal(b.kc.cpu().numpy(), kc), f"{what}: K cache differs from the oracle"
    assert np.array_equal(b.vc.cpu().numpy(), vc), f"{what}: V cache differs from the oracle"
    got = gu.to_f64(out)
    if reqs is not None:
        rows = gu.rows_of(w, reqs)
        got, ref = got[rows], ref[rows]
    return gu.assert_close(got, ref, what)


@pytest.mark.parametrize("ks,vs", [(1.0, 1.0), (0.0113, 0.0127), (0.25, 3.0)])
def test_quantising_write_bit_exact(ks, vs):
    w = wl.make_workload([0, 100, 7, 33], [64, 1, 40, 1], num_q_heads=32, num_kv_heads=8,
                         head_dim=128, seed=1102, pool_factor=1.3)
    b = Fp8Batch(w, ks, vs)
    sm = w.slot_mapping.copy()
    sm[3] = -1  # a padding token is skipped
    b.sm = torch.from_numpy(sm).cuda()
    b.write()
    torch.cuda.synchronize()
    gu.check_no_device_error()
    kc, vc = b.kc_cpu.copy(), b.vc_cpu.copy()
    oracle.write_kv_fp8(w.k_new, w.v_new, sm, kc, vc, ks, vs)
    assert np.array_equal(b.kc.cpu().numpy(), kc)
    assert np.array_equal(b.vc.cpu().numpy(), vc)


def test_quantising_write_saturates():
    """Values far beyond 448 * scale store the largest finite code."""
    w = wl.make_workload([0], [16], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=1103)
    big = wl.to_bf16_bits((wl.bf16_bits_to_f32(w.k_new) * 3000.0).astype(np.float32))
    w.k_new = big
    run(w, 1.0, 1.0, "saturating write")


SWEEP = [
    # (ctx_lens, q_lens, Hq, Hkv, D)
    ([0, 14, 15, 16, 31, 63, 64], [1] * 7, 8, 2, 128),
    ([8, 55, 16, 32, 200, 1000], [1] * 6, 4, 4, 64),
    ([100, 300, 17], [1, 1, 1], 32, 8, 128),
    ([50, 700, 2000], [1, 1, 1], 64, 8, 128),   # G 8
    ([90, 0, 400], [1, 40, 3], 16, 8, 64),       # G 2, a 40-token chunk
    ([0, 513], [100, 1], 32, 8, 128),            # a long chunk with no context
    ([300, 1000], [64, 37], 64, 8, 128),         # G 8 chunks on the tensor cores
    ([200, 5], [130, 16], 8, 8, 64),             # MHA, D 64, ragged key tiles
]


@pytest.mark.parametrize("i", range(len(SWEEP)))
@pytest.mark.parametrize("scales", [(1.0, 1.0), (0.0113, 0.0127)])
def test_attention_fp8_sweep(i, scales):
    ctx, ql, hq, hkv, d = SWEEP[i]
    w = wl.make_workload(ctx, ql, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=1110 + i,
                         pool_factor=1.3)
    run(w, *scales, f"fp8 sweep {i} scales {scales}")


def test_llama8b_decode_fp8_every_row():
    w = wl.make_config(2)
    run(w, 0.0113, 0.0127, "llama8b fp8, all rows")


def test_long_context_fp8_every_row():
    w = wl.make_config(5)
    run(w, 0.0113, 0.0127, "long context fp8, all rows")


# ---------------------------------------------------------------------------
# the tensor-core split-KV kernel over E4M3 codes (kind::f8f6f4: the queries
# split into two E4M3 terms, P' = 256 p split likewise), forced onto every
# group, and the CUDA-core kernel forced onto the groups it no longer takes
# ---------------------------------------------------------------------------
TC_CASES = [
    # (ctx_lens, q_lens, Hq, Hkv)
    ([0, 14, 15, 16, 31, 63, 64, 127, 128, 129], [1] * 10, 64, 8),  # seq_len edges, G 8
    ([2000, 3, 511, 512, 4095], [1] * 5, 32, 8),                      # G 4
    ([8, 55, 16, 32, 200, 1000], [1] * 6, 8, 8),                      # G 1
    ([300, 0, 5000, 17], [1, 1, 1, 1], 16, 8),                        # G 2
    ([0, 0, 10, 100, 250], [1, 2, 15, 7, 3], 8, 1),                   # short spans, G 8
]


TM_CPS_DEFAULT = 2  # PA_OPT_DECODE_TM_CTAS_PER_SM's default


@pytest.fixture
def decode_tc_option():
    yield binding.set_option
    binding.set_option("decode_tc", 1)
    binding.set_option("decode_max_workers", 0)
    binding.set_option("decode_token_major", 1)
    binding.set_option("decode_tm_ctas_per_sm", TM_CPS_DEFAULT)


@pytest.mark.parametrize("i", range(len(TC_CASES)))
@pytest.mark.parametrize("tc,tm", [(0, 1), (2, 1), (2, 0)])
def test_attention_fp8_both_split_kv_kernels(i, tc, tm, decode_tc_option):
    # tc 2 with eight KV heads: the token-major tiles (tm 1) or the
    # per-(token, kv head) tiles (tm 0)
    ctx, ql, hq, hkv = TC_CASES[i]
    w = wl.make_workload(ctx, ql, num_q_heads=hq, num_kv_heads=hkv, head_dim=128,
                         seed=1160 + i, pool_factor=1.3)
    decode_tc_option("decode_tc", tc)
    decode_tc_option("decode_token_major", tm)
    run(w, 0.0113, 0.0127, f"fp8 split-KV kernel {tc}/{tm} case {i}")


def test_attention_fp8_tensor_core_running_max_and_splits(decode_tc_option):
    # scores that grow along the sequence move the reference max (and rescale
    # both column groups of O); capping the workers splits it over 5 parts
    L0 = 1500
    w = wl.make_workload([L0 - 1], [1], num_q_heads=8, num_kv_heads=1, head_dim=128, seed=1170)
    w.q[...] = wl.to_bf16_bits(np.float32(1.0))
    for p in range(L0 - 1):
        w.k_cache[w.block_tables[0, p // 16], 0, p % 16, :] = wl.to_bf16_bits(
            np.float32(0.05 * (p // 64)))
    w.k_new[0] = wl.to_bf16_bits(np.float32(0.05 * ((L0 - 1) // 64)))
    decode_tc_option("decode_tc", 2)
    run(w, 0.03, 1.0, "fp8 tc running max")
    decode_tc_option("decode_max_workers", 5)
    run(w, 0.03, 1.0, "fp8 tc running max, 5 parts")


@pytest.mark.parametrize("cps", [1, 2])
@pytest.mark.parametrize("g", [1, 2, 4, 8])
def test_token_major_running_max_and_splits(g, cps, decode_tc_option):
    # Eight KV heads whose scores grow along the sequence at head-dependent
    # rates: references move in some half-warps and not others (O^T columns
    # rescaled per query head); then the same over 1, 2 and 7 workers (token
    # partials per kv head in slots (token + worker) * 8 + kv head)
    L0 = 1500
    w = wl.make_workload([L0 - 1, 300], [1, 1], num_q_heads=8 * g, num_kv_heads=8,
                         head_dim=128, seed=1180 + g)
    w.q[...] = wl.to_bf16_bits(np.float32(1.0))
    for kv in range(8):
        rate = 0.01 * kv
        for p in range(L0 - 1):
            w.k_cache[w.block_tables[0, p // 16], kv, p % 16, :] = wl.to_bf16_bits(
                np.float32(rate * (p // 64)))
        w.k_new[0, kv] = wl.to_bf16_bits(np.float32(rate * ((L0 - 1) // 64)))
    decode_tc_option("decode_tc", 2)
    decode_tc_option("decode_tm_ctas_per_sm", cps)  # 2: taken at G <= 4
    run(w, 0.03, 1.0, f"fp8 token-major running max, G {g}, {cps} CTAs per SM")
    for n in (1, 2, 7):
        decode_tc_option("decode_max_workers", n)
        run(w, 0.03, 1.0, f"fp8 token-major running max, G {g}, {n} parts")


@pytest.mark.parametrize("cps", [1, 2])
def test_token_major_random_batches(cps, decode_tc_option):
    # decode-only batches (self-planned) and batches with short spans and
    # tensor-core chunks (planner path), at every group size
    decode_tc_option("decode_tm_ctas_per_sm", cps)
    rng = np.random.default_rng(1190)
    for it in range(6):
        R = int(rng.integers(1, 50))
        ctx = rng.integers(0, 3000, size=R)
        ql = np.ones(R, np.int64) if it % 2 == 0 else np.where(
            rng.random(R) < 0.8, 1, rng.integers(0, 40, size=R))
        ctx = np.maximum(ctx, np.where(ql == 0, 1, 0))
        g = [1, 2, 4, 8][it % 4]
        w = wl.make_workload(ctx, ql, num_q_heads=8 * g, num_kv_heads=8, head_dim=128,
                             seed=1191 + it, pool_factor=1.2)
        run(w, 0.0113, 0.0127, f"fp8 token-major random batch {it}")


def test_token_major_two_ctas_per_sm_llama8b(decode_tc_option):
    # the Llama-8B batch (G 4) on two CTAs per SM (304 workers on 152 SMs,
    # the default): every row against the oracle, and close to the
    # one-CTA-per-SM result
    w = wl.make_config(2)
    decode_tc_option("decode_tm_ctas_per_sm", 2)
    run(w, 0.0113, 0.0127, "llama8b fp8, token-major, two CTAs per SM")
    b = Fp8Batch(w, 0.0113, 0.0127)
    b.write()
    a = gu.to_f64(b.attend())
    decode_tc_option("decode_tm_ctas_per_sm", 1)
    c = gu.to_f64(b.attend())
    torch.cuda.synchronize()
    gu.check_no_device_error()
    assert np.abs(a - c).max() <= gu.MAX_ABS


def test_token_major_against_per_head_tiles(decode_tc_option):
    # the two tile shapes agree within the tolerance on the Llama-8B batch
    w = wl.make_config(2)
    b = Fp8Batch(w, 0.0113, 0.0127)
    b.write()
    a = gu.to_f64(b.attend())
    decode_tc_option("decode_token_major", 0)
    c = gu.to_f64(b.attend())
    torch.cuda.synchronize()
    gu.check_no_device_error()
    assert np.abs(a - c).max() <= gu.MAX_ABS


def test_attention_fp8_extreme_query_rows(decode_tc_option):
    # query rows with large, tiny and zero magnitudes: each row's power-of-two
    # scale keeps its split exact
    w = wl.make_workload([300, 700, 40], [1, 1, 1], num_q_heads=32, num_kv_heads=8,
                         head_dim=128, seed=1171)
    q = wl.bf16_bits_to_f32(w.q).copy()
    q[0] *= 1e3
    q[1, :8] *= 1e-4
    q[2, 3] = 0.0
    w.q = wl.to_bf16_bits(q.astype(np.float32))
    w.scale = 1.0 / 128.0 / 30.0
    decode_tc_option("decode_tc", 2)
    run(w, 0.0113, 0.0127, "fp8 tc extreme q rows")


def test_mixed_batch_fp8_sampled():
    w = wl.make_config(3)
    R = w.num_reqs
    run(w, 0.0113, 0.0127, "mixed fp8", reqs=[0, 255, 511, R - 3, R - 1])


def test_fp8_close_to_bf16_at_unit_scale():
    """Sanity on the quantisation itself: at the pages' default scale 1.0 the
    FP8 result stays near the bf16 one (E4M3 keeps 3 mantissa bits)."""
    w = wl.make_workload([500, 900], [1, 1], num_q_heads=32, num_kv_heads=8, head_dim=128,
                         seed=1130)
    ref16 = gu.to_f64(gu.DeviceBatch(w).step())
    b = Fp8Batch(w, 1.0, 1.0)
    assert (b.kc_cpu[np.isnan(wl.bf16_bits_to_f32(w.k_cache))] == E4M3_NAN).all()  # sentinels
    b.write()
    got8 = gu.to_f64(b.attend())
    torch.cuda.synchronize()
    assert np.abs(got8 - ref16).max() < 0.1


def test_bad_scales_rejected():
    w = wl.make_workload([10], [1], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=1140)
    b = Fp8Batch(w, 1.0, 1.0)
    for ks, vs in [(0.0, 1.0), (1.0, -1.0), (float("inf"), 1.0), (float("nan"), 1.0)]:
        with pytest.raises(binding.PagedAttentionError) as e:
            binding.write_kv_fp8(b.k, b.v, b.sm, b.kc, b.vc, ks, vs)
        assert e.value.status == -1
        with pytest.raises(binding.PagedAttentionError) as e:
            binding.attention_fp8(b.q, b.kc, b.vc, b.bt, b.sl, b.qsl, w.scale, ks, vs,
                                  max_query_len=1, max_seq_len=w.max_seq_len)
        assert e.value.status == -1
