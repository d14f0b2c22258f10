"""Pins of the oracle's FP8 (E4M3) KV-cache paths, with no GPU.

The pages fix the format (E4M3 with an fp32 per-tensor scale, "vLLM: An
Exhaustive Technical Study for Kernel Engineers", 2.8). The pins come from
outside the oracle:
  * code values that follow from the OCP 8-bit format definition
    (tests/golden/e4m3_codes.json);
  * brute force over all 256 codes: every finite code decodes and encodes
    back to itself;
  * the library routine torch.float8_e4m3fn for in-range values, ties
    included (round to nearest even);
  * attention over an E4M3 cache with a power-of-two scale equals, bit for
    bit, the (already pinned) bf16 attention oracle on the same values,
    which bf16 represents exactly;
  * the quantising scatter writes exactly the quantised rows at the slots
    and leaves every other slot alone.
Planted mistakes (rounding toward zero, a wrong exponent bias) must fail a pin.
"""
from __future__ import annotations

import json
import os

import numpy as np
import pytest

import oracle
from paged_kv_cache_42_gb300 import workloads as wl

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "e4m3_codes.json")))
torch = pytest.importorskip("torch")


def pin_golden_codes(lib):
    for c, v in GOLD["values"]:
        got = oracle.e4m3_value(int(c, 16), lib=lib)
        assert got == v, (c, got, v)
    for c in GOLD["nan_codes"]:
        assert np.isnan(oracle.e4m3_value(int(c, 16), lib=lib))


def pin_round_trip(lib):
    for c in range(256):
        if c in (0x7F, 0xFF):
            continue
        v = oracle.e4m3_value(c, lib=lib)
        assert oracle.e4m3_encode(v, lib=lib) == c, c


def pin_against_torch(lib):
    rng = np.random.default_rng(17)
    mag = np.exp(rng.uniform(np.log(2.0 ** -12), np.log(440.0), 4000))
    x = (mag * rng.choice([-1.0, 1.0], 4000)).astype(np.float32)
    # exact midpoints between neighbouring codes: ties go to the even code
    finite = [oracle.e4m3_value(c, lib=lib) for c in range(0x00, 0x7E)]
    mids = np.array([(a + b) / 2 for a, b in zip(finite[:-1], finite[1:])], np.float32)
    x = np.concatenate([x, mids, -mids])
    ours = np.array([oracle.e4m3_encode(float(v), lib=lib) for v in x], np.uint8)
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours, ref)


def pin_saturation(lib):
    for y in (448.0, 460.0, 470.0, 1000.0, 3.0e38):
        assert oracle.e4m3_encode(y, lib=lib) == 0x7E
        assert oracle.e4m3_encode(-y, lib=lib) == 0xFE
    assert oracle.e4m3_encode(0.0, lib=lib) == 0x00
    assert oracle.e4m3_encode(2.0 ** -11, lib=lib) == 0x00   # below half the least subnormal
    assert oracle.e4m3_encode(2.0 ** -10, lib=lib) == 0x00   # a tie: to even (zero)
    assert oracle.e4m3_encode(3 * 2.0 ** -10, lib=lib) == 0x02  # a tie between 1 and 2: to 2


def pin_fp8_attention_equals_bf16(lib):
    """Power-of-two scales make code * scale exact in bf16: both oracle paths
    then see the same float64 keys and values."""
    rng = np.random.default_rng(23)
    w = wl.make_workload([30, 70, 5], [1, 4, 1], num_q_heads=8, num_kv_heads=2, head_dim=64,
                         seed=901, pool_factor=1.5)
    ks, vs = 2.0 ** -3, 2.0 ** 2
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    kc8 = rng.choice(finite[np.abs([oracle.e4m3_value(c, lib=lib) for c in finite]) <= 8.0],
                     size=w.k_cache.shape).astype(np.uint8)
    vc8 = rng.choice(finite, size=w.v_cache.shape).astype(np.uint8)

    def as_bf16(codes, scale):
        vals = np.vectorize(lambda c: oracle.e4m3_value(int(c), lib=lib))(codes) * scale
        return wl.to_bf16_bits(vals.astype(np.float32))

    kb, vb = as_bf16(kc8, ks), as_bf16(vc8, vs)
    assert np.array_equal(wl.bf16_bits_to_f32(kb).astype(np.float64),
                          np.vectorize(lambda c: oracle.e4m3_value(int(c), lib=lib))(kc8) * ks)
    a = oracle.attention_fp8(w.q, kc8, vc8, ks, vs, w.block_tables, w.seq_lens,
                             w.query_start_loc, w.scale, lib=lib)
    b = oracle.attention(w.q, kb, vb, w.block_tables, w.seq_lens, w.query_start_loc, w.scale,
                         lib=lib)
    assert np.array_equal(a, b)


def pin_quantising_scatter(lib):
    w = wl.make_workload([3, 20], [2, 5], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=902,
                         pool_factor=2.0)
    nb, hkv, bs, d = w.k_cache.shape
    kc = np.full((nb, hkv, bs, d), 0x7F, np.uint8)
    vc = kc.copy()
    sm = w.slot_mapping.copy()
    sm[1] = -1  # a padding token
    oracle.write_kv_fp8(w.k_new, w.v_new, sm, kc, vc, 0.05, 0.07, lib=lib)
    touched = np.zeros((nb, bs), bool)
    for t, s in enumerate(sm):
        if s < 0:
            continue
        b, o = divmod(int(s), bs)
        touched[b, o] = True
        for h in range(hkv):
            assert np.array_equal(kc[b, h, o], oracle.e4m3_quantize(w.k_new[t, h], 0.05, lib=lib))
            assert np.array_equal(vc[b, h, o], oracle.e4m3_quantize(w.v_new[t, h], 0.07, lib=lib))
    untouched = ~touched
    assert (kc.transpose(0, 2, 1, 3)[untouched] == 0x7F).all()
    assert (vc.transpose(0, 2, 1, 3)[untouched] == 0x7F).all()


def pin_quotient_in_binary32(lib):
    """code = E4M3(binary32(x / scale)): checked against torch doing the same
    binary32 division, then its own conversion."""
    rng = np.random.default_rng(29)
    x = wl.to_bf16_bits(rng.standard_normal(5000).astype(np.float32))
    for scale in (1.0, 0.0113, 0.3, 7.0):
        ours = oracle.e4m3_quantize(x, scale, lib=lib)
        q = torch.from_numpy(wl.bf16_bits_to_f32(x)) / torch.tensor(scale, dtype=torch.float32)
        q = q.clamp(-448.0, 448.0)
        ref = q.to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(ours, ref), scale


PINS = [pin_golden_codes, pin_round_trip, pin_against_torch, pin_saturation,
        pin_fp8_attention_equals_bf16, pin_quantising_scatter, pin_quotient_in_binary32]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_fp8_pin(pin, oracle_lib):
    pin(oracle_lib)


@pytest.mark.parametrize("mutant", [8, 9])
def test_fp8_pins_catch_planted_mistakes(mutant, tmp_path):
    lib = oracle.load(mutant=mutant, out_dir=str(tmp_path))
    assert lib.oracle_mutant_id() == mutant
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError):
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
