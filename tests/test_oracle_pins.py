"""Pins for the CPU oracle: what the pages and the mathematics fix, checked
against the oracle without any reference to the CUDA path.

Each ``pin_*`` function takes the oracle library handle so the mutation test
at the end can run every pin against deliberately broken builds of the oracle
and show that each planted mistake fails at least one pin.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import scipy.special

import oracle
from paged_kv_cache_42_gb300 import workloads as wl
from tests import brute

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "pages_examples.json")


def _f32(bits):
    return wl.bf16_bits_to_f32(bits).astype(np.float64)


def _run(w, lib, **kw):
    return oracle.attention(w.q, w.k_cache, w.v_cache, w.block_tables, w.seq_lens,
                            w.query_start_loc, w.scale, lib=lib, threads=4, **kw)


def _write_new_tokens(w, lib):
    oracle.write_kv(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache, lib=lib)
    return w


def _contiguous_case(ctx, ql, hq, hkv, d, seed, pool_factor=2.0):
    """Draws contiguous per-request K/V, then pages them through random block
    tables with a plain test-side scatter (no oracle code involved)."""
    w = wl.make_workload(ctx, ql, num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=seed,
                         pool_factor=pool_factor, fill_values=False)
    rng = np.random.Generator(np.random.PCG64(seed + 7))
    T = w.num_tokens
    w.q[...] = wl.to_bf16_bits(rng.standard_normal((T, hq, d), dtype=np.float32))
    seqs = []
    for r in range(w.num_reqs):
        L = int(w.seq_lens[r])
        K = wl.to_bf16_bits(rng.standard_normal((L, hkv, d), dtype=np.float32))
        V = wl.to_bf16_bits(rng.standard_normal((L, hkv, d), dtype=np.float32))
        for p in range(L):
            b = w.block_tables[r, p // 16]
            w.k_cache[b, :, p % 16, :] = K[p]
            w.v_cache[b, :, p % 16, :] = V[p]
        seqs.append((K, V))
    return w, seqs


# --------------------------------------------------------------------------
# pins on the generator / metadata (values the pages print)
# --------------------------------------------------------------------------
def test_golden_block_counts():
    g = json.load(open(GOLDEN))
    for ex in g["blocks_for_tokens"]:
        w = wl.make_workload([ex["tokens"] - 1], [1], num_q_heads=1, num_kv_heads=1,
                             head_dim=64, seed=1, fill_values=False)
        assert int((w.block_tables[0] >= 0).sum()) == ex["blocks"]
    for ex in g["full_blocks_for_prompt"]:
        w = wl.make_workload([0], [ex["tokens"]], num_q_heads=1, num_kv_heads=1, head_dim=64,
                             seed=2, fill_values=False)
        used = int((w.block_tables[0] >= 0).sum())
        assert used - 1 == ex["full_blocks"]
        assert (used - 1) * 16 == ex["tokens_in_full_blocks"]
        assert ex["tokens"] - (used - 1) * 16 == ex["tail_tokens"]


def test_golden_query_start_loc():
    g = json.load(open(GOLDEN))
    for ex in g["query_start_loc"]:
        n = ex["scheduled_tokens"]
        w = wl.make_workload([0] * len(n), n, num_q_heads=1, num_kv_heads=1, head_dim=64,
                             seed=3, fill_values=False)
        assert w.query_start_loc.tolist() == ex["query_start_loc"]
        if "last_row_per_request" in ex:
            assert (w.query_start_loc[1:] - 1).tolist() == ex["last_row_per_request"]


def test_waste_at_most_one_partial_block():
    g = json.load(open(GOLDEN))["waste_bound"]
    for idx in (1, 2, 3, 4):
        w = wl.make_config(idx, fill_values=False)
        nb = (w.block_tables >= 0).sum(axis=1)
        waste = nb * 16 - w.seq_lens
        assert (waste >= 0).all() and (waste <= g["max_waste_tokens_per_sequence"]).all()
        assert waste.sum() < w.num_reqs * 16


def test_config1_block_assignment():
    w = wl.make_config(1, fill_values=False)
    nb = (w.block_tables >= 0).sum(axis=1)
    assert nb.tolist() == [1, 4, 2, 3] and nb.sum() == 10
    assert w.num_blocks == 32
    ids = w.block_tables[w.block_tables >= 0]
    assert len(set(ids.tolist())) == 10  # a permutation prefix: distinct ids


def test_slot_mapping_points_at_the_token_position():
    w = wl.make_config(3, fill_values=False)
    for r in (0, 100, 512, 513, 514):
        for j in range(int(w.q_lens[r])):
            p = int(w.ctx_lens[r]) + j
            s = int(w.slot_mapping[w.query_start_loc[r] + j])
            assert s // 16 == w.block_tables[r, p // 16] and s % 16 == p % 16


def test_generator_pool_and_tables():
    for idx in (2, 4, 5):
        w = wl.make_config(idx, fill_values=False)
        ids = w.block_tables[w.block_tables >= 0]
        assert ids.min() >= 0 and ids.max() < w.num_blocks
        if idx == 4:
            assert (w.block_tables[:, :64] == w.block_tables[0, :64]).all()
            priv = w.block_tables[:, 64:]
            priv = priv[priv >= 0]
            assert len(set(priv.tolist())) == priv.size
            assert not set(priv.tolist()) & set(w.block_tables[0, :64].tolist())
        else:
            assert len(set(ids.tolist())) == ids.size
        if idx == 5:
            assert w.num_blocks == 16384 and ids.size == 16384


# --------------------------------------------------------------------------
# pins on the oracle's arithmetic
# --------------------------------------------------------------------------
def pin_brute_force(lib):
    cases = [
        ([8, 55, 16, 32], [1, 1, 1, 1], 4, 2, 64, 11),       # config-1 shaped decode
        ([0, 5, 20], [7, 3, 18], 4, 1, 16, 12),             # chunks on prefixes, MQA
        ([3, 0], [1, 17], 8, 2, 32, 13),                    # chunk crossing a block edge
        ([40], [2], 2, 2, 16, 14),                          # MHA (G=1), 2-token verify span
    ]
    for ctx, ql, hq, hkv, d, seed in cases:
        w, seqs = _contiguous_case(ctx, ql, hq, hkv, d, seed)
        got = _run(w, lib)
        for r, (K, V) in enumerate(seqs):
            q0, q1 = int(w.query_start_loc[r]), int(w.query_start_loc[r + 1])
            qrows = [[_f32(w.q[t, h]).tolist() for h in range(hq)] for t in range(q0, q1)]
            kseq = [[_f32(K[p, h]).tolist() for h in range(hkv)] for p in range(K.shape[0])]
            vseq = [[_f32(V[p, h]).tolist() for h in range(hkv)] for p in range(V.shape[0])]
            ref = brute.attention(qrows, kseq, vseq, int(w.ctx_lens[r]), hkv, w.scale)
            np.testing.assert_allclose(got[q0:q1], np.array(ref), rtol=1e-12, atol=1e-13)


def pin_single_key_returns_its_value(lib):
    w = wl.make_workload([0, 0], [1, 1], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=21)
    _write_new_tokens(w, lib)
    got = _run(w, lib)
    for t in range(2):
        for h in range(4):
            assert np.array_equal(got[t, h], _f32(w.v_new[t, h // 2]))


def pin_equal_keys_average_values(lib):
    w = wl.make_workload([37, 5], [1, 9], num_q_heads=4, num_kv_heads=2, head_dim=64, seed=22)
    _write_new_tokens(w, lib)
    # make every key of every request identical: all scores tie
    valid = ~np.isnan(wl.bf16_bits_to_f32(w.k_cache))
    w.k_cache[valid] = wl.to_bf16_bits(np.float32(0.75))
    got = _run(w, lib)
    for r in range(2):
        for j in range(int(w.q_lens[r])):
            t = int(w.query_start_loc[r]) + j
            last = int(w.ctx_lens[r]) + j
            for h in range(4):
                vals = np.array([_f32(w.v_cache[w.block_tables[r, p // 16], h // 2, p % 16])
                                 for p in range(last + 1)])
                np.testing.assert_allclose(got[t, h], vals.mean(axis=0), rtol=1e-12, atol=1e-14)


def pin_zero_query_averages_values(lib):
    w = wl.make_workload([20], [1], num_q_heads=2, num_kv_heads=1, head_dim=64, seed=23)
    _write_new_tokens(w, lib)
    w.q[...] = 0
    got = _run(w, lib)
    vals = np.array([_f32(w.v_cache[w.block_tables[0, p // 16], 0, p % 16]) for p in range(21)])
    for h in range(2):
        np.testing.assert_allclose(got[0, h], vals.mean(axis=0), rtol=1e-12, atol=1e-14)


def pin_two_keys_logistic(lib):
    # two keys: the weight of key 1 is the logistic function of the score gap
    w = wl.make_workload([1], [1], num_q_heads=1, num_kv_heads=1, head_dim=64, seed=24)
    _write_new_tokens(w, lib)
    got = _run(w, lib)[0, 0]
    q = _f32(w.q[0, 0])
    k0 = _f32(w.k_cache[w.block_tables[0, 0], 0, 0]); v0 = _f32(w.v_cache[w.block_tables[0, 0], 0, 0])
    k1 = _f32(w.k_new[0, 0]); v1 = _f32(w.v_new[0, 0])
    gap = w.scale * (float(q @ k1) - float(q @ k0))
    a = scipy.special.expit(gap)
    np.testing.assert_allclose(got, (1 - a) * v0 + a * v1, rtol=1e-12, atol=1e-14)


def pin_causal_chunk_is_textbook(lib):
    # ctx = 0, qlen = L: plain causal self-attention over a contiguous sequence
    hq, hkv, d, L = 4, 2, 32, 37
    w = wl.make_workload([0], [L], num_q_heads=hq, num_kv_heads=hkv, head_dim=d, seed=25)
    _write_new_tokens(w, lib)
    got = _run(w, lib)
    Q = _f32(w.q)                   # [L, hq, d]
    K = _f32(w.k_new); V = _f32(w.v_new)
    mask = np.triu(np.ones((L, L), bool), k=1)
    for h in range(hq):
        S = w.scale * (Q[:, h, :] @ K[:, h // 2, :].T)
        S[mask] = -np.inf
        P = scipy.special.softmax(S, axis=1)
        np.testing.assert_allclose(got[:, h, :], P @ V[:, h // 2, :], rtol=1e-11, atol=1e-13)


def pin_permutation_invariance(lib):
    w = wl.make_workload([30, 0, 70], [1, 12, 5], num_q_heads=4, num_kv_heads=2, head_dim=64,
                         seed=26, pool_factor=1.5)
    _write_new_tokens(w, lib)
    a = _run(w, lib)
    b = _run(wl.permute_physical_blocks(w, seed=99), lib)
    assert np.array_equal(a, b)


def pin_shared_prefix_equals_private_copies(lib):
    w = wl.make_workload([40, 33, 60], [1, 1, 1], num_q_heads=4, num_kv_heads=2, head_dim=64,
                         seed=27, shared_prefix_blocks=2)
    _write_new_tokens(w, lib)
    a = _run(w, lib)
    b = _run(wl.unshare_prefix(w, seed=5), lib)
    assert np.array_equal(a, b)


def pin_mixed_batch_is_union(lib):
    w = wl.make_workload([15, 16, 17, 0, 31], [1, 1, 1, 20, 9], num_q_heads=4, num_kv_heads=1,
                         head_dim=64, seed=28)
    _write_new_tokens(w, lib)
    a = _run(w, lib)
    dec = wl.subset_requests(w, [0, 1, 2])
    pre = wl.subset_requests(w, [3, 4])
    b = np.concatenate([_run(dec, lib), _run(pre, lib)])
    assert np.array_equal(a, b)


def pin_write_scatter(lib):
    w = wl.make_workload([3, 30, 0], [1, 4, 18], num_q_heads=4, num_kv_heads=2, head_dim=64,
                         seed=29, pool_factor=2.0)
    kc0, vc0 = w.k_cache.copy(), w.v_cache.copy()
    sm = w.slot_mapping.copy()
    sm[2] = -1  # a padding token: skipped
    oracle.write_kv(w.k_new, w.v_new, sm, w.k_cache, w.v_cache, lib=lib)
    touched = np.zeros(w.k_cache.shape[:1] + w.k_cache.shape[2:3], bool)  # [blocks, bs]
    for t, s in enumerate(sm):
        if s < 0:
            continue
        touched[s // 16, s % 16] = True
        assert np.array_equal(w.k_cache[s // 16, :, s % 16, :], w.k_new[t])
        assert np.array_equal(w.v_cache[s // 16, :, s % 16, :], w.v_new[t])
    untouched = ~touched
    assert np.array_equal(w.k_cache.transpose(0, 2, 1, 3)[untouched],
                          kc0.transpose(0, 2, 1, 3)[untouched])
    assert np.array_equal(w.v_cache.transpose(0, 2, 1, 3)[untouched],
                          vc0.transpose(0, 2, 1, 3)[untouched])
    assert touched.sum() == int((sm >= 0).sum())
    bad = sm.copy()
    bad[0] = w.num_blocks * 16
    with pytest.raises(oracle.OracleError):
        oracle.write_kv(w.k_new, w.v_new, bad, w.k_cache, w.v_cache, lib=lib)


PINS = [pin_brute_force, pin_single_key_returns_its_value, pin_equal_keys_average_values,
        pin_zero_query_averages_values, pin_two_keys_logistic, pin_causal_chunk_is_textbook,
        pin_permutation_invariance, pin_shared_prefix_equals_private_copies,
        pin_mixed_batch_is_union, pin_write_scatter]


@pytest.mark.parametrize("pin", PINS, ids=lambda f: f.__name__)
def test_pin(pin, oracle_lib):
    pin(oracle_lib)


def test_oracle_never_reads_unused_slots(oracle_lib):
    # every unused slot holds NaN; a finite result shows only valid KV was read
    for idx in (1,):
        w = wl.make_config(idx)
        oracle.write_kv(w.k_new, w.v_new, w.slot_mapping, w.k_cache, w.v_cache, lib=oracle_lib)
        out = _run(w, oracle_lib)
        assert np.isfinite(out).all()


# Each mutant plants one plausible mistake in the oracle (see ORACLE_MUTANT in
# pa_oracle.c): 1 causal off-by-one, 2 wrong GQA mapping, 3 transposed
# operand, 4 dropped scale, 5 swapped block index / offset, 6 no causal mask
# inside a chunk, 7 dropped normaliser.
@pytest.mark.parametrize("mutant", [1, 2, 3, 4, 5, 6, 7])
def test_pins_catch_planted_mistakes(mutant, tmp_path):
    lib = oracle.load(mutant=mutant, out_dir=str(tmp_path))
    assert lib.oracle_mutant_id() == mutant
    caught = []
    for pin in PINS:
        try:
            pin(lib)
        except (AssertionError, oracle.OracleError, FloatingPointError):
            caught.append(pin.__name__)
    assert caught, f"mutant {mutant} passed every pin"
