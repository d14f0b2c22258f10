"""Scheduler-driven steps on the GPU: the host runtime (block pool, prefix
cache, token-budget scheduler) produces each step's metadata, the library's
kernels write the new K/V and run attention, and every step is checked
against the oracle.

K/V at a position are a deterministic function of the request's token
prefix up to it (a stand-in for a model layer), so a prefix-cache hit is
correct exactly when the hit blocks hold the K/V the request would have
computed itself. After every step the test reads the cache back and checks
that, position by position, for every scheduled request.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from paged_kv_cache_42_gb300 import binding, host
from paged_kv_cache_42_gb300 import workloads as wl

from tests.gpu_util import assert_close, bf16_tensor, check_no_device_error, to_bits, to_f64

pytestmark = pytest.mark.gpu

NAN_BITS = 0x7FC0
MASK = (1 << 64) - 1


def _mix(h: int, token: int) -> int:
    """splitmix64 step over (previous state, token)."""
    z = (h ^ (token & 0xFFFFFFFF)) + 0x9E3779B97F4A7C15 & MASK
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9 & MASK
    z = (z ^ (z >> 27)) * 0x94D049BB133111EB & MASK
    return z ^ (z >> 31)


class Requests:
    """Token lists and prefix states of the test's requests."""

    def __init__(self, hkv: int, d: int):
        self.tokens, self.state = {}, {}
        self.hkv, self.d = hkv, d
        self._kv = {}

    def add(self, rid: int, prompt):
        self.tokens[rid] = list(prompt)
        self.state[rid] = []

    def prefix_state(self, rid: int, p: int) -> int:
        st = self.state[rid]
        while len(st) <= p:
            st.append(_mix(st[-1] if st else 0x243F6A8885A308D3, self.tokens[rid][len(st)]))
        return st[p]

    def kv(self, rid: int, p: int):
        key = self.prefix_state(rid, p)
        if key not in self._kv:
            g = np.random.default_rng(key)
            x = g.standard_normal((2, self.hkv, self.d)).astype(np.float32)
            self._kv[key] = wl.to_bf16_bits(x)
        return self._kv[key]


def _run_engine(seed: int, *, num_blocks: int, budget: int, steps: int, hq=16, hkv=4, d=128,
                max_len=1024, threshold=0):
    rng = np.random.default_rng(seed)
    bs = 16
    pool = host.BlockPool(num_blocks=num_blocks, block_size=bs)
    sched = host.Scheduler(pool, token_budget=budget, max_model_len=max_len,
                           long_prefill_threshold=threshold, prefix_caching=True)
    reqs = Requests(hkv, d)
    system = rng.integers(0, 50000, 96).tolist()  # a shared 6-block system prompt
    next_id = 0

    def add_some(n):
        nonlocal next_id
        for _ in range(n):
            plen = int(rng.integers(8, 320))
            body = rng.integers(0, 50000, plen).tolist()
            prompt = (system + body) if rng.random() < 0.6 else body
            prompt = prompt[:max_len // 2]
            reqs.add(next_id, prompt)
            sched.add_request(next_id, prompt)
            next_id += 1

    add_some(12)
    shape = (num_blocks, hkv, bs, d)
    kc_cpu = np.full(shape, NAN_BITS, np.uint16)
    vc_cpu = np.full(shape, NAN_BITS, np.uint16)
    kc = bf16_tensor(kc_cpu)
    vc = bf16_tensor(vc_cpu)
    scale = 1.0 / np.sqrt(d)
    stats = dict(hits=0, preempted=0, prefill_spans=0, decodes=0)
    for step in range(steps):
        live = list(reqs.tokens)
        running_before = {rid for rid in live if sched.request_state(rid)["running"]}
        out = sched.step()
        T, R = out["num_tokens"], len(out["req_ids"])
        if T == 0:
            add_some(4)
            continue
        stats["preempted"] += len(out["preempted_ids"])
        stats["hits"] += sum(1 for rid, c in zip(out["req_ids"], out["num_computed"])
                             if int(rid) not in running_before and c > 0)
        stats["prefill_spans"] += int(np.sum(out["num_scheduled"] >= 16))
        stats["decodes"] += out["num_decode_reqs"]
        # new K/V for the scheduled positions, q at random
        k_new = np.empty((T, hkv, d), np.uint16)
        v_new = np.empty((T, hkv, d), np.uint16)
        t = 0
        for rid, n, ctx in zip(out["req_ids"], out["num_scheduled"], out["num_computed"]):
            for j in range(int(n)):
                kv = reqs.kv(int(rid), int(ctx) + j)
                k_new[t], v_new[t] = kv[0], kv[1]
                t += 1
        q = wl.to_bf16_bits(rng.standard_normal((T, hq, d)).astype(np.float32))
        dev = lambda a: torch.from_numpy(np.ascontiguousarray(a)).cuda()
        binding.write_kv(bf16_tensor(k_new), bf16_tensor(v_new), dev(out["slot_mapping"]), kc, vc)
        got = binding.attention(bf16_tensor(q), kc, vc, dev(out["block_tables"]),
                                dev(out["seq_lens"]), dev(out["query_start_loc"]), scale,
                                max_query_len=out["max_query_len"],
                                max_seq_len=out["max_seq_len"])
        torch.cuda.synchronize()
        check_no_device_error()
        # oracle on the CPU copy of the caches
        oracle.write_kv(k_new, v_new, out["slot_mapping"], kc_cpu, vc_cpu)
        assert np.array_equal(to_bits(kc), kc_cpu) and np.array_equal(to_bits(vc), vc_cpu), \
            f"step {step}: cache differs from the oracle's scatter"
        ref = oracle.attention(q, kc_cpu, vc_cpu, out["block_tables"], out["seq_lens"],
                               out["query_start_loc"], scale)
        assert_close(to_f64(got), ref, f"engine step {step}")
        # every position a scheduled request attends to holds its own K/V
        for r, rid in enumerate(out["req_ids"]):
            for p in range(int(out["seq_lens"][r])):
                blk = int(out["block_tables"][r][p // bs])
                kv = reqs.kv(int(rid), p)
                assert np.array_equal(kc_cpu[blk, :, p % bs], kv[0]), (step, int(rid), p)
                assert np.array_equal(vc_cpu[blk, :, p % bs], kv[1]), (step, int(rid), p)
        # sample, finish, admit
        for r, rid in enumerate(out["req_ids"]):
            rid = int(rid)
            st = sched.request_state(rid)
            if st["num_computed"] == st["num_tokens"]:
                if st["num_tokens"] - st["prompt_len"] >= int(rng.integers(4, 40)) or \
                        st["num_tokens"] >= max_len:
                    sched.finish(rid)
                    del reqs.tokens[rid]
                else:
                    tok = int(rng.integers(0, 50000))
                    reqs.tokens[rid].append(tok)
                    sched.append_token(rid, tok)
        if rng.random() < 0.3:
            add_some(int(rng.integers(1, 5)))
    return stats


def test_engine_steps_match_oracle():
    s = _run_engine(5, num_blocks=400, budget=512, steps=24)
    assert s["hits"] > 0 and s["prefill_spans"] > 0 and s["decodes"] > 0, s


def test_engine_steps_with_preemption():
    s = _run_engine(9, num_blocks=90, budget=384, steps=30, threshold=160)
    assert s["preempted"] > 0, s
