"""Host runtime: block pool, chained block hash, prefix lookup and the
token-budget scheduler. CPU only.

Three layers of checks:
  * the pages' printed worked examples (tests/golden/pages_host_examples.json)
    run on both the oracle model (oracle/host_ref.py) and the library's C++
    runtime, and planted mistakes in the oracle must break them;
  * invariants that hold for any correct pool and scheduler (reference counts
    equal table occurrences, the free queue holds exactly the unreferenced
    blocks, every computed position of a running request finds its own token
    in the cache, prefix hits included, the budget is never exceeded);
  * random operation sequences run through both sides must agree exactly,
    step by step, on every metadata array and on the pool's state.
"""
from __future__ import annotations

import collections
import hashlib
import json
import os

import numpy as np
import pytest

from oracle import host_ref

HERE = os.path.dirname(os.path.abspath(__file__))
GOLD = json.load(open(os.path.join(HERE, "golden", "pages_host_examples.json")))


@pytest.fixture(scope="module")
def host():
    from paged_kv_cache_42_gb300 import build, host as h
    build.build()
    return h


# ----------------------------------------------------------------- adapters

class OracleSide:
    name = "oracle"

    def __init__(self, ref=host_ref):
        self.ref = ref

    def pool(self, ids, bs):
        return self.ref.Pool(ids, bs)

    def refs(self, pool, b):
        return pool.refs[b]

    def cached(self, pool, b):
        return b in pool.hash_of

    def free(self, pool):
        return list(pool.free)

    def scheduler(self, pool, **kw):
        return self.ref.Scheduler(pool, **kw)

    def reusable(self, *a):
        return self.ref.reusable_tokens(*a)


class LibrarySide:
    name = "library"

    def __init__(self, h):
        self.h = h

    def pool(self, ids, bs):
        return self.h.BlockPool(ids=ids, block_size=bs)

    def refs(self, pool, b):
        return pool.ref_count(b)

    def cached(self, pool, b):
        return pool.is_cached(b)

    def free(self, pool):
        return pool.free_queue()

    def scheduler(self, pool, **kw):
        return self.h.Scheduler(pool, **kw)

    def reusable(self, *a):
        return self.h.reusable_tokens(*a)


@pytest.fixture(params=["oracle", "library"])
def side(request):
    if request.param == "oracle":
        return OracleSide()
    return LibrarySide(request.getfixturevalue("host"))


def label_hash(label: str) -> bytes:
    return hashlib.sha256(label.encode()).digest()


# ---------------------------------------------------- pages' worked examples

def run_free_queue_example(side):
    g = GOLD["free_queue_example"]
    ids = [12, 41, 73, 90]
    pool = side.pool(ids, g["block_size"])
    assert pool.allocate(4) == ids  # the figure's four live slots
    pool.touch([12])                # R1 shares R0's first block
    for b, lab in g["hashes"].items():
        pool.cache_block(int(b), label_hash(lab))
    tables = {k: list(v) for k, v in g["tables"].items()}
    before = ({b: side.refs(pool, b) for b in ids}, side.free(pool),
              {b: side.cached(pool, b) for b in ids})
    with pytest.raises(MemoryError):
        pool.allocate(1)
    after = ({b: side.refs(pool, b) for b in ids}, side.free(pool),
             {b: side.cached(pool, b) for b in ids})
    assert after == before
    pool.release(tables.pop("R0"))
    assert side.refs(pool, 12) == 1 and side.free(pool) == [41]
    assert side.cached(pool, 41)
    tables["R2"] = pool.allocate(1)
    assert tables["R2"] == g["expect"]["R2_allocates"] and not side.cached(pool, 41)
    counts = collections.Counter(b for t in tables.values() for b in t)
    assert {b: side.refs(pool, b) for b in ids} == {b: counts.get(b, 0) for b in ids}
    pool.release(tables.pop("R1"))
    assert side.free(pool) == g["expect"]["after_release_R1"]["free"]
    assert side.refs(pool, 41) == g["expect"]["after_release_R1"]["ref_41"]


def test_free_queue_example(side):
    run_free_queue_example(side)


def run_head_tail_rule(side):
    """The release rule with a non-empty queue ("Deep Dive - vLLM", "Block
    pool, prefix cache, and eviction": cached blocks to the tail, non-cached
    ones to the head for earlier reuse). In the printed example the queue is
    empty when the uncached block is released, so it cannot tell the two
    apart."""
    pool = side.pool([0, 1, 2, 3], 4)
    a, b = pool.allocate(2)
    pool.cache_block(a, label_hash("ABCD"))
    pool.release([a])
    assert side.free(pool) == [2, 3, a]
    pool.release([b])
    assert side.free(pool) == [b, 2, 3, a]
    assert pool.allocate(1) == [b] and side.cached(pool, a)


def test_head_tail_rule(side):
    run_head_tail_rule(side)


def run_reusable(side):
    g = GOLD["reusable_tokens"]
    for shared, length, want in g["cases"]:
        assert side.reusable(shared, length, g["block_size"]) == want, (shared, length)
    for args in g["invalid"]:
        with pytest.raises((ValueError, RuntimeError)):
            side.reusable(*args)


def test_reusable_tokens(side):
    run_reusable(side)


def test_reusable_tokens_rejects_non_integers():
    for args in [(6.5, 9, 4), (6, 9, True)]:
        with pytest.raises(ValueError):
            host_ref.reusable_tokens(*args)


def toks(s: str) -> list:
    return [ord(c) for c in s]


def drive(sched, steps: int, on_step=None) -> list:
    """Run steps; after each, every request whose tokens are all computed
    gets a sampled token (its id + 1000, deterministic)."""
    outs = []
    for _ in range(steps):
        out = sched.step()
        outs.append(out)
        for rid in list(out["req_ids"]):
            st = state(sched, int(rid))
            if st["num_computed"] == st["num_tokens"]:
                sched.append_token(int(rid), 1000 + int(rid))
        if on_step:
            on_step(out)
    return outs


def state(sched, rid: int) -> dict:
    if hasattr(sched, "request_state"):
        return sched.request_state(rid)
    r = sched.reqs[rid]
    return dict(num_computed=r.num_computed, num_tokens=len(r.tokens), prompt_len=r.prompt_len,
                num_blocks=len(r.blocks), running=int(r.running))


def trace_rows(outs, prompt_len_r1: int) -> dict:
    rows = dict(r0_decode=[], r1_prefill=[], r1_decode=[], used=[])
    for out in outs:
        grant = {int(r): (int(n), int(c)) for r, n, c in
                 zip(out["req_ids"], out["num_scheduled"], out["num_computed"])}
        n0 = grant.get(0, (0, 0))[0]
        n1, c1 = grant.get(1, (0, 0))
        rows["r0_decode"].append(n0)
        rows["r1_prefill"].append(n1 if c1 < prompt_len_r1 else 0)
        rows["r1_decode"].append(n1 if c1 >= prompt_len_r1 else 0)
        rows["used"].append(int(sum(out["num_scheduled"])))
    return rows


def run_budget_trace(side):
    g = GOLD["token_budget_trace"]
    pool = side.pool(list(range(64)), 4)
    s = side.scheduler(pool, token_budget=g["budget"], max_model_len=64, prefix_caching=False)
    s.add_request(0, toks("XYZ"))
    drive(s, 1)                      # R0's prompt; it is decoding from now on
    s.add_request(1, toks("ABCDEFXYZ"))
    rows = trace_rows(drive(s, 3), 9)
    for k in ("r0_decode", "r1_prefill", "r1_decode", "used"):
        assert rows[k] == g[k], (k, rows[k])


def test_token_budget_trace(side):
    run_budget_trace(side)


def run_apc_trace(side):
    g, a = GOLD["token_budget_trace"], GOLD["apc_example"]
    pool = side.pool(list(range(64)), a["block_size"])
    s = side.scheduler(pool, token_budget=g["budget"], max_model_len=64, prefix_caching=True)
    s.add_request(0, toks(a["r0_prompt"]))
    drive(s, 2)                      # 6 + 2 prompt tokens: ABCD and EFGH cached
    assert state(s, 0)["num_tokens"] == 9
    s.add_request(1, toks(a["r1_prompt"]))
    out = drive(s, 1)[0]
    grant = dict(zip(map(int, out["req_ids"]), map(int, out["num_scheduled"])))
    ctx = dict(zip(map(int, out["req_ids"]), map(int, out["num_computed"])))
    assert ctx[1] == a["r1_cached_tokens"] and grant[1] == a["r1_prefill_tokens"]
    assert grant[1] == g["with_prefix_caching"]["r1_prefill_step0"]
    assert sum(grant.values()) == g["with_prefix_caching"]["used_step0"]
    # R1 shares R0's first block (one reference each)
    b0 = int(out["block_tables"][list(map(int, out["req_ids"])).index(1)][0])
    b0_r0 = int(out["block_tables"][list(map(int, out["req_ids"])).index(0)][0])
    assert b0 == b0_r0 and side.refs(pool, b0) == 2


def test_prefix_caching_trace(side):
    run_apc_trace(side)


def test_lookup_stops_at_first_miss(side):
    """A chained hash cannot match past a missing parent ("vLLM v1 Deep Dive",
    Part 3, Step 3: the longest-prefix scan stops at the first miss)."""
    bs = 4
    pool = side.pool([0, 1, 2, 3], bs)
    a, b = pool.allocate(2)
    h0 = host_ref.block_hash(None, toks("ABCD"))
    h1 = host_ref.block_hash(h0, toks("EFGH"))
    pool.cache_block(a, h0)
    pool.cache_block(b, h1)
    assert pool.find_cached_prefix(toks("ABCDEFGHJ")) == [a, b]
    assert pool.find_cached_prefix(toks("ABCDEFGH")) == [a]  # one position left to compute
    pool.release([b, a])  # a, then b, to the tail: free = [2, 3, a, b]
    taken = pool.allocate(3)  # evicts a (ABCD); b (its child) stays cached
    assert taken[-1] == a and side.cached(pool, b) and not side.cached(pool, a)
    assert pool.find_cached_prefix(toks("ABCDEFGHJ")) == []
    pool.release(taken)


def _signature(out) -> str:
    return (f"execute_context_{out['num_context_reqs']}({out['num_context_tokens']})"
            f"_generation_{out['num_generation_reqs']}({out['num_generation_tokens']})")


@pytest.mark.parametrize("ex", range(len(GOLD["step_signature"]["examples"])))
def test_step_signature_examples(side, ex):
    """The pages' printed step annotations, reproduced by scheduling the
    batches they describe: decoding requests first, then whole prompts."""
    g = GOLD["step_signature"]["examples"][ex]
    prompts, n_gen = g["context_prompts"], g["decodes"]
    pool = side.pool(list(range(2000)), 16)
    s = side.scheduler(pool, token_budget=sum(prompts) + n_gen + 64, max_model_len=2048,
                       prefix_caching=False)
    for i in range(n_gen):
        s.add_request(i, [i + 1] * 3)
    drive(s, 1)  # their prompts are computed; each now decodes
    for j, n in enumerate(prompts):
        s.add_request(1000 + j, [7 + j] * n)
    out = s.step()
    assert _signature(out) == g["signature"]
    if side.name == "library":
        from paged_kv_cache_42_gb300 import host as h
        assert h.step_signature(out) == g["signature"]


# --------------------------------------------------------------- SHA-256 --

def test_sha256_fips_example(host):
    g = GOLD["sha256_abc"]
    assert host.sha256(g["message"].encode()).hex() == g["digest"]


def test_sha256_matches_hashlib_across_padding_boundaries(host):
    rng = np.random.default_rng(7)
    for n in list(range(0, 140)) + [1000, 4096, 65537]:
        m = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
        assert host.sha256(m) == hashlib.sha256(m).digest(), n


def test_block_hash_chain(host):
    rng = np.random.default_rng(3)
    parent = None
    for _ in range(5):
        t = rng.integers(-2**31, 2**31 - 1, 16, dtype=np.int64).astype(np.int32)
        extra = rng.integers(0, 256, rng.integers(0, 40), dtype=np.uint8).tobytes()
        got = host.block_hash(parent, t, extra)
        assert got == host_ref.block_hash(parent, t.tolist(), extra)
        parent = got
    # the parent and the extra keys both change the hash
    t = list(range(16))
    assert host.block_hash(None, t) != host.block_hash(b"\x01" * 32, t)
    assert host.block_hash(None, t, b"lora:a") != host.block_hash(None, t, b"salt:a")


# ------------------------------------------------------------------ XXH64 --

XXH64_GOLD = json.load(open(os.path.join(HERE, "golden", "xxh64_vectors.json")))["vectors"]


@pytest.mark.parametrize("v", XXH64_GOLD, ids=lambda v: repr(v["input"][:12]))
def test_xxh64_published_values(host, v):
    want = int(v["digest"], 16)
    assert host_ref.xxh64(v["input"].encode(), v["seed"]) == want
    assert host.xxh64(v["input"].encode(), v["seed"]) == want


def test_xxh64_library_and_oracle_agree_at_every_length(host):
    # the published values reach the 32-byte stripes, the 4-byte word and
    # the byte tail; lengths 0..300 also reach every count of 8-byte words
    rng = np.random.default_rng(17)
    for n in range(301):
        data = rng.integers(0, 256, n, dtype=np.uint8).tobytes()
        seed = int(rng.integers(0, 2**63)) if n % 3 else 0
        assert host.xxh64(data, seed) == host_ref.xxh64(data, seed), n


def test_xxh64_planted_mistakes_break_a_published_value(monkeypatch):
    # a wrong constant or a dropped final step in the oracle's XXH64 fails
    # one of the published values
    def fails():
        return any(host_ref.xxh64(v["input"].encode(), v["seed"]) != int(v["digest"], 16)
                   for v in XXH64_GOLD)
    for k in range(5):
        bad = list(host_ref._XP)
        bad[k] ^= 1 << 40
        monkeypatch.setattr(host_ref, "_XP", tuple(bad))
        assert fails(), k
        monkeypatch.undo()
    monkeypatch.setattr(host_ref, "_rotl64", lambda x, r: ((x << (r + 1)) | (x >> (63 - r))) & host_ref._M64)
    assert fails()


def test_block_hash_chain_xxh64(host):
    rng = np.random.default_rng(5)
    parent = None
    for _ in range(6):
        t = rng.integers(-2**31, 2**31 - 1, 16, dtype=np.int64).astype(np.int32)
        extra = rng.integers(0, 256, rng.integers(0, 300), dtype=np.uint8).tobytes()
        got = host.block_hash(parent, t, extra, algo="xxh64")
        assert got == host_ref.block_hash(parent, t.tolist(), extra, algo="xxh64")
        assert got[8:] == bytes(24)
        parent = got
    # chaining: the parent changes the digest
    t = list(range(16))
    assert host.block_hash(None, t, algo="xxh64") != host.block_hash(b"\x01" * 32, t, algo="xxh64")


def test_pool_hash_algo_switches_only_while_empty(host):
    p = host.BlockPool(num_blocks=4, block_size=16)
    assert p.hash_algo == "sha256"
    p.set_hash_algo("xxh64")
    assert p.hash_algo == "xxh64"
    b = p.allocate(1)[0]
    p.cache_block(b, b"\x07" * 32)
    with pytest.raises(RuntimeError):
        p.set_hash_algo("sha256")  # a digest is in the table
    with pytest.raises(ValueError):
        host.BlockPool(num_blocks=4, block_size=16, hash_algo="md5")
    # a scheduler over an xxh64 pool finds its own prefix again
    pool = host.BlockPool(num_blocks=16, block_size=4, hash_algo="xxh64")
    s = host.Scheduler(pool, token_budget=64, max_model_len=64)
    prompt = list(range(20))
    s.add_request(0, prompt)
    s.step()
    s.finish(0)
    want = [host.block_hash(None, prompt[:4], algo="xxh64")]
    for k in range(1, 4):
        want.append(host.block_hash(want[-1], prompt[4 * k:4 * k + 4], algo="xxh64"))
    assert [pool.lookup(h) >= 0 for h in want] == [True] * 4
    s.add_request(1, prompt)
    out = s.step()
    assert out["num_computed"][0] == 16  # four cached blocks, the fifth recomputed


# ------------------------------------------------------------ host errors --

def test_pool_rejects_bad_calls(host):
    with pytest.raises(ValueError):
        host.BlockPool(ids=[1, 1], block_size=16)
    with pytest.raises(ValueError):
        host.BlockPool(ids=[-1], block_size=16)
    p = host.BlockPool(num_blocks=4, block_size=16)
    ids = p.allocate(2)
    with pytest.raises(RuntimeError):
        p.release([ids[0], ids[0]])  # one reference only
    with pytest.raises(RuntimeError):
        p.release([99])
    assert p.ref_count(ids[0]) == 1 and p.num_free() == 2
    with pytest.raises(RuntimeError):
        p.cache_block(p.free_queue()[0], b"\0" * 32)  # a free block cannot be registered
    p.cache_block(ids[0], b"\1" * 32)
    with pytest.raises(RuntimeError):
        p.cache_block(ids[0], b"\2" * 32)
    p.cache_block(ids[1], b"\1" * 32)  # same hash: the first block keeps it
    assert p.lookup(b"\1" * 32) == ids[0] and not p.is_cached(ids[1])


def test_rejected_release_changes_nothing(host):
    # a release naming a block more often than it is referenced, or an
    # unknown id, is refused whole; the next valid release then succeeds
    p = host.BlockPool(num_blocks=6, block_size=16)
    a = p.allocate(3)
    p.touch([a[0]])  # two references
    queue = p.free_queue()
    for bad in ([a[0], a[0], a[0]], [a[1], 99], [a[2], a[2]], [77], [a[0], a[1], a[1]]):
        with pytest.raises(RuntimeError):
            p.release(bad)
        assert [p.ref_count(b) for b in a] == [2, 1, 1] and p.free_queue() == queue
    p.release([a[0], a[0], a[1]])
    assert [p.ref_count(b) for b in a] == [0, 0, 1] and p.num_free() == 5


def test_scheduler_rejects_bad_calls(host):
    p = host.BlockPool(num_blocks=8, block_size=16)
    with pytest.raises(ValueError):
        host.Scheduler(p, token_budget=0, max_model_len=64)
    with pytest.raises(ValueError):
        host.Scheduler(p, token_budget=8, max_model_len=64, max_blocks_per_req=3)
    s = host.Scheduler(p, token_budget=8, max_model_len=32)
    with pytest.raises(RuntimeError):
        s.add_request(0, list(range(33)))  # longer than max_model_len
    s.add_request(0, [1, 2, 3])
    with pytest.raises(RuntimeError):
        s.add_request(0, [1])  # id in use
    with pytest.raises(RuntimeError):
        s.append_token(0, 5)   # still waiting: no logits yet
    s.step()
    s.append_token(0, 5)
    with pytest.raises(RuntimeError):
        s.append_token(0, 6)   # token 5 not computed yet
    s.finish(0)
    assert p.num_free() == 8
    with pytest.raises(RuntimeError):
        s.finish(0)


def test_prefix_map_under_colliding_digests(host):
    """The prefix-cache map against a dict, with digests crowded into a few
    home slots (the map's home slot is taken from a digest's first bytes;
    0 and the last slot test the wrap-around), through registrations, hits
    that pull a free block back, and evictions by allocation (the free
    queue's head loses its digest), so long probe runs form and are cut by
    deletions."""
    n = 64  # a table of 128 slots
    pool = host.BlockPool(num_blocks=n, block_size=16)
    rng = np.random.default_rng(11)

    def digest():
        home = int(rng.choice([0, 1, 2, 127, 64]))
        first = (int(rng.integers(0, 2**24)) << 7) | home  # same low 7 bits
        rest = rng.integers(0, 256, 28, dtype=np.uint8).tobytes()
        return first.to_bytes(4, "little") + rest

    by_hash, of_block, live = {}, {}, []
    for _ in range(3000):
        op = rng.integers(0, 4)
        if op == 0 and pool.num_free() > 0:  # allocate: the head blocks lose their digests
            k = int(rng.integers(1, min(4, pool.num_free()) + 1))
            head = pool.free_queue()[:k]
            got = pool.allocate(k)
            assert got == head
            for b in got:
                h = of_block.pop(b, None)
                if h is not None:
                    del by_hash[h]
            live += got
        elif op == 1 and live:  # register a referenced, unregistered block
            b = live[int(rng.integers(0, len(live)))]
            if b in of_block:
                continue
            h = digest() if rng.random() < 0.8 or not by_hash else list(by_hash)[0]
            pool.cache_block(b, h)
            if h not in by_hash:
                by_hash[h] = b
                of_block[b] = h
        elif op == 2 and live:  # release one reference
            b = live.pop(int(rng.integers(0, len(live))))
            pool.release([b])
        elif op == 3 and by_hash:  # a hit takes a reference (and the block off the queue)
            h = list(by_hash)[int(rng.integers(0, len(by_hash)))]
            b = pool.lookup(h)
            assert b == by_hash[h]
            pool.touch([b])
            live.append(b)
        for h, b in by_hash.items():
            assert pool.lookup(h) == b
        for b in range(n):
            assert pool.is_cached(b) == (b in of_block)
    assert len(by_hash) > 8  # the run kept a crowded map
    for h in [digest() for _ in range(50)]:
        assert pool.lookup(h) == by_hash.get(h, -1)


@pytest.mark.parametrize("seed", [0, 1, 2, 3])
def test_retained_block_tables_match_full_rows(host, seed):
    """pa_sched_output.block_tables_retained: a step that writes only what
    changed since its last step leaves the same table as one that writes
    every row, through admissions, prefix hits, chunked prefills, growth by
    a block, preemption (a small pool), finishes and reused request ids."""
    rng = np.random.default_rng(600 + seed)
    bs = 16
    shared = rng.integers(0, 1000, 64).tolist()
    sides = []
    for retained in (True, False):
        pool = host.BlockPool(num_blocks=24, block_size=bs)
        s = host.Scheduler(pool, token_budget=48, max_model_len=256, long_prefill_threshold=24,
                           max_reqs=64, retained_block_tables=retained)
        sides.append((pool, s))
    ops = np.random.default_rng(700 + seed)
    live, next_id, preempted = set(), 0, 0
    for it in range(300):
        if ops.random() < 0.25 and len(live) < 12:
            n = int(ops.integers(1, 80))
            prompt = (shared[:int(ops.integers(0, 64))] + ops.integers(0, 1000, n).tolist())[:200]
            rid = int(ops.integers(0, 6)) if ops.random() < 0.3 else 100 + next_id
            if rid in live:
                rid = 100 + next_id
            next_id += 1
            for _, s in sides:
                s.add_request(rid, prompt)
            live.add(rid)
        outs = [s.step() for _, s in sides]
        a, b = outs
        for k in a:
            if k != "block_tables":
                assert np.array_equal(np.asarray(a[k]), np.asarray(b[k])), (it, k)
        # retained rows are max_blocks_per_req (16) wide: the full-mode rows,
        # then -1
        ta, tb = a["block_tables"], b["block_tables"]
        assert ta.shape == (tb.shape[0], 16), (it, ta.shape)
        assert np.array_equal(ta[:, :tb.shape[1]], tb), it
        assert np.all(ta[:, tb.shape[1]:] == -1), it
        preempted += len(a["preempted_ids"])
        for rid in a["req_ids"].tolist():
            st = sides[0][1].request_state(rid)
            if st["num_computed"] == st["num_tokens"]:
                if ops.random() < 0.02 or st["num_tokens"] >= 250:
                    for _, s in sides:
                        s.finish(rid)
                    live.discard(rid)
                else:
                    tok = int(ops.integers(0, 1000))
                    for _, s in sides:
                        s.append_token(rid, tok)
    assert next_id > 10 and preempted > 0


def test_retained_mode_toggled_and_buffer_swapped(host):
    """Switching block_tables_retained on and off between steps, and moving
    to a new table buffer, leaves every table equal to a full write: a step
    only reuses rows written into the same buffer at the same stride."""
    rng = np.random.default_rng(650)
    sides = []
    for _ in range(2):
        pool = host.BlockPool(num_blocks=32, block_size=16)
        sides.append(host.Scheduler(pool, token_budget=40, max_model_len=256,
                                    long_prefill_threshold=20, max_reqs=8))
    a, b = sides  # a toggles and moves; b writes every row at the widest stride
    live, nid, swaps, reuse_steps = set(), 0, 0, 0
    for it in range(400):
        if rng.random() < 0.2 and len(live) < 10:
            prompt = rng.integers(0, 500, int(rng.integers(1, 60))).tolist()
            for s in sides:
                s.add_request(nid, prompt)
            live.add(nid)
            nid += 1
        a.retained = bool(rng.random() < 0.7)
        a._out.block_tables_retained = int(a.retained)
        if rng.random() < 0.05:
            a._alloc(a._max_reqs + 1)  # new buffers at new addresses
            a._out.block_tables_retained = int(a.retained)
            swaps += 1
        oa, ob = a.step(), b.step()
        reuse_steps += a.retained
        ta, tb = oa["block_tables"], ob["block_tables"]
        w = tb.shape[1]
        assert ta.shape[0] == tb.shape[0] and ta.shape[1] >= w, it
        assert np.array_equal(ta[:, :w], tb) and np.all(ta[:, w:] == -1), it
        for rid in oa["req_ids"].tolist():
            st = a.request_state(rid)
            if st["num_computed"] == st["num_tokens"]:
                if rng.random() < 0.05 or st["num_tokens"] >= 250:
                    for s in sides:
                        s.finish(rid)
                    live.discard(rid)
                else:
                    tok = int(rng.integers(0, 500))
                    for s in sides:
                        s.append_token(rid, tok)
    assert swaps > 5 and reuse_steps > 100


# ---------------------------------------- invariants and random parity ----

class KVModel:
    """What the GPU cache would hold: the token id written at each slot."""

    def __init__(self):
        self.slot = {}

    def write(self, out):
        for s, t in zip(out["slot_mapping"], out["input_tokens"]):
            self.slot[int(s)] = int(t)


def check_invariants(sched, pool, out, budget, bs, kv: KVModel):
    assert int(np.sum(out["num_scheduled"])) <= budget
    assert out["num_tokens"] == int(np.sum(out["num_scheduled"]))
    qsl = np.asarray(out["query_start_loc"])
    assert qsl[0] == 0 and np.all(np.diff(qsl) == np.asarray(out["num_scheduled"]))
    # reference counts equal the number of running requests holding a block
    counts = collections.Counter(b for r in sched.running for b in r.blocks)
    for b, n in pool.refs.items():
        assert n == counts.get(b, 0)
    assert sorted(pool.free) == sorted(b for b, n in pool.refs.items() if n == 0)
    assert set(pool.block_of.values()) == set(pool.hash_of) and \
        all(pool.block_of[h] == b for b, h in pool.hash_of.items())
    # every computed position of a running request holds its own token
    for r in sched.running:
        assert len(r.blocks) == -(-r.num_computed // bs)
        for p in range(r.num_computed):
            assert kv.slot.get(r.blocks[p // bs] * bs + p % bs) == r.tokens[p], (r.id, p)


def random_run(seed: int, lib_host=None, steps: int = 120, algo: str = "sha256"):
    rng = np.random.default_rng(seed)
    bs = int(rng.choice([2, 4, 16]))
    n_blocks = int(rng.integers(6, 40))
    budget = int(rng.integers(4, 40))
    max_len = int(rng.integers(2, 6)) * bs * 2
    cfg = dict(token_budget=budget, max_model_len=max_len,
               max_running=int(rng.choice([0, 2, 5])),
               long_prefill_threshold=int(rng.choice([0, 0, 3, 7])),
               prefix_caching=bool(rng.integers(0, 4)), chunked_prefill=bool(rng.integers(0, 4)))
    ids = rng.permutation(1000)[:n_blocks].tolist()
    o_pool = host_ref.Pool(ids, bs, hash_algo=algo)
    o = host_ref.Scheduler(o_pool, **cfg)
    if lib_host is not None:
        l_pool = lib_host.BlockPool(ids=ids, block_size=bs, hash_algo=algo)
        lib = lib_host.Scheduler(l_pool, **cfg)
    kv = KVModel()
    prefixes = [rng.integers(0, 5, int(rng.integers(1, 3 * bs))).tolist() for _ in range(3)]
    next_id, live = 0, []
    n_preempt = n_hits = 0
    for step in range(steps):
        if rng.random() < 0.5 or not live:
            pre = prefixes[int(rng.integers(0, 3))]
            plen = int(rng.integers(1, max_len // 2 + 1))
            prompt = (pre + rng.integers(0, 5, plen).tolist())[:plen]
            extra = b"" if rng.random() < 0.8 else b"salt"
            o.add_request(next_id, prompt, extra)
            if lib_host is not None:
                lib.add_request(next_id, prompt, extra)
            live.append(next_id)
            next_id += 1
        was_waiting = {r.id for r in o.waiting}
        out = o.step()
        kv.write(out)
        n_preempt += len(out["preempted_ids"])
        n_hits += sum(1 for c, rid in zip(out["num_computed"], out["req_ids"])
                      if rid in was_waiting and c > 0)
        check_invariants(o, o_pool, out, budget, bs, kv)
        if lib_host is not None:
            got = lib.step()
            for k in ("req_ids", "num_scheduled", "num_computed", "query_start_loc", "seq_lens",
                      "block_tables", "slot_mapping", "positions", "input_tokens",
                      "preempted_ids"):
                assert np.array_equal(np.asarray(got[k]).reshape(-1),
                                      np.asarray(out[k], dtype=np.int64).reshape(-1)), (seed, step, k)
            for k in ("num_tokens", "max_query_len", "max_seq_len", "num_decode_reqs",
                      "num_context_reqs", "num_context_tokens", "num_generation_reqs",
                      "num_generation_tokens"):
                assert got[k] == out[k], (seed, step, k)
            assert l_pool.free_queue() == list(o_pool.free), (seed, step)
            # the same digests, under the same blocks
            for h, b in o_pool.block_of.items():
                assert l_pool.lookup(h) == b, (seed, step)
            assert sum(l_pool.is_cached(b) for b in ids) == len(o_pool.block_of), (seed, step)
        for rid in list(out["req_ids"]):
            r = o.reqs[rid]
            if r.num_computed == len(r.tokens):
                if len(r.tokens) >= max_len or rng.random() < 0.1:
                    o.finish(rid)
                    if lib_host is not None:
                        lib.finish(rid)
                    live.remove(rid)
                else:
                    tok = int(rng.integers(0, 5))
                    o.append_token(rid, tok)
                    if lib_host is not None:
                        lib.append_token(rid, tok)
    return n_preempt, n_hits


@pytest.mark.parametrize("algo", ["sha256", "xxh64"])
def test_oracle_invariants_random(algo):
    total_pre = total_hits = 0
    for seed in range(30):
        p, h = random_run(seed, algo=algo)
        total_pre += p
        total_hits += h
    assert total_pre > 0 and total_hits > 0  # the sweep reaches preemption and prefix hits


@pytest.mark.parametrize("algo", ["sha256", "xxh64"])
def test_library_matches_oracle_random(host, algo):
    for seed in range(100, 160):
        random_run(seed, lib_host=host, algo=algo)


# ----------------------------------------------- planted oracle mistakes --

class _ForwardRelease(host_ref.Pool):
    def release(self, ids):
        for slot in ids:  # mistake: first block first
            self.refs[slot] -= 1
            if self.refs[slot] == 0:
                (self.free.append if slot in self.hash_of else self.free.appendleft)(slot)


class _AllToTail(host_ref.Pool):
    def release(self, ids):
        for slot in reversed(list(ids)):
            self.refs[slot] -= 1
            if self.refs[slot] == 0:
                self.free.append(slot)  # mistake: uncached blocks to the tail too


class _KeepsHash(host_ref.Pool):
    def allocate(self, n):
        if n > len(self.free):
            raise MemoryError("No free KV block")
        out = [self.free.popleft() for _ in range(n)]  # mistake: hash survives reuse
        for b in out:
            self.refs[b] = 1
        return out


class _WaitingFirst(host_ref.Scheduler):
    def step(self):
        self.running, waiting_first = [], self.running  # mistake: admit before running
        out = super().step()
        self.running = waiting_first + self.running
        return out


class _Mut:
    def __init__(self, **over):
        self.__dict__.update(over)

    def __getattr__(self, k):
        return getattr(host_ref, k)


@pytest.mark.parametrize("mutant,runner", [
    (_Mut(Pool=_ForwardRelease), run_free_queue_example),
    (_Mut(Pool=_AllToTail), run_head_tail_rule),
    (_Mut(Pool=_KeepsHash), run_free_queue_example),
    (_Mut(reusable_tokens=lambda s, p, b: s // b * b), run_reusable),
    (_Mut(Scheduler=_WaitingFirst), run_budget_trace),
])
def test_planted_oracle_mistakes_break_a_pin(mutant, runner):
    with pytest.raises(AssertionError):
        runner(OracleSide(mutant))


def test_pool_closed_before_its_scheduler(host):
    # Finalizers of objects collected together run in any order: closing the
    # pool first must destroy the scheduler still drawing from it (which
    # releases its blocks into the pool) rather than leave it to release them
    # into freed memory later.
    pool = host.BlockPool(num_blocks=8, block_size=16)
    s = host.Scheduler(pool, token_budget=16, max_model_len=64)
    s.add_request(0, list(range(40)))
    s.step()
    assert pool.num_free() < 8
    pool.close()
    with pytest.raises(RuntimeError):
        s.step()
    s.close()  # a no-op now
    s2 = host.Scheduler(host.BlockPool(num_blocks=8, block_size=16), token_budget=16,
                        max_model_len=64)
    s2.close()
    s2.pool.close()
