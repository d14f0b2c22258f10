"""Plain Python model of the host runtime: block pool, chained block hash,
prefix lookup and the token-budget scheduler step.

TEST INFRASTRUCTURE ONLY: the tests (and nothing in the product) use this
module to check the library's C++ host runtime. It shares no code with it:
it is written from the pages' description with Python containers (a deque
for the free queue, dicts for reference counts and the hash map, lists for
the request queues), ``hashlib`` for SHA-256 and a plain restatement of
XXH64 for the fast-hash option, with no attention to speed.

Sources (page title, section):
  * "Deep Dive - vLLM", "Block pool, prefix cache, and eviction": reference
    counts; a released block goes to the free queue's tail if it holds a hash
    and to its head if not; a request's blocks are released last first;
    allocation pops the head and removes the block's hash before reuse; only
    whole blocks are reused and at most prompt_length - 1 tokens; the block
    hash chains the parent hash, the block's tokens and extra keys (SHA-256).
  * "Inside the vLLM Engine", "The pool, the queue, and the hash": a free
    block keeps its hash until reused and a lookup can take it back out of
    the free queue.
  * "Deep Dive - vLLM", "The V1 scheduler: one token budget", and "vLLM v1
    Deep Dive: How LLM(...) and the Server Boot and Generate", Part 3
    "Step 3 - Scheduler iteration": running requests first, then waiting
    ones, each granted min(deficit, long-prefill threshold, budget left,
    room under max_model_len); on an allocation failure the last running
    request is preempted until the blocks fit or the request itself went;
    waiting requests start from their longest cached prefix, stop admission
    when they do not fit (without chunked prefill) or cannot get blocks, and
    respect max_num_seqs; computed counts advance when the step is planned.

Readings where the pages leave a step open (the same ones the library takes):
  * a step that preempted admits no waiting request;
  * preemption recomputes: blocks released, computed count reset to 0, the
    request goes back to the front of the waiting queue;
  * a newly full block whose hash another block already holds stays
    unregistered (block tables are append-only);
  * hash input = parent (32 zero bytes for the first block) + token ids as
    int32 little endian + the request's extra key bytes.
"""
from __future__ import annotations

import hashlib
import struct
from collections import deque

ZERO_HASH = bytes(32)

_M64 = (1 << 64) - 1
# XXH64's five constants, as its published description gives them
_XP = (0x9E3779B185EBCA87, 0xC2B2AE3D27D4EB4F, 0x165667B19E3779F9, 0x85EBCA77C2B2AE63,
       0x27D4EB2F165667C5)


def _rotl64(x: int, r: int) -> int:
    return ((x << r) | (x >> (64 - r))) & _M64


def _xround(acc: int, lane: int) -> int:
    return _rotl64((acc + lane * _XP[1]) & _M64, 31) * _XP[0] & _M64


def xxh64(data: bytes, seed: int = 0) -> int:
    """XXH64 of ``data`` (the xxHash family's 64-bit function, by its
    published description): four accumulators over 32-byte stripes, folded
    and merged; then the length, 8-byte words, a 4-byte word and single
    bytes mixed in; then the final avalanche. Words are little endian."""
    data = bytes(data)
    n, pos = len(data), 0
    word = lambda at, size: int.from_bytes(data[at:at + size], "little")
    if n >= 32:
        acc = [(seed + _XP[0] + _XP[1]) & _M64, (seed + _XP[1]) & _M64, seed & _M64,
               (seed - _XP[0]) & _M64]
        while n - pos >= 32:
            acc = [_xround(acc[k], word(pos + 8 * k, 8)) for k in range(4)]
            pos += 32
        h = sum(_rotl64(a, r) for a, r in zip(acc, (1, 7, 12, 18))) & _M64
        for a in acc:
            h = ((h ^ _xround(0, a)) * _XP[0] + _XP[3]) & _M64
    else:
        h = (seed + _XP[4]) & _M64
    h = (h + n) & _M64
    while n - pos >= 8:
        h = (_rotl64(h ^ _xround(0, word(pos, 8)), 27) * _XP[0] + _XP[3]) & _M64
        pos += 8
    if n - pos >= 4:
        h = (_rotl64(h ^ (word(pos, 4) * _XP[0] & _M64), 23) * _XP[1] + _XP[2]) & _M64
        pos += 4
    for b in data[pos:]:
        h = _rotl64(h ^ (b * _XP[4] & _M64), 11) * _XP[0] & _M64
    for shift, mul in ((33, _XP[1]), (29, _XP[2]), (32, None)):
        h ^= h >> shift
        if mul is not None:
            h = h * mul & _M64
    return h


def block_hash(parent: bytes | None, tokens, extra: bytes = b"", algo: str = "sha256") -> bytes:
    """Chained hash of one block ("Deep Dive - vLLM", "Block pool, prefix
    cache, and eviction": hash of the parent hash, the block tokens and the
    extra keys; SHA-256 by default, a faster xxhash variant selectable).
    ``algo`` "xxh64": the 64-bit XXH64 of the same bytes, little endian, in
    the first 8 of 32 bytes."""
    data = (parent if parent is not None else ZERO_HASH) + struct.pack(
        "<%di" % len(tokens), *[int(t) for t in tokens]) + bytes(extra)
    if algo == "xxh64":
        return xxh64(data).to_bytes(8, "little") + bytes(24)
    if algo != "sha256":
        raise ValueError(f"unknown hash algorithm {algo!r}")
    return hashlib.sha256(data).digest()


def prompt_block_hashes(tokens, block_size: int, extra: bytes = b"",
                        algo: str = "sha256") -> list:
    """Hashes of every full block of ``tokens``, each chained to the one
    before it."""
    out, parent = [], None
    for b in range(len(tokens) // block_size):
        parent = block_hash(parent, tokens[b * block_size:(b + 1) * block_size], extra, algo)
        out.append(parent)
    return out


def reusable_tokens(shared: int, prompt_length: int, block_size: int) -> int:
    """Prompt tokens a prefix hit can skip ("Deep Dive - vLLM", "Block pool,
    prefix cache, and eviction"): the shared prefix, cut to leave one
    position for the logits, rounded down to whole blocks."""
    for x in (shared, prompt_length, block_size):
        if type(x) is not int:
            raise ValueError("counts must be plain integers")
    if block_size <= 0 or prompt_length <= 0 or not 0 <= shared <= prompt_length:
        raise ValueError("need a nonempty prompt and 0 <= shared <= prompt_length")
    return min(shared, prompt_length - 1) // block_size * block_size


class Pool:
    """Block pool: reference counts, an LRU free queue and the prefix-cache
    map ("Deep Dive - vLLM", "Block pool, prefix cache, and eviction")."""

    def __init__(self, ids, block_size: int, hash_algo: str = "sha256"):
        ids = [int(i) for i in ids]
        if len(set(ids)) != len(ids) or any(i < 0 for i in ids) or block_size <= 0:
            raise ValueError("ids must be distinct and >= 0; block_size > 0")
        if hash_algo not in ("sha256", "xxh64"):
            raise ValueError(f"unknown hash algorithm {hash_algo!r}")
        self.block_size = block_size
        self.hash_algo = hash_algo
        self.refs = {i: 0 for i in ids}
        self.hash_of = {}       # block id -> hash
        self.block_of = {}      # hash -> block id
        self.free = deque(ids)  # head = left

    def num_free(self) -> int:
        return len(self.free)

    def allocate(self, n: int) -> list:
        """Pop n blocks from the head; each loses its hash before reuse."""
        if n > len(self.free):
            raise MemoryError("No free KV block")
        out = []
        for _ in range(n):
            slot = self.free.popleft()
            assert self.refs[slot] == 0
            h = self.hash_of.pop(slot, None)
            if h is not None:
                del self.block_of[h]
            self.refs[slot] = 1
            out.append(slot)
        return out

    def release(self, ids) -> None:
        """Drop one reference per id, last id first; a block whose count hits
        zero goes to the tail if it holds a hash, else to the head."""
        need = {}
        for slot in ids:
            need[slot] = need.get(slot, 0) + 1
            if slot not in self.refs or need[slot] > self.refs[slot]:
                raise ValueError(f"release of block {slot} without a reference")
        for slot in reversed(list(ids)):
            self.refs[slot] -= 1
            if self.refs[slot] == 0:
                if slot in self.hash_of:
                    self.free.append(slot)
                else:
                    self.free.appendleft(slot)

    def touch(self, ids) -> None:
        """A prefix hit: one more reference; a free block leaves the queue."""
        for slot in ids:
            if slot not in self.refs:
                raise ValueError(f"unknown block {slot}")
        for slot in ids:
            if self.refs[slot] == 0:
                self.free.remove(slot)
            self.refs[slot] += 1

    def cache_block(self, slot: int, h: bytes) -> None:
        if slot not in self.refs or self.refs[slot] == 0 or slot in self.hash_of:
            raise ValueError("only a live block without a hash can be registered")
        if h in self.block_of:
            return  # the block that registered first keeps the hash
        self.block_of[h] = slot
        self.hash_of[slot] = h

    def lookup(self, h: bytes):
        return self.block_of.get(h, -1)

    def find_cached_prefix(self, tokens, extra: bytes = b"") -> list:
        """Leading full prompt blocks present in the cache, stopping at the
        first miss, within num_tokens - 1 tokens."""
        limit = (len(tokens) - 1) // self.block_size
        hits = []
        for h in prompt_block_hashes(tokens[:limit * self.block_size], self.block_size, extra,
                                     self.hash_algo):
            slot = self.block_of.get(h)
            if slot is None:
                break
            hits.append(slot)
        return hits


class Request:
    def __init__(self, req_id: int, prompt, extra: bytes = b""):
        self.id = req_id
        self.tokens = [int(t) for t in prompt]
        self.prompt_len = len(self.tokens)
        self.extra = bytes(extra)
        self.num_computed = 0
        self.blocks = []
        self.running = False


class Scheduler:
    """One token budget over running, then waiting, requests ("Deep Dive -
    vLLM", "The V1 scheduler: one token budget"; "vLLM v1 Deep Dive", Part 3
    "Step 3 - Scheduler iteration")."""

    def __init__(self, pool: Pool, *, token_budget: int, max_model_len: int,
                 max_running: int = 0, long_prefill_threshold: int = 0,
                 max_blocks_per_req: int | None = None, prefix_caching: bool = True,
                 chunked_prefill: bool = True):
        self.pool = pool
        self.budget = token_budget
        self.max_model_len = max_model_len
        self.max_running = max_running
        self.threshold = long_prefill_threshold
        self.stride = max_blocks_per_req or -(-max_model_len // pool.block_size)
        self.prefix_caching = prefix_caching
        self.chunked = chunked_prefill
        self.reqs = {}
        self.running = []
        self.waiting = deque()

    def add_request(self, req_id: int, prompt, extra: bytes = b"") -> None:
        if req_id in self.reqs or not 0 < len(prompt) <= self.max_model_len:
            raise ValueError("bad request")
        r = Request(req_id, prompt, extra)
        self.reqs[req_id] = r
        self.waiting.append(r)

    def append_token(self, req_id: int, token: int) -> None:
        r = self.reqs[req_id]
        if not r.running or r.num_computed != len(r.tokens) or len(r.tokens) >= self.max_model_len:
            raise ValueError("request cannot take a sampled token now")
        r.tokens.append(int(token))

    def finish(self, req_id: int) -> None:
        r = self.reqs.pop(req_id)
        if r.running:
            self.running.remove(r)
            self.pool.release(r.blocks)
            r.blocks = []
        else:
            self.waiting.remove(r)

    def _blocks_for(self, n: int) -> int:
        return -(-n // self.pool.block_size)

    def _preempt(self, r: Request) -> None:
        self.pool.release(r.blocks)
        r.blocks = []
        r.num_computed = 0
        r.running = False
        self.waiting.appendleft(r)

    def step(self) -> dict:
        pool, bs = self.pool, self.pool.block_size
        budget = self.budget
        scheduled = []   # (request, granted tokens)
        preempted = []

        # running requests first, in order
        i = 0
        while i < len(self.running) and budget > 0:
            r = self.running[i]
            n = len(r.tokens) - r.num_computed
            if 0 < self.threshold < n:
                n = self.threshold
            n = min(n, budget, self.max_model_len - r.num_computed)
            if n <= 0:
                i += 1
                continue
            need = self._blocks_for(r.num_computed + n) - len(r.blocks)
            gone = False
            while need > pool.num_free():
                victim = self.running.pop()
                self._preempt(victim)
                preempted.append(victim.id)
                if victim is r:
                    gone = True
                    break
            if gone:
                break
            r.blocks += pool.allocate(need)
            scheduled.append((r, n))
            budget -= n
            i += 1

        # then waiting requests, unless this step had to preempt
        while not preempted and self.waiting and budget > 0:
            if self.max_running > 0 and len(self.running) >= self.max_running:
                break
            r = self.waiting[0]
            hits = pool.find_cached_prefix(r.tokens, r.extra) if self.prefix_caching else []
            cached = len(hits) * bs
            n = len(r.tokens) - cached
            if 0 < self.threshold < n:
                n = self.threshold
            if not self.chunked and n > budget:
                break
            n = min(n, budget)
            need = self._blocks_for(cached + n) - len(hits)
            evictable = sum(1 for b in hits if pool.refs[b] == 0)
            if need + evictable > pool.num_free():
                break
            pool.touch(hits)
            r.blocks = list(hits) + pool.allocate(need)
            r.num_computed = cached
            r.running = True
            self.waiting.popleft()
            self.running.append(r)
            scheduled.append((r, n))
            budget -= n

        # the batch the kernels take
        out = dict(req_ids=[], num_scheduled=[], num_computed=[], query_start_loc=[0],
                   seq_lens=[], block_tables=[], slot_mapping=[], positions=[],
                   input_tokens=[], preempted_ids=preempted, num_decode_reqs=0,
                   num_context_reqs=0, num_context_tokens=0, num_generation_reqs=0,
                   num_generation_tokens=0)
        width = max([len(r.blocks) for r, _ in scheduled] + [1])  # widest scheduled request
        for r, n in scheduled:
            ctx = r.num_computed
            out["req_ids"].append(r.id)
            out["num_scheduled"].append(n)
            out["num_computed"].append(ctx)
            out["query_start_loc"].append(out["query_start_loc"][-1] + n)
            out["seq_lens"].append(ctx + n)
            out["block_tables"].append(r.blocks + [-1] * (width - len(r.blocks)))
            for p in range(ctx, ctx + n):
                out["positions"].append(p)
                out["input_tokens"].append(r.tokens[p])
                out["slot_mapping"].append(r.blocks[p // bs] * bs + p % bs)
            if n == 1 and ctx >= r.prompt_len:
                out["num_decode_reqs"] += 1
            # the step's profile signature ("vLLM v1 Deep Dive", Part 3, Step 4c):
            # a span that starts inside the prompt is context, otherwise generation
            phase = "context" if ctx < r.prompt_len else "generation"
            out[f"num_{phase}_reqs"] += 1
            out[f"num_{phase}_tokens"] += n
        out["num_tokens"] = out["query_start_loc"][-1]
        out["max_query_len"] = max(out["num_scheduled"], default=0)
        out["max_seq_len"] = max(out["seq_lens"], default=0)

        # planned state: computed counts advance; newly full blocks are cached
        for r, n in scheduled:
            old = r.num_computed
            r.num_computed += n
            if self.prefix_caching:
                hashes = prompt_block_hashes(r.tokens[:r.num_computed // bs * bs], bs, r.extra,
                                             pool.hash_algo)
                for b in range(old // bs, r.num_computed // bs):
                    if r.blocks[b] not in pool.hash_of:
                        pool.cache_block(r.blocks[b], hashes[b])
        return out
