"""Python binding of the library's host runtime (``include/pa_host.h``):
block pool, chained block hash and token-budget scheduler.

Argument marshalling only; every operation runs in the library's C++ code.
Arrays come back as numpy arrays so they can be copied to the GPU in one
step (``torch.from_numpy(...).cuda()``) and handed to :func:`binding.attention`.
"""
from __future__ import annotations

import ctypes
import time

import numpy as np

from . import binding as _binding

_c_i = ctypes.c_int
_c_p = ctypes.c_void_p
_i32p = ctypes.POINTER(ctypes.c_int32)
_i64p = ctypes.POINTER(ctypes.c_int64)
_u8p = ctypes.c_char_p


class SchedConfig(ctypes.Structure):
    _fields_ = [("token_budget", _c_i), ("max_running", _c_i), ("long_prefill_threshold", _c_i),
                ("max_model_len", _c_i), ("max_blocks_per_req", _c_i),
                ("enable_prefix_caching", _c_i), ("enable_chunked_prefill", _c_i)]


class SchedOutput(ctypes.Structure):
    _fields_ = [("max_reqs", _c_i), ("max_tokens", _c_i), ("max_preempted", _c_i),
                ("req_ids", _i64p), ("num_scheduled", _i32p), ("num_computed", _i32p),
                ("query_start_loc", _i32p), ("seq_lens", _i32p), ("block_tables", _i32p),
                ("slot_mapping", _i64p), ("positions", _i32p), ("input_tokens", _i32p),
                ("preempted_ids", _i64p), ("num_reqs", _c_i), ("num_tokens", _c_i),
                ("num_preempted", _c_i), ("max_query_len", _c_i), ("max_seq_len", _c_i),
                ("block_table_stride", _c_i), ("num_decode_reqs", _c_i),
                ("num_context_reqs", _c_i), ("num_context_tokens", _c_i),
                ("num_generation_reqs", _c_i), ("num_generation_tokens", _c_i),
                ("block_tables_retained", _c_i)]


_READY = False


def lib() -> ctypes.CDLL:
    global _READY
    L = _binding.lib()
    if not _READY:
        L.pa_pool_create.argtypes = [_c_i, _c_i, _i32p]
        L.pa_pool_create.restype = _c_p
        L.pa_pool_destroy.argtypes = [_c_p]
        L.pa_pool_destroy.restype = None
        for f in ("pa_pool_num_blocks", "pa_pool_block_size", "pa_pool_num_free"):
            getattr(L, f).argtypes = [_c_p]
            getattr(L, f).restype = _c_i
        L.pa_pool_allocate.argtypes = [_c_p, _c_i, _i32p]
        L.pa_pool_free.argtypes = [_c_p, _i32p, _c_i]
        L.pa_pool_touch.argtypes = [_c_p, _i32p, _c_i]
        L.pa_pool_cache_block.argtypes = [_c_p, ctypes.c_int32, _u8p]
        L.pa_pool_lookup.argtypes = [_c_p, _u8p]
        L.pa_pool_lookup.restype = ctypes.c_int32
        L.pa_pool_ref_count.argtypes = [_c_p, ctypes.c_int32]
        L.pa_pool_is_cached.argtypes = [_c_p, ctypes.c_int32]
        L.pa_pool_free_queue.argtypes = [_c_p, _i32p, _c_i]
        L.pa_block_hash.argtypes = [_u8p, _i32p, _c_i, _u8p, _c_i, ctypes.c_char_p]
        L.pa_block_hash.restype = None
        L.pa_sha256.argtypes = [_u8p, ctypes.c_size_t, ctypes.c_char_p]
        L.pa_sha256.restype = None
        L.pa_block_hash_algo.argtypes = [_c_i, _u8p, _i32p, _c_i, _u8p, _c_i, ctypes.c_char_p]
        L.pa_xxh64.argtypes = [_u8p, ctypes.c_size_t, ctypes.c_uint64]
        L.pa_xxh64.restype = ctypes.c_uint64
        L.pa_pool_set_hash_algo.argtypes = [_c_p, _c_i]
        L.pa_pool_hash_algo.argtypes = [_c_p]
        L.pa_pool_find_cached_prefix.argtypes = [_c_p, _i32p, _c_i, _u8p, _c_i, _i32p, _c_i]
        L.pa_reusable_tokens.argtypes = [_c_i, _c_i, _c_i, ctypes.POINTER(_c_i)]
        L.pa_sched_create.argtypes = [_c_p, ctypes.POINTER(SchedConfig)]
        L.pa_sched_create.restype = _c_p
        L.pa_sched_destroy.argtypes = [_c_p]
        L.pa_sched_destroy.restype = None
        L.pa_sched_add_request.argtypes = [_c_p, ctypes.c_int64, _i32p, _c_i, _u8p, _c_i]
        L.pa_sched_append_token.argtypes = [_c_p, ctypes.c_int64, ctypes.c_int32]
        L.pa_sched_finish.argtypes = [_c_p, ctypes.c_int64]
        L.pa_sched_step.argtypes = [_c_p, ctypes.POINTER(SchedOutput)]
        L.pa_sched_num_running.argtypes = [_c_p]
        L.pa_sched_num_waiting.argtypes = [_c_p]
        ip = ctypes.POINTER(_c_i)
        L.pa_sched_request_state.argtypes = [_c_p, ctypes.c_int64, ip, ip, ip, ip, ip]
        L.pa_sched_request_blocks.argtypes = [_c_p, ctypes.c_int64, _i32p, _c_i]
        _READY = True
    return L


def _i32(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int32))


def _p32(a: np.ndarray):
    return a.ctypes.data_as(_i32p)


def _check(st: int, what: str) -> None:
    if st != 0:
        raise _binding.PagedAttentionError(st, what)


def sha256(data: bytes) -> bytes:
    out = ctypes.create_string_buffer(32)
    lib().pa_sha256(bytes(data), len(data), out)
    return out.raw


HASH_ALGOS = {"sha256": 0, "xxh64": 1}  # PA_HASH_SHA256, PA_HASH_XXH64


def xxh64(data: bytes, seed: int = 0) -> int:
    return int(lib().pa_xxh64(bytes(data), len(data), seed))


def block_hash(parent: bytes | None, tokens, extra: bytes = b"", algo: str = "sha256") -> bytes:
    t = _i32(tokens)
    out = ctypes.create_string_buffer(32)
    _check(lib().pa_block_hash_algo(HASH_ALGOS[algo], parent, _p32(t), int(t.size),
                                    bytes(extra) or None, len(extra), out), "pa_block_hash_algo")
    return out.raw


def reusable_tokens(shared: int, prompt_length: int, block_size: int) -> int:
    v = _c_i(0)
    _check(lib().pa_reusable_tokens(shared, prompt_length, block_size, ctypes.byref(v)),
           "pa_reusable_tokens")
    return int(v.value)


class BlockPool:
    """pa_pool_*: physical blocks with reference counts, the free queue and
    the prefix-cache map."""

    def __init__(self, num_blocks: int | None = None, block_size: int = 16, ids=None,
                 hash_algo: str = "sha256"):
        L = lib()
        if ids is not None:
            arr = _i32(ids)
            num_blocks = int(arr.size)
            self._h = L.pa_pool_create(num_blocks, block_size, _p32(arr))
        else:
            self._h = L.pa_pool_create(int(num_blocks), block_size, None)
        if not self._h:
            raise ValueError("pa_pool_create rejected its arguments")
        if hash_algo not in HASH_ALGOS:
            L.pa_pool_destroy(self._h)
            self._h = None
            raise ValueError(f"unknown hash algorithm {hash_algo!r}")
        _check(L.pa_pool_set_hash_algo(self._h, HASH_ALGOS[hash_algo]), "pa_pool_set_hash_algo")
        # one-element lists shared with the schedulers drawing from this pool,
        # each holding that scheduler's handle until it is destroyed
        self._sched_cells = []

    def close(self) -> None:
        if getattr(self, "_h", None):
            # A scheduler releases its blocks into the pool when destroyed, so
            # any still open goes first: finalizers of objects collected
            # together may run in any order.
            for cell in self._sched_cells:
                _destroy_sched(cell)
            lib().pa_pool_destroy(self._h)
            self._h = None

    __del__ = close

    @property
    def handle(self):
        return self._h

    @property
    def hash_algo(self) -> str:
        v = lib().pa_pool_hash_algo(self._h)
        return next(k for k, a in HASH_ALGOS.items() if a == v)

    def set_hash_algo(self, algo: str) -> None:
        """Only while no block holds a hash."""
        _check(lib().pa_pool_set_hash_algo(self._h, HASH_ALGOS[algo]), "pa_pool_set_hash_algo")

    def num_free(self) -> int:
        return lib().pa_pool_num_free(self._h)

    def num_blocks(self) -> int:
        return lib().pa_pool_num_blocks(self._h)

    def allocate(self, n: int) -> list:
        out = np.empty(max(n, 1), np.int32)
        st = lib().pa_pool_allocate(self._h, n, _p32(out))
        if st == -5:
            raise MemoryError("No free KV block")
        _check(st, "pa_pool_allocate")
        return out[:n].tolist()

    def release(self, ids) -> None:
        a = _i32(ids)
        _check(lib().pa_pool_free(self._h, _p32(a), int(a.size)), "pa_pool_free")

    def touch(self, ids) -> None:
        a = _i32(ids)
        _check(lib().pa_pool_touch(self._h, _p32(a), int(a.size)), "pa_pool_touch")

    def cache_block(self, block: int, h: bytes) -> None:
        _check(lib().pa_pool_cache_block(self._h, block, bytes(h)), "pa_pool_cache_block")

    def lookup(self, h: bytes) -> int:
        return int(lib().pa_pool_lookup(self._h, bytes(h)))

    def ref_count(self, block: int) -> int:
        return int(lib().pa_pool_ref_count(self._h, block))

    def is_cached(self, block: int) -> bool:
        v = lib().pa_pool_is_cached(self._h, block)
        if v < 0:
            raise KeyError(block)
        return bool(v)

    def free_queue(self) -> list:
        n = lib().pa_pool_free_queue(self._h, None, 0)
        out = np.empty(max(n, 1), np.int32)
        lib().pa_pool_free_queue(self._h, _p32(out), n)
        return out[:n].tolist()

    def find_cached_prefix(self, tokens, extra: bytes = b"") -> list:
        t = _i32(tokens)
        out = np.empty(max(int(t.size), 1), np.int32)
        n = lib().pa_pool_find_cached_prefix(self._h, _p32(t), int(t.size), bytes(extra) or None,
                                             len(extra), _p32(out), int(out.size))
        if n < 0:
            _check(n, "pa_pool_find_cached_prefix")
        bs = lib().pa_pool_block_size(self._h)
        return out[:n // bs].tolist()


def _destroy_sched(cell: list) -> None:
    if cell[0]:
        h, cell[0] = cell[0], None
        lib().pa_sched_destroy(h)


class Scheduler:
    """pa_sched_*: the token-budget scheduler over a :class:`BlockPool`."""

    def __init__(self, pool: BlockPool, *, token_budget: int, max_model_len: int,
                 max_running: int = 0, long_prefill_threshold: int = 0,
                 max_blocks_per_req: int | None = None, prefix_caching: bool = True,
                 chunked_prefill: bool = True, max_reqs: int = 4096,
                 retained_block_tables: bool = False):
        bs = lib().pa_pool_block_size(pool.handle)
        self.stride = max_blocks_per_req or -(-max_model_len // bs)
        self.cfg = SchedConfig(token_budget, max_running, long_prefill_threshold, max_model_len,
                               self.stride, int(prefix_caching), int(chunked_prefill))
        self.retained = bool(retained_block_tables)
        self.pool = pool  # keeps the pool alive
        h = lib().pa_sched_create(pool.handle, ctypes.byref(self.cfg))
        if not h:
            raise ValueError("pa_sched_create rejected its configuration")
        self._cell = [h]  # shared with the pool, which may destroy it first
        pool._sched_cells.append(self._cell)
        self._alloc(max_reqs)

    @property
    def _h(self):
        h = self._cell[0]
        if not h:
            raise RuntimeError("scheduler closed (or its pool was)")
        return h

    def _alloc(self, max_reqs: int) -> None:
        T = self.cfg.token_budget
        self._arrays = dict(
            req_ids=np.empty(max_reqs, np.int64), num_scheduled=np.empty(max_reqs, np.int32),
            num_computed=np.empty(max_reqs, np.int32),
            query_start_loc=np.empty(max_reqs + 1, np.int32),
            seq_lens=np.empty(max_reqs, np.int32),
            block_tables=np.empty(max_reqs * self.stride, np.int32),
            slot_mapping=np.empty(T, np.int64), positions=np.empty(T, np.int32),
            input_tokens=np.empty(T, np.int32), preempted_ids=np.empty(max_reqs, np.int64))
        a = self._arrays
        o = SchedOutput()
        o.max_reqs, o.max_tokens, o.max_preempted = max_reqs, T, max_reqs
        # retained tables: the buffer is this object's alone (step() returns
        # copies), so the scheduler may leave entries as its last step wrote them
        o.block_tables_retained = int(self.retained)
        for k, v in a.items():
            setattr(o, k, v.ctypes.data_as(_i64p if v.dtype == np.int64 else _i32p))
        self._out = o
        self._max_reqs = max_reqs

    def close(self) -> None:
        cell = getattr(self, "_cell", None)  # absent if the constructor raised
        if cell is not None:
            _destroy_sched(cell)

    __del__ = close

    def add_request(self, req_id: int, prompt, extra: bytes = b"") -> None:
        t = _i32(prompt)
        _check(lib().pa_sched_add_request(self._h, req_id, _p32(t), int(t.size),
                                          bytes(extra) or None, len(extra)),
               "pa_sched_add_request")

    def append_token(self, req_id: int, token: int) -> None:
        _check(lib().pa_sched_append_token(self._h, req_id, token), "pa_sched_append_token")

    def finish(self, req_id: int) -> None:
        _check(lib().pa_sched_finish(self._h, req_id), "pa_sched_finish")

    def num_running(self) -> int:
        return lib().pa_sched_num_running(self._h)

    def num_waiting(self) -> int:
        return lib().pa_sched_num_waiting(self._h)

    def request_state(self, req_id: int) -> dict:
        v = [_c_i(0) for _ in range(5)]
        _check(lib().pa_sched_request_state(self._h, req_id, *[ctypes.byref(x) for x in v]),
               "pa_sched_request_state")
        keys = ("num_computed", "num_tokens", "prompt_len", "num_blocks", "running")
        return {k: int(x.value) for k, x in zip(keys, v)}

    def request_blocks(self, req_id: int) -> list:
        n = lib().pa_sched_request_blocks(self._h, req_id, None, 0)
        if n < 0:
            _check(n, "pa_sched_request_blocks")
        out = np.empty(max(n, 1), np.int32)
        lib().pa_sched_request_blocks(self._h, req_id, _p32(out), n)
        return out[:n].tolist()

    def step(self) -> dict:
        """One step; returns the batch as numpy arrays (copies)."""
        live = self.num_running() + self.num_waiting()
        need = max(min(live, self.cfg.token_budget), self.num_running())
        if need > self._max_reqs:
            self._alloc(need * 2)
        o = self._out
        L, ref = lib(), ctypes.byref(o)
        t0 = time.perf_counter()
        st = L.pa_sched_step(self._h, ref)
        self.last_step_seconds = time.perf_counter() - t0  # the C call alone
        _check(st, "pa_sched_step")
        a, R, T = self._arrays, o.num_reqs, o.num_tokens
        return dict(
            req_ids=a["req_ids"][:R].copy(), num_scheduled=a["num_scheduled"][:R].copy(),
            num_computed=a["num_computed"][:R].copy(),
            query_start_loc=a["query_start_loc"][:R + 1].copy(),
            seq_lens=a["seq_lens"][:R].copy(),
            block_tables=a["block_tables"][:R * o.block_table_stride].reshape(
                R, o.block_table_stride).copy(),
            slot_mapping=a["slot_mapping"][:T].copy(), positions=a["positions"][:T].copy(),
            input_tokens=a["input_tokens"][:T].copy(),
            preempted_ids=a["preempted_ids"][:o.num_preempted].copy(),
            num_tokens=T, max_query_len=o.max_query_len, max_seq_len=o.max_seq_len,
            num_decode_reqs=o.num_decode_reqs, num_context_reqs=o.num_context_reqs,
            num_context_tokens=o.num_context_tokens, num_generation_reqs=o.num_generation_reqs,
            num_generation_tokens=o.num_generation_tokens)


def step_signature(out: dict) -> str:
    """Profile name of a scheduled step, execute_context_A(a)_generation_B(b)
    ("vLLM v1 Deep Dive", Part 3, Step 4c): A requests with a tokens in their
    prompt (prefill), B requests with b tokens past it (decode)."""
    return (f"execute_context_{out['num_context_reqs']}({out['num_context_tokens']})"
            f"_generation_{out['num_generation_reqs']}({out['num_generation_tokens']})")
