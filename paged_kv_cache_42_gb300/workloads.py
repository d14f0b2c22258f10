"""Seeded synthetic workloads for paged-KV attention.

This module only draws inputs: block assignments, lengths, the per-token
slot_mapping a scheduler would hand the kernels, and bf16 values. It holds
none of the attention arithmetic, and both the CUDA path's tests and the CPU
oracle's tests take their inputs from here.

Recipe (every workload):
  * ``numpy.random.Generator(PCG64(seed))``; values are float32 draws from
    N(0, 1) rounded to bf16 round-to-nearest-even and kept as raw uint16 bits.
  * Request r has ``ctx_r`` tokens already cached and ``qlen_r`` new tokens
    this step, so its total length is ``L_r = ctx_r + qlen_r``. It owns
    ``ceil(L_r / 16)`` blocks (on-demand allocation, "Inside the vLLM Engine",
    "A memory problem wearing a throughput costume": 56 tokens -> 4 blocks).
  * Physical block ids come from one random permutation of the pool, taken in
    order: the shared prefix blocks first (if any), then each request's own
    blocks. Pool size is given, or ``ceil(pool_factor * blocks needed)``.
  * Cache slots never assigned, and the slots of this step's new tokens, hold
    a bf16 NaN sentinel; any read outside a request's own valid KV shows up
    as NaN in the output.
  * ``slot_mapping[t]`` for new token j of request r is
    ``block_tables[r][p // 16] * 16 + p % 16`` with p = ctx_r + j ("vLLM v1
    Deep Dive", Part 3, Aside on the KV cache: block_id * block_size + offset).
  * Requests are laid out decode-first (qlen 1 before chunks) where a config
    mixes them, the order the token-budget scheduler emits them in.

Draw order, fixed: block permutation; shared-prefix K then V; for each request
its cached K then V; then q, new k, new v for all T new tokens.
"""
from __future__ import annotations

import dataclasses
import math

import numpy as np

BLOCK_SIZE = 16
BF16_NAN = np.uint16(0x7FC0)


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """float32 -> bf16 bit pattern, round to nearest even (finite inputs)."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    return ((u + (((u >> 16) & 1) + 0x7FFF)) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """bf16 bit pattern -> float32 (exact)."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


@dataclasses.dataclass
class Workload:
    name: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    block_size: int
    num_blocks: int
    ctx_lens: np.ndarray          # int32 [R]
    q_lens: np.ndarray            # int32 [R]
    seq_lens: np.ndarray          # int32 [R]
    query_start_loc: np.ndarray   # int32 [R+1]
    block_tables: np.ndarray      # int32 [R, max_blocks], -1 past each request's blocks
    slot_mapping: np.ndarray      # int64 [T]
    q: np.ndarray                 # uint16 [T, Hq, D]
    k_new: np.ndarray             # uint16 [T, Hkv, D]
    v_new: np.ndarray             # uint16 [T, Hkv, D]
    k_cache: np.ndarray           # uint16 [num_blocks, Hkv, bs, D]
    v_cache: np.ndarray           # uint16 [num_blocks, Hkv, bs, D]
    scale: float
    seed: int
    shared_prefix_blocks: int = 0

    @property
    def num_reqs(self) -> int:
        return int(self.seq_lens.shape[0])

    @property
    def num_tokens(self) -> int:
        return int(self.query_start_loc[-1])

    @property
    def max_blocks_per_req(self) -> int:
        return int(self.block_tables.shape[1])

    @property
    def max_query_len(self) -> int:
        return int(self.q_lens.max()) if self.num_reqs else 0

    @property
    def max_seq_len(self) -> int:
        return int(self.seq_lens.max()) if self.num_reqs else 0

    def blocks_per_req(self) -> np.ndarray:
        return (self.seq_lens.astype(np.int64) + self.block_size - 1) // self.block_size


def make_workload(ctx_lens, q_lens, *, num_q_heads: int, num_kv_heads: int, head_dim: int,
                  seed: int, name: str = "custom", pool_blocks: int | None = None,
                  pool_factor: float = 1.1, shared_prefix_blocks: int = 0,
                  max_blocks_per_req: int | None = None, scale: float | None = None,
                  fill_values: bool = True) -> Workload:
    bs = BLOCK_SIZE
    ctx = np.asarray(ctx_lens, dtype=np.int64)
    ql = np.asarray(q_lens, dtype=np.int64)
    assert ctx.shape == ql.shape and (ctx >= 0).all() and (ql >= 0).all()
    R = int(ctx.shape[0])
    L = ctx + ql
    nb = (L + bs - 1) // bs
    P = int(shared_prefix_blocks)
    if P:
        # every request's first P blocks are the same physical blocks, fully cached
        assert (ctx >= P * bs).all(), "shared prefix must be cached in every request"
    private = nb - P if P else nb
    needed = P + int(private.sum())
    if pool_blocks is None:
        pool_blocks = int(math.ceil(pool_factor * needed))
    assert pool_blocks >= needed, "pool smaller than the blocks needed"
    mb = int(max_blocks_per_req or max(1, int(nb.max()) if R else 1))
    assert R == 0 or mb >= int(nb.max())

    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(pool_blocks).astype(np.int32)
    shared_ids = perm[:P]
    bt = np.full((R, mb), -1, dtype=np.int32)
    cur = P
    for r in range(R):
        n = int(private[r])
        if P:
            bt[r, :P] = shared_ids
            bt[r, P:P + n] = perm[cur:cur + n]
        else:
            bt[r, :n] = perm[cur:cur + n]
        cur += n

    Hq, Hkv, D = int(num_q_heads), int(num_kv_heads), int(head_dim)
    k_cache = np.full((pool_blocks, Hkv, bs, D), BF16_NAN, dtype=np.uint16)
    v_cache = np.full((pool_blocks, Hkv, bs, D), BF16_NAN, dtype=np.uint16)

    def draw(n_tok: int, heads: int) -> np.ndarray:
        return to_bf16_bits(rng.standard_normal((n_tok, heads, D), dtype=np.float32))

    def put(cache: np.ndarray, ids: np.ndarray, vals: np.ndarray) -> None:
        # vals: [n, Hkv, D] for logical positions 0..n-1 of the block list ids
        n = vals.shape[0]
        nf = n // bs
        if nf:
            cache[ids[:nf]] = vals[:nf * bs].reshape(nf, bs, Hkv, D).transpose(0, 2, 1, 3)
        rem = n - nf * bs
        if rem:
            cache[ids[nf], :, :rem, :] = vals[nf * bs:].transpose(1, 0, 2)

    if fill_values:
        if P:
            kp = draw(P * bs, Hkv)
            vp = draw(P * bs, Hkv)
            put(k_cache, shared_ids, kp)
            put(v_cache, shared_ids, vp)
        for r in range(R):
            start = P * bs if P else 0
            n = int(ctx[r]) - start
            if n <= 0:
                continue
            kr = draw(n, Hkv)
            vr = draw(n, Hkv)
            # positions start .. ctx-1 live in blocks start//bs ...
            ids = bt[r, start // bs:]
            put(k_cache, ids, kr)
            put(v_cache, ids, vr)

    qsl = np.zeros(R + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(ql)
    T = int(qsl[-1])
    if fill_values:
        q = draw(T, Hq)
        k_new = draw(T, Hkv)
        v_new = draw(T, Hkv)
    else:
        q = np.zeros((T, Hq, D), dtype=np.uint16)
        k_new = np.zeros((T, Hkv, D), dtype=np.uint16)
        v_new = np.zeros((T, Hkv, D), dtype=np.uint16)

    slot = np.empty(T, dtype=np.int64)
    for r in range(R):
        p = ctx[r] + np.arange(int(ql[r]), dtype=np.int64)
        slot[qsl[r]:qsl[r + 1]] = bt[r, p // bs].astype(np.int64) * bs + p % bs

    return Workload(
        name=name, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=D, block_size=bs,
        num_blocks=int(pool_blocks), ctx_lens=ctx.astype(np.int32), q_lens=ql.astype(np.int32),
        seq_lens=L.astype(np.int32), query_start_loc=qsl.astype(np.int32), block_tables=bt,
        slot_mapping=slot, q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
        scale=float(scale if scale is not None else 1.0 / math.sqrt(D)), seed=int(seed),
        shared_prefix_blocks=P)


# ---------------------------------------------------------------------------
# The five benchmark shapes. Seeds are 42 + the config number.
# ---------------------------------------------------------------------------
CONFIG_NAMES = {
    1: "tiny-decode",
    2: "llama8b-decode",
    3: "mixed-chunked-prefill",
    4: "prefix-share-decode",
    5: "long-context-decode",
}

CONFIG_DESCRIPTIONS = {
    1: "4 seqs, L={9,56,17,33}, Hq 4 / Hkv 2, D 64, bs 16, pool 32 (random permutation), "
       "write newest token then attend",
    2: "64 seqs, L~U[512,4096], Hq 32 / Hkv 8, D 128, bs 16, pool 1.1x needed, random "
       "permutation, write newest token then attend",
    3: "512 decodes L~U[128,2048] + 3 chunks of 512 on ctx {0,1024,2048}, T=2048, "
       "Hq 32 / Hkv 8, D 128, bs 16",
    4: "128 seqs sharing one 64-block (1024-token) prefix, private suffix U[64,512], "
       "Hq 32 / Hkv 8, D 128, bs 16",
    5: "8 seqs x 32768, Hq 64 / Hkv 8, D 128, bs 16, pool 16384 fully permuted",
}


def config_lengths(idx: int, seed: int | None = None):
    """(ctx_lens, q_lens, kwargs) of benchmark config ``idx`` (1..5)."""
    seed = 42 + idx if seed is None else seed
    rng = np.random.Generator(np.random.PCG64(seed + 1_000_003))  # lengths only
    if idx == 1:
        L = np.array([9, 56, 17, 33])
        return L - 1, np.ones(4, np.int64), dict(num_q_heads=4, num_kv_heads=2, head_dim=64,
                                                  pool_blocks=32)
    if idx == 2:
        L = rng.integers(512, 4096, size=64, endpoint=True)
        return L - 1, np.ones(64, np.int64), dict(num_q_heads=32, num_kv_heads=8, head_dim=128)
    if idx == 3:
        Ld = rng.integers(128, 2048, size=512, endpoint=True)
        ctx = np.concatenate([Ld - 1, [0, 1024, 2048]])
        ql = np.concatenate([np.ones(512, np.int64), [512, 512, 512]])
        return ctx, ql, dict(num_q_heads=32, num_kv_heads=8, head_dim=128)
    if idx == 4:
        s = rng.integers(64, 512, size=128, endpoint=True)
        L = 1024 + s
        return L - 1, np.ones(128, np.int64), dict(num_q_heads=32, num_kv_heads=8,
                                                   head_dim=128, shared_prefix_blocks=64)
    if idx == 5:
        L = np.full(8, 32768)
        return L - 1, np.ones(8, np.int64), dict(num_q_heads=64, num_kv_heads=8, head_dim=128,
                                                 pool_blocks=16384)
    raise ValueError(f"unknown config {idx}")


def make_config(idx: int, seed: int | None = None, fill_values: bool = True) -> Workload:
    seed = 42 + idx if seed is None else seed
    ctx, ql, kw = config_lengths(idx, seed)
    return make_workload(ctx, ql, seed=seed, name=CONFIG_NAMES[idx], fill_values=fill_values,
                         **kw)


def permute_physical_blocks(w: Workload, seed: int) -> Workload:
    """Same logical content under a relabelling of physical block ids.

    Block b moves to id perm[b]; the pool and every table entry are permuted
    together, so each request's logical K/V sequence is unchanged.
    """
    rng = np.random.Generator(np.random.PCG64(seed))
    perm = rng.permutation(w.num_blocks).astype(np.int32)
    k2 = np.empty_like(w.k_cache)
    v2 = np.empty_like(w.v_cache)
    k2[perm] = w.k_cache
    v2[perm] = w.v_cache
    bt2 = np.where(w.block_tables >= 0, perm[np.maximum(w.block_tables, 0)], -1).astype(np.int32)
    bs = w.block_size
    slot2 = np.where(w.slot_mapping >= 0,
                     perm[np.maximum(w.slot_mapping, 0) // bs].astype(np.int64) * bs
                     + w.slot_mapping % bs, w.slot_mapping)
    return dataclasses.replace(w, k_cache=k2, v_cache=v2, block_tables=bt2, slot_mapping=slot2)


def unshare_prefix(w: Workload, seed: int) -> Workload:
    """Give every request private copies of its shared prefix blocks.

    The copies take fresh physical ids (the pool grows), with the same content,
    so the logical K/V of every request is unchanged.
    """
    P = w.shared_prefix_blocks
    assert P > 0
    R = w.num_reqs
    extra = R * P
    nb = w.num_blocks + extra
    rng = np.random.Generator(np.random.PCG64(seed))
    new_ids = (w.num_blocks + rng.permutation(extra)).astype(np.int32)
    k2 = np.full((nb,) + w.k_cache.shape[1:], BF16_NAN, dtype=np.uint16)
    v2 = np.full_like(k2, BF16_NAN)
    k2[:w.num_blocks] = w.k_cache
    v2[:w.num_blocks] = w.v_cache
    bt2 = w.block_tables.copy()
    for r in range(R):
        ids = new_ids[r * P:(r + 1) * P]
        k2[ids] = w.k_cache[w.block_tables[r, :P]]
        v2[ids] = w.v_cache[w.block_tables[r, :P]]
        bt2[r, :P] = ids
    return dataclasses.replace(w, k_cache=k2, v_cache=v2, block_tables=bt2, num_blocks=nb,
                               shared_prefix_blocks=0)


def subset_requests(w: Workload, reqs) -> Workload:
    """A batch made of some of ``w``'s requests (same pool, same values)."""
    reqs = np.asarray(reqs, dtype=np.int64)
    ql = w.q_lens[reqs].astype(np.int64)
    qsl = np.zeros(len(reqs) + 1, dtype=np.int64)
    qsl[1:] = np.cumsum(ql)
    rows = np.concatenate([np.arange(w.query_start_loc[r], w.query_start_loc[r + 1])
                           for r in reqs]) if len(reqs) else np.zeros(0, np.int64)
    return dataclasses.replace(
        w, ctx_lens=w.ctx_lens[reqs], q_lens=w.q_lens[reqs], seq_lens=w.seq_lens[reqs],
        query_start_loc=qsl.astype(np.int32), block_tables=w.block_tables[reqs],
        slot_mapping=w.slot_mapping[rows], q=w.q[rows], k_new=w.k_new[rows],
        v_new=w.v_new[rows], shared_prefix_blocks=0)
