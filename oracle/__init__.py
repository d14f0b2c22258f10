"""CPU oracle for attention over a paged KV cache (ctypes front end).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline arm use this package; the product library never
imports, links or calls it, and it imports nothing from the product.

The arithmetic lives in ``pa_oracle.c`` (plain C, double precision, the plain
definition of the KV scatter and of causal softmax attention over each
request's block-table-gathered K/V). This module only marshals numpy arrays.
bf16 tensors are handled as their raw ``uint16`` bit patterns.
"""
from __future__ import annotations

import ctypes
import os

import numpy as np

from . import build as _build

_LIBS: dict = {}

_ERRORS = {1: "bad argument", 2: "slot outside the pool", 3: "block id outside the pool",
           4: "seq_len shorter than the query span", 5: "out of memory"}


class OracleError(RuntimeError):
    pass


def load(mutant: int = 0, out_dir: str | None = None) -> ctypes.CDLL:
    key = (mutant, out_dir)
    if key not in _LIBS:
        path = _build.build(mutant=mutant, out_dir=out_dir)
        lib = ctypes.CDLL(path)
        p = ctypes.c_void_p
        i = ctypes.c_int
        lib.oracle_write_kv.argtypes = [p, p, p, p, p, i, i, i, i, i]
        lib.oracle_write_kv.restype = i
        lib.oracle_attention.argtypes = [p, p, p, p, i, p, p, ctypes.c_double, p,
                                         i, i, i, i, i, i, p, i, i]
        lib.oracle_attention.restype = i
        lib.oracle_mutant_id.restype = i
        lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
        lib.oracle_e4m3_value.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
        lib.oracle_e4m3_encode.restype = ctypes.c_uint8
        lib.oracle_e4m3_quantize.argtypes = [p, ctypes.c_float, p, ctypes.c_int64]
        lib.oracle_e4m3_quantize.restype = None
        lib.oracle_write_kv_fp8.argtypes = [p, p, p, p, p, ctypes.c_float, ctypes.c_float,
                                            i, i, i, i, i]
        lib.oracle_write_kv_fp8.restype = i
        lib.oracle_attention_fp8.argtypes = [p, p, p, ctypes.c_double, ctypes.c_double, p, i, p,
                                             p, ctypes.c_double, p, i, i, i, i, i, i, p, i, i]
        lib.oracle_attention_fp8.restype = i
        _LIBS[key] = lib
    return _LIBS[key]


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle arrays must be C-contiguous"
    return a.ctypes.data


def write_kv(k, v, slot_mapping, k_cache, v_cache, *, lib=None) -> None:
    """Scatter new K/V rows into the caches in place (bit copy).

    k, v: uint16 [T, Hkv, D]; slot_mapping: int64 [T]; caches: uint16
    [num_blocks, Hkv, block_size, D].
    """
    lib = lib or load()
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert k_cache.dtype == np.uint16 and v_cache.dtype == np.uint16
    nb, hkv, bs, d = k_cache.shape
    st = lib.oracle_write_kv(_ptr(k), _ptr(v), _ptr(sm), _ptr(k_cache), _ptr(v_cache),
                             int(sm.shape[0]), hkv, d, bs, nb)
    if st:
        raise OracleError(_ERRORS.get(st, str(st)))


def attention(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, *,
              reqs=None, threads: int | None = None, out=None, lib=None) -> np.ndarray:
    """Exact causal softmax attention per request, in float64.

    q: uint16 [T, Hq, D]; caches uint16 [num_blocks, Hkv, bs, D];
    block_tables int32 [R, max_blocks]; seq_lens int32 [R];
    query_start_loc int32 [R+1]. Returns float64 [T, Hq, D]; rows of requests
    not listed in ``reqs`` stay NaN (or keep ``out``'s values).
    """
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d == d2
    if out is None:
        out = np.full((T, hq, d), np.nan, dtype=np.float64)
    rl = None
    if reqs is not None:
        rl = np.ascontiguousarray(np.asarray(reqs, dtype=np.int32))
    threads = threads or os.cpu_count() or 1
    st = lib.oracle_attention(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt), int(bt.shape[1]),
                              _ptr(sl), _ptr(qsl), float(scale), _ptr(out), int(sl.shape[0]),
                              hq, hkv, d, bs, nb,
                              None if rl is None else _ptr(rl),
                              0 if rl is None else int(rl.shape[0]), int(threads))
    if st:
        raise OracleError(_ERRORS.get(st, str(st)))
    return out


# ---------------------------------------------------------------------------
# FP8 (E4M3) KV cache
# ---------------------------------------------------------------------------
def e4m3_value(code: int, *, lib=None) -> float:
    """Value of one E4M3 code (OCP 8-bit format, max 448, no infinities)."""
    return float((lib or load()).oracle_e4m3_value(int(code) & 0xFF))


def e4m3_encode(y: float, *, lib=None) -> int:
    """Nearest E4M3 code to the binary32 value y (ties to even, saturating)."""
    return int((lib or load()).oracle_e4m3_encode(float(y)))


def e4m3_quantize(x_bits, scale: float, *, lib=None) -> np.ndarray:
    """E4M3 codes of bf16 values x / scale (quotient in binary32)."""
    lib = lib or load()
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    out = np.empty(x.shape, dtype=np.uint8)
    lib.oracle_e4m3_quantize(_ptr(x), float(scale), _ptr(out), int(x.size))
    return out


def write_kv_fp8(k, v, slot_mapping, k_cache, v_cache, k_scale: float, v_scale: float, *,
                 lib=None) -> None:
    """Quantising scatter into uint8 E4M3 caches [num_blocks, Hkv, bs, D], in place."""
    lib = lib or load()
    k = np.ascontiguousarray(k, dtype=np.uint16)
    v = np.ascontiguousarray(v, dtype=np.uint16)
    sm = np.ascontiguousarray(slot_mapping, dtype=np.int64)
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    nb, hkv, bs, d = k_cache.shape
    st = lib.oracle_write_kv_fp8(_ptr(k), _ptr(v), _ptr(sm), _ptr(k_cache), _ptr(v_cache),
                                 float(k_scale), float(v_scale), int(sm.shape[0]), hkv, d, bs, nb)
    if st:
        raise OracleError(_ERRORS.get(st, str(st)))


def attention_fp8(q, k_cache, v_cache, k_scale: float, v_scale: float, block_tables, seq_lens,
                  query_start_loc, scale, *, reqs=None, threads: int | None = None, out=None,
                  lib=None) -> np.ndarray:
    """Attention over E4M3 caches (keys code * k_scale, values code * v_scale),
    in float64; otherwise as :func:`attention`."""
    lib = lib or load()
    q = np.ascontiguousarray(q, dtype=np.uint16)
    bt = np.ascontiguousarray(block_tables, dtype=np.int32)
    sl = np.ascontiguousarray(seq_lens, dtype=np.int32)
    qsl = np.ascontiguousarray(query_start_loc, dtype=np.int32)
    assert k_cache.dtype == np.uint8 and v_cache.dtype == np.uint8
    T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    assert d == d2
    if out is None:
        out = np.full((T, hq, d), np.nan, dtype=np.float64)
    rl = None
    if reqs is not None:
        rl = np.ascontiguousarray(np.asarray(reqs, dtype=np.int32))
    threads = threads or os.cpu_count() or 1
    st = lib.oracle_attention_fp8(_ptr(q), _ptr(k_cache), _ptr(v_cache), float(k_scale),
                                  float(v_scale), _ptr(bt), int(bt.shape[1]), _ptr(sl), _ptr(qsl),
                                  float(scale), _ptr(out), int(sl.shape[0]), hq, hkv, d, bs, nb,
                                  None if rl is None else _ptr(rl),
                                  0 if rl is None else int(rl.shape[0]), int(threads))
    if st:
        raise OracleError(_ERRORS.get(st, str(st)))
    return out
