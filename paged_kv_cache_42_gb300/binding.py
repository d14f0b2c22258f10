"""Python binding of libpagedattn (ctypes): argument marshalling only.

Every step of the path runs in the library's CUDA kernels; this module checks
tensor dtypes/devices, passes raw device pointers and the current CUDA stream
through the C ABI declared in ``include/pa_api.h``, and turns a non-zero status
into an exception. There is no fallback: if the compiled library is missing
the import-time loader raises.

Function names follow the C ABI: ``pa_write_kv`` -> :func:`write_kv`,
``pa_attention`` -> :func:`attention`, and so on.

The attention calls also take a pinned CPU tensor as ``out``. It is passed by
its mapped device address (``pa_mapped_pointer``), and the kernels store the
result straight into host memory. That overlaps the device-to-host transfer
with the computation::

    host_out = torch.empty(q.shape, dtype=torch.bfloat16).pin_memory()
    attention(q, k_cache, v_cache, block_tables, seq_lens, qsl, scale,
              max_query_len=1, max_seq_len=L, out=host_out)
    torch.cuda.current_stream().synchronize()  # host_out now holds the result
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

_LIB = None

_c_p = ctypes.c_void_p
_c_i = ctypes.c_int

STATUS = {0: "PA_OK", -1: "PA_ERR_INVALID_ARG", -2: "PA_ERR_UNSUPPORTED",
          -3: "PA_ERR_WORKSPACE", -4: "PA_ERR_CUDA", -5: "PA_ERR_BOUNDS", -6: "PA_ERR_TIMEOUT"}
DEVICE_ERRORS = {0: "none", 1: "slot outside the pool", 2: "block id outside the pool",
                 3: "inconsistent lengths", 4: "query_start_loc out of range",
                 5: "bounded wait timed out", 6: "table does not start with the common prefix"}
KERNEL_IDS = {"write_kv": 0, "plan": 1, "decode": 2, "prefill": 3, "prefix": 4, "merge": 5}


class PagedAttentionError(RuntimeError):
    def __init__(self, status: int, what: str):
        super().__init__(f"{what}: {STATUS.get(status, status)}")
        self.status = status


def library_path() -> str:
    return _build.LIB_PATH


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m paged_kv_cache_42_gb300.build` "
                "(there is no CPU fallback)")
        L = ctypes.CDLL(path)
        L.pa_init.argtypes = []
        L.pa_init.restype = _c_i
        L.pa_write_kv.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, _c_i, _c_i, _c_i, _c_i, _c_i, _c_p]
        L.pa_write_kv.restype = _c_i
        L.pa_attention_workspace_size.argtypes = [_c_i, _c_i, _c_i, _c_i, _c_i]
        L.pa_attention_workspace_size.restype = ctypes.c_size_t
        L.pa_attention.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, ctypes.c_float, _c_p,
                                   _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i,
                                   _c_p, ctypes.c_size_t, _c_p]
        L.pa_attention.restype = _c_i
        L.pa_attention_cascade_workspace_size.argtypes = [_c_i, _c_i, _c_i, _c_i, _c_i]
        L.pa_attention_cascade_workspace_size.restype = ctypes.c_size_t
        L.pa_attention_cascade.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, ctypes.c_float,
                                           _c_p, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i,
                                           _c_i, _c_i, _c_i, _c_p, ctypes.c_size_t, _c_p]
        L.pa_attention_cascade.restype = _c_i
        L.pa_write_kv_fp8.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, ctypes.c_float,
                                      ctypes.c_float, _c_i, _c_i, _c_i, _c_i, _c_i, _c_p]
        L.pa_write_kv_fp8.restype = _c_i
        L.pa_attention_fp8.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, ctypes.c_float,
                                       ctypes.c_float, ctypes.c_float, _c_p, _c_i, _c_i, _c_i,
                                       _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_p,
                                       ctypes.c_size_t, _c_p]
        L.pa_attention_fp8.restype = _c_i
        L.pa_status_string.argtypes = [_c_i]
        L.pa_status_string.restype = ctypes.c_char_p
        L.pa_get_device_error.argtypes = [ctypes.POINTER(_c_i), ctypes.POINTER(ctypes.c_longlong),
                                          _c_i]
        L.pa_get_device_error.restype = _c_i
        L.pa_set_kernel_timer.argtypes = [_c_i, _c_p, _c_p]
        L.pa_set_kernel_timer.restype = _c_i
        L.pa_mapped_pointer.argtypes = [_c_p, ctypes.POINTER(ctypes.c_void_p)]
        L.pa_mapped_pointer.restype = _c_i
        L.pa_launch_count.argtypes = []
        L.pa_launch_count.restype = ctypes.c_longlong
        L.pa_version.argtypes = []
        L.pa_version.restype = _c_i
        _LIB = L
    return _LIB


def _check(status: int, what: str) -> None:
    if status != 0:
        raise PagedAttentionError(status, what)


def _stream_ptr(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return int(stream.cuda_stream)


def _dev(t: torch.Tensor, dtype, name: str) -> int:
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _out(t: torch.Tensor) -> int:
    """Address of an output tensor: a CUDA tensor, or a pinned CPU tensor
    reached through its mapped device address (pa_mapped_pointer)."""
    if isinstance(t, torch.Tensor) and not t.is_cuda:
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise TypeError("out must be a contiguous bf16 tensor")
        if not t.is_pinned():
            raise ValueError("a host out tensor must be pinned")
        return mapped_pointer(t)
    return _dev(t, torch.bfloat16, "out")


def mapped_pointer(t: torch.Tensor) -> int:
    """pa_mapped_pointer: the device address of a pinned host tensor."""
    dp = ctypes.c_void_p()
    _check(lib().pa_mapped_pointer(t.data_ptr(), ctypes.byref(dp)), "pa_mapped_pointer")
    return int(dp.value)


def status_string(status: int) -> str:
    return lib().pa_status_string(status).decode()


def init() -> None:
    _check(lib().pa_init(), "pa_init")


def write_kv(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
             k_cache: torch.Tensor, v_cache: torch.Tensor, stream=None) -> None:
    """pa_write_kv: scatter k/v [T, Hkv, D] into caches [num_blocks, Hkv, 16, D]."""
    T, hkv, d = k.shape
    nb, hkv2, bs, d2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or hkv2 != hkv or d2 != d:
        raise ValueError("shape mismatch between k/v and the caches")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    st = lib().pa_write_kv(_dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
                           _dev(slot_mapping, torch.int64, "slot_mapping"),
                           _dev(k_cache, torch.bfloat16, "k_cache"),
                           _dev(v_cache, torch.bfloat16, "v_cache"), T, hkv, d, bs, nb,
                           _stream_ptr(stream))
    _check(st, "pa_write_kv")


def workspace_size(num_reqs: int, num_tokens: int, num_q_heads: int, num_kv_heads: int,
                   head_dim: int) -> int:
    return int(lib().pa_attention_workspace_size(num_reqs, num_tokens, num_q_heads,
                                                 num_kv_heads, head_dim))


def attention(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
              block_tables: torch.Tensor, seq_lens: torch.Tensor,
              query_start_loc: torch.Tensor, scale: float, *, max_query_len: int,
              max_seq_len: int, out: torch.Tensor | None = None,
              workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """pa_attention for a mixed batch; returns ``out`` [T, Hq, D] bf16.

    ``workspace`` (uint8, >= workspace_size(...) bytes) is allocated here with
    torch if not given; pass a persistent one on hot loops.
    """
    T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    R = int(seq_lens.shape[0])
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q and the caches")
    if query_start_loc.shape != (R + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != R:
        raise ValueError("metadata shapes must be qsl [R+1], block_tables [R, max_blocks]")
    if out is None:
        out = torch.empty_like(q)
    need = workspace_size(R, T, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().pa_attention(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_tables, torch.int32, "block_tables"),
        _dev(seq_lens, torch.int32, "seq_lens"),
        _dev(query_start_loc, torch.int32, "query_start_loc"), float(scale),
        _out(out), R, T, hq, hkv, d, bs, nb, int(block_tables.shape[1]),
        int(max_query_len), int(max_seq_len), _dev(workspace, torch.uint8, "workspace"),
        int(workspace.numel()), _stream_ptr(stream))
    _check(st, "pa_attention")
    return out


def write_kv_fp8(k: torch.Tensor, v: torch.Tensor, slot_mapping: torch.Tensor,
                 k_cache: torch.Tensor, v_cache: torch.Tensor, k_scale: float, v_scale: float,
                 stream=None) -> None:
    """pa_write_kv_fp8: quantise k/v [T, Hkv, D] bf16 into E4M3 caches
    [num_blocks, Hkv, 16, D] (uint8) with per-tensor scales."""
    T, hkv, d = k.shape
    nb, hkv2, bs, d2 = k_cache.shape
    if v.shape != k.shape or v_cache.shape != k_cache.shape or hkv2 != hkv or d2 != d:
        raise ValueError("shape mismatch between k/v and the caches")
    if slot_mapping.shape != (T,):
        raise ValueError("slot_mapping must be [num_tokens]")
    st = lib().pa_write_kv_fp8(_dev(k, torch.bfloat16, "k"), _dev(v, torch.bfloat16, "v"),
                               _dev(slot_mapping, torch.int64, "slot_mapping"),
                               _dev(k_cache, torch.uint8, "k_cache"),
                               _dev(v_cache, torch.uint8, "v_cache"), float(k_scale),
                               float(v_scale), T, hkv, d, bs, nb, _stream_ptr(stream))
    _check(st, "pa_write_kv_fp8")


def attention_fp8(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                  block_tables: torch.Tensor, seq_lens: torch.Tensor,
                  query_start_loc: torch.Tensor, scale: float, k_scale: float, v_scale: float,
                  *, max_query_len: int, max_seq_len: int, out: torch.Tensor | None = None,
                  workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """pa_attention_fp8 over E4M3 caches (uint8 [num_blocks, Hkv, 16, D])."""
    T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    R = int(seq_lens.shape[0])
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q and the caches")
    if query_start_loc.shape != (R + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != R:
        raise ValueError("metadata shapes must be qsl [R+1], block_tables [R, max_blocks]")
    if out is None:
        out = torch.empty_like(q)
    need = workspace_size(R, T, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().pa_attention_fp8(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.uint8, "k_cache"),
        _dev(v_cache, torch.uint8, "v_cache"), _dev(block_tables, torch.int32, "block_tables"),
        _dev(seq_lens, torch.int32, "seq_lens"),
        _dev(query_start_loc, torch.int32, "query_start_loc"), float(scale), float(k_scale),
        float(v_scale), _out(out), R, T, hq, hkv, d, bs, nb,
        int(block_tables.shape[1]), int(max_query_len), int(max_seq_len),
        _dev(workspace, torch.uint8, "workspace"), int(workspace.numel()), _stream_ptr(stream))
    _check(st, "pa_attention_fp8")
    return out


def cascade_workspace_size(num_reqs: int, num_tokens: int, num_q_heads: int, num_kv_heads: int,
                           head_dim: int) -> int:
    return int(lib().pa_attention_cascade_workspace_size(num_reqs, num_tokens, num_q_heads,
                                                         num_kv_heads, head_dim))


def attention_cascade(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor,
                      query_start_loc: torch.Tensor, scale: float, *, common_prefix_len: int,
                      max_query_len: int, max_seq_len: int, out: torch.Tensor | None = None,
                      workspace: torch.Tensor | None = None, stream=None) -> torch.Tensor:
    """pa_attention_cascade: every request shares the first ``common_prefix_len``
    keys (the same blocks); the prefix is attended once for the whole batch."""
    T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    R = int(seq_lens.shape[0])
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q and the caches")
    if query_start_loc.shape != (R + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != R:
        raise ValueError("metadata shapes must be qsl [R+1], block_tables [R, max_blocks]")
    if out is None:
        out = torch.empty_like(q)
    need = cascade_workspace_size(R, T, hq, hkv, d)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=q.device)
    st = lib().pa_attention_cascade(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_tables, torch.int32, "block_tables"),
        _dev(seq_lens, torch.int32, "seq_lens"),
        _dev(query_start_loc, torch.int32, "query_start_loc"), float(scale),
        _out(out), R, T, hq, hkv, d, bs, nb, int(block_tables.shape[1]),
        int(max_query_len), int(max_seq_len), int(common_prefix_len),
        _dev(workspace, torch.uint8, "workspace"), int(workspace.numel()), _stream_ptr(stream))
    _check(st, "pa_attention_cascade")
    return out


def get_device_error(clear: bool = True) -> tuple[int, int]:
    """(code, detail) of the device error word (synchronises)."""
    code = _c_i(0)
    detail = ctypes.c_longlong(0)
    _check(lib().pa_get_device_error(ctypes.byref(code), ctypes.byref(detail), int(clear)),
           "pa_get_device_error")
    return int(code.value), int(detail.value)


def set_kernel_timer(kernel: str, start: torch.cuda.Event | None,
                     stop: torch.cuda.Event | None) -> None:
    """Record CUDA events around every later launch of one library kernel."""
    sp = None if start is None else ctypes.c_void_p(start.cuda_event)
    ep = None if stop is None else ctypes.c_void_p(stop.cuda_event)
    _check(lib().pa_set_kernel_timer(KERNEL_IDS[kernel], sp, ep), "pa_set_kernel_timer")


OPTIONS = {"decode_self_plan": 1, "decode_tc": 2, "decode_max_workers": 3, "mixed_overlap": 4, "decode_token_major": 5, "cascade_overlap": 6, "decode_tm_ctas_per_sm": 7, "mixed_prefill_ctas": 8}


def set_option(name: str, value: int) -> None:
    """pa_set_option: process-wide library options (see include/pa_api.h)."""
    L = lib()
    L.pa_set_option.argtypes = [_c_i, _c_i]
    L.pa_set_option.restype = _c_i
    _check(L.pa_set_option(OPTIONS[name], int(value)), "pa_set_option")


def launch_count() -> int:
    return int(lib().pa_launch_count())


def noalloc_scratch_bytes() -> int:
    """Size of the fixed scratch array behind :func:`attention_noalloc`."""
    L = lib()
    L.pa_noalloc_scratch_bytes.argtypes = []
    L.pa_noalloc_scratch_bytes.restype = ctypes.c_size_t
    return int(L.pa_noalloc_scratch_bytes())


def attention_noalloc(q: torch.Tensor, k_cache: torch.Tensor, v_cache: torch.Tensor,
                      block_tables: torch.Tensor, seq_lens: torch.Tensor,
                      query_start_loc: torch.Tensor, scale: float, *, max_query_len: int,
                      max_seq_len: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """pa_attention_noalloc: attention with the library's fixed scratch array
    as workspace, for callers that cannot allocate device memory.

    Nothing is allocated by the call (``out`` must be given). Batches larger
    than the scratch array raise PA_ERR_WORKSPACE; calls that overlap on the
    GPU share the scratch and must be serialised by the caller.
    """
    L = lib()
    L.pa_attention_noalloc.argtypes = [_c_p, _c_p, _c_p, _c_p, _c_p, _c_p, ctypes.c_float, _c_p,
                                       _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i, _c_i,
                                       _c_i, _c_p]
    L.pa_attention_noalloc.restype = _c_i
    T, hq, d = q.shape
    nb, hkv, bs, d2 = k_cache.shape
    R = int(seq_lens.shape[0])
    if d2 != d or v_cache.shape != k_cache.shape:
        raise ValueError("shape mismatch between q and the caches")
    if query_start_loc.shape != (R + 1,) or block_tables.dim() != 2 or block_tables.shape[0] != R:
        raise ValueError("metadata shapes must be qsl [R+1], block_tables [R, max_blocks]")
    if out.shape != q.shape:
        raise ValueError("out must have q's shape")
    st = L.pa_attention_noalloc(
        _dev(q, torch.bfloat16, "q"), _dev(k_cache, torch.bfloat16, "k_cache"),
        _dev(v_cache, torch.bfloat16, "v_cache"), _dev(block_tables, torch.int32, "block_tables"),
        _dev(seq_lens, torch.int32, "seq_lens"),
        _dev(query_start_loc, torch.int32, "query_start_loc"), float(scale),
        _out(out), R, T, hq, hkv, d, bs, nb, int(block_tables.shape[1]),
        int(max_query_len), int(max_seq_len), _stream_ptr(stream))
    _check(st, "pa_attention_noalloc")
    return out
