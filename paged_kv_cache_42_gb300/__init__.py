"""Attention over a paged KV cache for NVIDIA GB300 (sm_103a).

The compute lives in ``libpagedattn.so`` (CUDA C++, C ABI, see
``include/pa_api.h``); :mod:`paged_kv_cache_42_gb300.binding` marshals torch
tensors into it. :mod:`paged_kv_cache_42_gb300.workloads` draws seeded
synthetic inputs.
"""

__all__ = ["binding", "workloads"]
