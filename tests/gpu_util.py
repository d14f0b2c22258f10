"""Helpers for the GPU tests: move a seeded workload to the device, run the
library through its binding, compare with the CPU oracle."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from paged_kv_cache_42_gb300 import binding
from paged_kv_cache_42_gb300 import workloads as wl

# bf16 attention output vs the float64 oracle (spec tolerances)
MAX_ABS = 2e-2
MEAN_ABS = 2e-3


def bf16_tensor(bits: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def to_bits(t: torch.Tensor) -> np.ndarray:
    return t.detach().view(torch.int16).cpu().numpy().view(np.uint16)


def to_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


class DeviceBatch:
    """A workload resident on the GPU."""

    def __init__(self, w: wl.Workload, device="cuda"):
        self.w = w
        self.q = bf16_tensor(w.q, device)
        self.k = bf16_tensor(w.k_new, device)
        self.v = bf16_tensor(w.v_new, device)
        self.k_cache = bf16_tensor(w.k_cache, device)
        self.v_cache = bf16_tensor(w.v_cache, device)
        self.block_tables = torch.from_numpy(w.block_tables).to(device)
        self.seq_lens = torch.from_numpy(w.seq_lens).to(device)
        self.qsl = torch.from_numpy(w.query_start_loc).to(device)
        self.slot_mapping = torch.from_numpy(w.slot_mapping).to(device)
        self.out = torch.full_like(self.q, float("nan"))
        self.workspace = torch.empty(
            binding.workspace_size(w.num_reqs, w.num_tokens, w.num_q_heads, w.num_kv_heads,
                                   w.head_dim), dtype=torch.uint8, device=device)

    def write(self):
        binding.write_kv(self.k, self.v, self.slot_mapping, self.k_cache, self.v_cache)

    def attend(self, out=None):
        w = self.w
        return binding.attention(self.q, self.k_cache, self.v_cache, self.block_tables,
                                 self.seq_lens, self.qsl, w.scale, max_query_len=w.max_query_len,
                                 max_seq_len=w.max_seq_len, out=self.out if out is None else out,
                                 workspace=self.workspace)

    def step(self):
        self.write()
        return self.attend()


def oracle_reference(w: wl.Workload, reqs=None) -> np.ndarray:
    """Oracle result after this step's write (on a CPU copy of the caches)."""
    kc = w.k_cache.copy()
    vc = w.v_cache.copy()
    oracle.write_kv(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    return oracle.attention(w.q, kc, vc, w.block_tables, w.seq_lens, w.query_start_loc, w.scale,
                            reqs=reqs)


def rows_of(w: wl.Workload, reqs) -> np.ndarray:
    return np.concatenate([np.arange(w.query_start_loc[r], w.query_start_loc[r + 1])
                           for r in reqs]).astype(np.int64)


def assert_close(got: np.ndarray, ref: np.ndarray, what: str = ""):
    assert got.shape == ref.shape
    assert np.isfinite(got).all(), f"{what}: non-finite output (read outside valid KV?)"
    err = np.abs(got - ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= MAX_ABS and mean <= MEAN_ABS, f"{what}: max abs {mx:.3g}, mean abs {mean:.3g}"
    return mx, mean


def check_no_device_error():
    code, detail = binding.get_device_error(clear=True)
    assert code == 0, f"device error {binding.DEVICE_ERRORS.get(code, code)} at {detail}"
