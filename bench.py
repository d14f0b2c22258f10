#!/usr/bin/env python3
"""Benchmark: one step of the paged-KV attention hot path on GB300.

A step is the whole path over one synthetic batch: the KV write of this
step's new tokens (pa_write_kv) followed by attention for the batch
(pa_attention: planner + split-KV kernel), with every input resident in HBM
when timing starts. The headline workload is the Llama-3.1-8B-shaped decode
batch (64 sequences, context U[512, 4096], 32 query / 8 KV heads, head_dim
128, block_size 16); `value` is its algorithmic bytes per step divided by the
device time per step (GB/s). The mixed chunked-prefill batch (512 decodes + 3
chunks of 512, T = 2048) is measured in the same run and reported as
tokens/s per layer under "mixed_batch".

Timing: W warm-up steps, then K timed steps; before every step a buffer of
twice the L2 size is written (outside the events) so no step starts with a
warm L2; each step is bracketed by CUDA events on the launching stream. The
decode kernel is also timed on its own (library timer events) for the
roofline. SM clocks and throttle reasons are sampled with nvidia-smi while the
timed loop runs.

`--impl reference` times the CPU oracle (plain C, float64, all host cores) on
a bounded sample of the same workload per step, and prints the same kind of
line with "impl": "reference".

With N > 1 (torchrun), every rank runs its own replica batch of the same
shape (independent requests: weak scaling, no collective on the data path);
timing is the max over ranks.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from paged_kv_cache_42_gb300 import workloads as wl  # noqa: E402

METRIC = "paged-attn decode KV GB/s (frac of HBM peak); mixed-batch tokens/s per layer"
HEADLINE_CONFIG = 2
MIXED_CONFIG = 3
PREFIX_CONFIG = 4
LONG_CONFIG = 5
FP8_SCALES = (0.0113, 0.0127)  # k_scale, v_scale of the E4M3 cache runs
FALLBACK_HBM_GBS = 6800.0


# ---------------------------------------------------------------------------
# algorithmic work of one step (what a perfect implementation must move)
# ---------------------------------------------------------------------------
def step_bytes(w: wl.Workload, fp8: bool = False) -> dict:
    """Bytes one step must move at minimum (no re-reads, no partials); with
    fp8, the cache holds one-byte E4M3 codes instead of bf16."""
    D, Hq, Hkv, T = w.head_dim, w.num_q_heads, w.num_kv_heads, w.num_tokens
    L = w.seq_lens.astype(np.int64)
    nb = (L + 15) // 16
    eb = 1 if fp8 else 2                            # bytes per cached element
    kv = int((L * Hkv * D * 2 * eb).sum())          # K and V rows
    if w.shared_prefix_blocks:
        # unique bytes: the shared prefix blocks are stored (and need reading) once
        P = w.shared_prefix_blocks
        kv_unique = kv - (w.num_reqs - 1) * P * 16 * Hkv * D * 2 * eb
    else:
        kv_unique = kv
    qo = 2 * T * Hq * D * 2                         # q in, out out
    meta = int(nb.sum()) * 4 + w.num_reqs * 8 + 4
    attn = kv + qo + meta
    write = T * Hkv * D * 2 * (2 + eb) + T * 8      # read k,v new (bf16); write cache rows
    return {"kv": kv, "kv_unique": kv_unique, "attention": attn, "write": write,
            "step": attn + write}


def prefill_flops(w: wl.Workload) -> int:
    f = 0
    for r in range(w.num_reqs):
        ql, ctx = int(w.q_lens[r]), int(w.ctx_lens[r])
        if ql > 1:
            f += sum(ctx + j + 1 for j in range(ql)) * w.num_q_heads * 4 * w.head_dim
    return f


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        try:
            d = json.load(open(p))
            return {"hbm_gbs": float(d["hbm_gbs"]), "source": "of measured"}
        except Exception:
            pass
    return {"hbm_gbs": FALLBACK_HBM_GBS, "source": "of fallback"}


# The split-KV kernel a call routes to (the library's default routing): the
# tensor-core kernel for groups of 4 or 8 query heads per KV head at head_dim
# 128, over a bf16 or an E4M3 cache (eight KV heads over E4M3: its
# token-major form), except a cascade's suffix pass; the CUDA-core kernel
# otherwise. Forced ("tensor-core"), it also takes the other
# groups and (bf16) a cascade's suffixes.
def split_kv_kernel(w: wl.Workload, fp8: bool = False, cascade: bool = False,
                    force: str = "auto") -> tuple:
    g = w.num_q_heads // w.num_kv_heads
    tc_ok = w.head_dim == 128 and not (fp8 and cascade)
    if force == "cuda-core" or not tc_ok:
        return "pa_decode_kernel", "decode.cu"
    if force == "tensor-core" or (g >= 4 and not cascade):
        if fp8 and w.num_kv_heads == 8:  # E4M3 over eight KV heads: token-major tiles
            return "pa_decode_tm_kernel", "decode_tm.cu"
        return "pa_decode_tc_kernel", "decode_tc.cu"
    return "pa_decode_kernel", "decode.cu"


def ncu_traffic(workload: str, src_name: str = "decode.cu"):
    """DRAM bytes per split-KV launch from the committed ncu summary, if it
    was taken with that kernel's source as it is now; else None."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    src = os.path.join(ROOT, "paged_kv_cache_42_gb300", "csrc", src_name)
    if not os.path.exists(p):
        return None
    try:
        d = json.load(open(p))
        sha = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
        e = d.get(workload)
        if e and e.get("source_sha", e.get("decode_cu_sha")) == sha and \
                e.get("source", "decode.cu") == src_name:
            return float(e["dram_bytes_per_launch"])
    except Exception:
        pass
    return None


# The pages' own figures, quoted as context (system-level; none is a target
# and none was measured on this hardware).
PAGES_CONTEXT = [
    {"figure": "2-4x serving throughput over FasterTransformer and Orca at comparable latency",
     "hardware": "not stated on the pages",
     "source": "Deep Dive - vLLM (leetllm), introduction; Inside the vLLM Engine, "
               "'A memory problem wearing a throughput costume'"},
    {"figure": "20.4-38.2% of KV-cache memory holds token state in prior systems",
     "hardware": "not stated on the pages",
     "source": "Inside the vLLM Engine, 'A memory problem wearing a throughput costume'"},
    {"figure": "under 4% of KV memory wasted with paging (60-80% in prior systems)",
     "hardware": "not stated on the pages",
     "source": "vLLM: An Exhaustive Technical Study for Kernel Engineers, 2.1"},
]


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# distributed plumbing (replicas; one process per GPU)
# ---------------------------------------------------------------------------
def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    if ws <= 1:
        return 0, 1, 0, None
    import torch
    import torch.distributed as dist
    rank = int(os.environ["RANK"])
    local = int(os.environ.get("LOCAL_RANK", rank))
    backend = "nccl" if torch.cuda.is_available() else "gloo"
    if backend == "nccl":
        torch.cuda.set_device(local)
    dist.init_process_group(backend)
    return rank, ws, local, dist


def max_over_ranks(x: float, dist) -> float:
    if dist is None:
        return x
    import torch
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(dist):
    if dist is not None:
        dist.barrier()


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
class Resident:
    """A workload resident on the device plus the pinned host copies used by
    the end-to-end measurement."""

    def __init__(self, w: wl.Workload, torch, binding, cascade_len: int = 0, fp8_scales=None):
        self.w = w
        self.torch = torch
        self.binding = binding
        self.cascade_len = cascade_len  # > 0: attention through pa_attention_cascade
        self.fp8 = fp8_scales           # (k_scale, v_scale): an E4M3 cache
        self.signature = workload_signature(w)  # the NVTX range name of a step
        dev = torch.device("cuda")

        def bf(bits):
            return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)

        # The per-step inputs live in one pinned host buffer and one device
        # buffer (each tensor a 256-byte-aligned view), so a step's inputs
        # cross PCIe/C2C in a single copy.
        srcs = {"q": bf(w.q), "k": bf(w.k_new), "v": bf(w.v_new),
                "slot_mapping": torch.from_numpy(w.slot_mapping),
                "block_tables": torch.from_numpy(w.block_tables),
                "seq_lens": torch.from_numpy(w.seq_lens),
                "qsl": torch.from_numpy(w.query_start_loc)}
        offs, total = {}, 0
        for name, t in srcs.items():
            offs[name] = total
            total += (t.numel() * t.element_size() + 255) // 256 * 256
        self.h_pack = torch.empty(total, dtype=torch.uint8).pin_memory()
        self.d_pack = torch.empty(total, dtype=torch.uint8, device=dev)

        def view(buf, name, t):
            nbytes = t.numel() * t.element_size()
            return buf[offs[name]:offs[name] + nbytes].view(t.dtype).view(t.shape)

        self.h = {n: view(self.h_pack, n, t) for n, t in srcs.items()}
        self.d = {n: view(self.d_pack, n, t) for n, t in srcs.items()}
        for n, t in srcs.items():
            self.h[n].copy_(t)
        self.d_pack.copy_(self.h_pack)
        self.k_cache = bf(w.k_cache).to(dev)
        self.v_cache = bf(w.v_cache).to(dev)
        if self.fp8:
            # the cached context as E4M3 codes (torch's own conversion: set-up only)
            def codes(c, scale):
                x = (c.float() / scale).clamp(-448.0, 448.0)
                return x.to(torch.float8_e4m3fn).view(torch.uint8)
            self.k_cache = codes(self.k_cache, self.fp8[0])
            self.v_cache = codes(self.v_cache, self.fp8[1])
        self.out = torch.empty_like(self.d["q"])
        self.h_out = torch.empty(self.out.shape, dtype=torch.bfloat16).pin_memory()
        wsize = binding.cascade_workspace_size if cascade_len else binding.workspace_size
        self.ws = torch.empty(wsize(w.num_reqs, w.num_tokens, w.num_q_heads, w.num_kv_heads,
                                    w.head_dim), dtype=torch.uint8, device=dev)
        self.h2d_bytes = self.h_pack.numel()  # copied per step (inputs plus alignment padding)
        self.d2h_bytes = self.out.numel() * self.out.element_size()

    def step(self, out=None):
        """One step (KV write, then attention) into `out` (the device output
        unless given)."""
        d, w, b = self.d, self.w, self.binding
        out = self.out if out is None else out
        if self.fp8:
            ks, vs = self.fp8
            b.write_kv_fp8(d["k"], d["v"], d["slot_mapping"], self.k_cache, self.v_cache, ks, vs)
            b.attention_fp8(d["q"], self.k_cache, self.v_cache, d["block_tables"], d["seq_lens"],
                            d["qsl"], w.scale, ks, vs, max_query_len=w.max_query_len,
                            max_seq_len=w.max_seq_len, out=out, workspace=self.ws)
            return
        b.write_kv(d["k"], d["v"], d["slot_mapping"], self.k_cache, self.v_cache)
        if self.cascade_len:
            b.attention_cascade(d["q"], self.k_cache, self.v_cache, d["block_tables"],
                                d["seq_lens"], d["qsl"], w.scale,
                                common_prefix_len=self.cascade_len,
                                max_query_len=w.max_query_len, max_seq_len=w.max_seq_len,
                                out=out, workspace=self.ws)
        else:
            b.attention(d["q"], self.k_cache, self.v_cache, d["block_tables"], d["seq_lens"],
                        d["qsl"], w.scale, max_query_len=w.max_query_len,
                        max_seq_len=w.max_seq_len, out=out, workspace=self.ws)

    def step_e2e(self):
        # all of the step's inputs in one copy; the attention kernels store
        # the result straight into pinned host memory (pa_mapped_pointer), so
        # the device-to-host transfer overlaps the computation
        self.d_pack.copy_(self.h_pack, non_blocking=True)
        self.step(out=self.h_out)


def workload_signature(w: wl.Workload) -> str:
    """The step's profile name, execute_context_A(a)_generation_B(b). A
    synthetic batch has no prompts, so a request with more than one query
    token counts as a prefill chunk (context) and a one-token query as a
    decode (generation)."""
    from paged_kv_cache_42_gb300 import host

    ql = np.diff(np.asarray(w.query_start_loc, dtype=np.int64))
    ctx = ql > 1
    return host.step_signature({
        "num_context_reqs": int(ctx.sum()), "num_context_tokens": int(ql[ctx].sum()),
        "num_generation_reqs": int((~ctx).sum()), "num_generation_tokens": int(ql[~ctx].sum())})


def time_steps(res: Resident, steps: int, warmup: int, flush, torch, binding, dist,
               e2e: bool = False, clocks: ClockSampler | None = None, timers: bool = False):
    """Time `steps` steps (CUDA events on the launching stream, L2 flushed
    before each). With timers, the library also records events around its
    decode and tensor-core launches (kernel durations for the roofline); those
    events serialise the chained launches, so the step time is taken from a
    pass without them."""
    fn = res.step_e2e if e2e else res.step
    for _ in range(warmup):
        flush()
        fn()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    dk = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    pk = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    # the tensor-core kernel of the step: the cascade prefix pass, or prefill chunks
    pre_kernel = "prefix" if res.cascade_len else "prefill"
    has_prefill = bool(res.cascade_len) or res.w.max_query_len >= 16
    for a, b in dk + pk:  # materialise the event handles before handing them to the library
        a.record()
        b.record()
    torch.cuda.synchronize()
    barrier(dist)
    torch.cuda.synchronize()
    if clocks:
        clocks.start()
        time.sleep(0.3)
    n0 = binding.launch_count()
    stream = torch.cuda.current_stream()
    nvtx = torch.cuda.nvtx
    for i in range(steps):
        flush()
        if timers:
            binding.set_kernel_timer("decode", dk[i][0], dk[i][1])
            if has_prefill:
                binding.set_kernel_timer(pre_kernel, pk[i][0], pk[i][1])
        ev[i][0].record(stream)
        nvtx.range_push(res.signature)
        fn()
        nvtx.range_pop()
        ev[i][1].record(stream)
    binding.set_kernel_timer("decode", None, None)
    binding.set_kernel_timer(pre_kernel, None, None)
    launches = binding.launch_count() - n0
    torch.cuda.synchronize()
    clk = clocks.stop() if clocks else None
    barrier(dist)
    step_ms = [a.elapsed_time(b) for a, b in ev]
    dec_ms = [a.elapsed_time(b) for a, b in dk] if timers else [0.0]
    pre_ms = [a.elapsed_time(b) for a, b in pk] if (timers and has_prefill) else [0.0]
    return {"ms_per_step": sum(step_ms) / steps, "ms_median": statistics.median(step_ms),
            "decode_ms": sum(dec_ms) / len(dec_ms), "prefill_ms": sum(pre_ms) / len(pre_ms),
            "launches": launches, "clocks": clk}


def time_kernels(res: Resident, steps: int, warmup: int, flush, torch, binding, dist) -> dict:
    """Kernel durations (decode / tensor-core) from a separate timed pass.
    The events around each launch serialise the grids, so a mixed batch and a
    cascade are timed here with their overlaps off: every kernel on the whole
    GPU, one after the other."""
    binding.set_option("mixed_overlap", 0)
    binding.set_option("cascade_overlap", 0)
    try:
        t = time_steps(res, steps, warmup, flush, torch, binding, dist, timers=True)
    finally:
        binding.set_option("mixed_overlap", 1)
        binding.set_option("cascade_overlap", 1)
    return {"decode_ms": max_over_ranks(t["decode_ms"], dist),
            "prefill_ms": max_over_ranks(t["prefill_ms"], dist)}


def prefix_share_timing(args, flush, torch, binding, dist, rank, world) -> dict:
    """The prefix-sharing batch (every request shares one cached prefix),
    stepped through pa_attention and through pa_attention_cascade."""
    w = wl.make_config(PREFIX_CONFIG, seed=42 + PREFIX_CONFIG + 1000 * rank)
    sb = step_bytes(w)
    unique_attn = sb["attention"] - sb["kv"] + sb["kv_unique"]
    steps = max(50, args.steps // 10)
    out = {"workload": f"{wl.CONFIG_NAMES[PREFIX_CONFIG]}: "
                       f"{wl.CONFIG_DESCRIPTIONS[PREFIX_CONFIG]}",
           "steps": steps, "kv_bytes_logical": sb["kv"], "kv_bytes_unique": sb["kv_unique"]}
    for name, casc in (("plain", 0), ("cascade", w.shared_prefix_blocks * 16)):
        res = Resident(w, torch, binding, cascade_len=casc)
        t = time_steps(res, steps, args.warmup, flush, torch, binding, dist)
        tk = time_kernels(res, steps, args.warmup, flush, torch, binding, dist)
        if casc:  # the same step with the prefix pass first, on every SM
            binding.set_option("cascade_overlap", 0)
            try:
                ts = time_steps(res, steps, args.warmup, flush, torch, binding, dist)
            finally:
                binding.set_option("cascade_overlap", 1)
        code, detail = binding.get_device_error(clear=True)
        if code:
            raise RuntimeError(f"device error {code} at {detail}")
        ms = max_over_ranks(t["ms_per_step"], dist)
        dec = tk["decode_ms"]
        pre = tk["prefill_ms"] if casc else 0.0
        attn_ms = dec + pre
        out[name] = {"ms_per_step": round(ms, 5), "decode_kernel_ms": round(dec, 5),
                     "tokens_per_s": round(world * w.num_tokens / (ms * 1e-3), 1),
                     "attention_logical_gbs": round(sb["attention"] / (attn_ms * 1e-3) / 1e9, 1),
                     "attention_unique_gbs": round(unique_attn / (attn_ms * 1e-3) / 1e9, 1)}
        if casc:
            out[name]["prefix_kernel_ms"] = round(pre, 5)
            out[name]["common_prefix_len"] = casc
            out[name]["serial_ms_per_step"] = round(max_over_ranks(ts["ms_per_step"], dist), 5)
            out[name]["overlap"] = ("prefix pass on a few SMs beside the suffix pass; "
                                    "serial_ms_per_step: the prefix pass first; kernel times "
                                    "from a pass with the overlap off")
        del res
        torch.cuda.empty_cache()
    out["cascade_speedup"] = round(out["plain"]["ms_per_step"] / out["cascade"]["ms_per_step"], 3)
    return out


def fp8_timing(args, flush, torch, binding, dist, rank, world, peaks) -> dict:
    """The headline decode batch with an E4M3 KV cache (per-tensor scales)."""
    w = wl.make_config(HEADLINE_CONFIG, seed=42 + HEADLINE_CONFIG + 1000 * rank)
    sb = step_bytes(w, fp8=True)
    kv8, attn8 = sb["kv"], sb["attention"]
    steps = max(50, args.steps // 10)
    res = Resident(w, torch, binding, fp8_scales=FP8_SCALES)
    t = time_steps(res, steps, args.warmup, flush, torch, binding, dist)
    tk = time_kernels(res, steps, args.warmup, flush, torch, binding, dist)
    code, detail = binding.get_device_error(clear=True)
    if code:
        raise RuntimeError(f"device error {code} at {detail}")
    ms = max_over_ranks(t["ms_per_step"], dist)
    dec = tk["decode_ms"]
    del res
    torch.cuda.empty_cache()
    achieved = attn8 / (dec * 1e-3) / 1e9
    return {"workload": f"{wl.CONFIG_NAMES[HEADLINE_CONFIG]} with an E4M3 KV cache "
                        "(k_scale 0.0113, v_scale 0.0127)",
            "steps": steps, "ms_per_step": round(ms, 5), "decode_kernel_ms": round(dec, 5),
            "kv_bytes": kv8, "algorithmic_bytes_per_launch": attn8,
            "achieved_gbs": round(achieved, 1), "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": ncu_traffic(wl.CONFIG_NAMES[HEADLINE_CONFIG] + "-e4m3",
                                   split_kv_kernel(w, fp8=True, cascade=False)[1]),
            "peak_source": peaks["source"],
            "requests_per_s": round(world * w.num_reqs / (ms * 1e-3), 1)}


def long_context_timing(args, flush, torch, binding, dist, rank, world, peaks) -> dict:
    """The long-context decode batch (8 x 32768 tokens, 64 query / 8 KV heads):
    the split-KV showcase, on the kernel the library routes it to."""
    w = wl.make_config(LONG_CONFIG, seed=42 + LONG_CONFIG + 1000 * rank)
    sb = step_bytes(w)
    steps = max(50, args.steps // 10)
    res = Resident(w, torch, binding)
    t = time_steps(res, steps, args.warmup, flush, torch, binding, dist)
    tk = time_kernels(res, steps, args.warmup, flush, torch, binding, dist)
    code, detail = binding.get_device_error(clear=True)
    if code:
        raise RuntimeError(f"device error {code} at {detail}")
    ms = max_over_ranks(t["ms_per_step"], dist)
    dec = tk["decode_ms"]
    del res
    torch.cuda.empty_cache()
    kname, ksrc = split_kv_kernel(w, force=args.split_kv)
    achieved = sb["attention"] / (dec * 1e-3) / 1e9
    return {"workload": f"{wl.CONFIG_NAMES[LONG_CONFIG]}: {wl.CONFIG_DESCRIPTIONS[LONG_CONFIG]}",
            "steps": steps, "ms_per_step": round(ms, 5), "kernel": kname,
            "decode_kernel_ms": round(dec, 5), "algorithmic_bytes_per_launch": sb["attention"],
            "achieved_gbs": round(achieved, 1), "peak": peaks["hbm_gbs"],
            "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
            "traffic": ncu_traffic(wl.CONFIG_NAMES[LONG_CONFIG], ksrc),
            "step_gbs": round(world * sb["step"] / (ms * 1e-3) / 1e9, 1)}


def graph_steps(res: Resident, steps: int, warmup: int, flush, torch, dist) -> float:
    """ms per step when the step's calls (write + attention) are captured once
    in a CUDA graph and replayed; the L2 flush stays outside the timed region."""
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        res.step()
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        res.step()
    for _ in range(warmup):
        flush()
        g.replay()
    torch.cuda.synchronize()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
          for _ in range(steps)]
    barrier(dist)
    stream = torch.cuda.current_stream()
    for i in range(steps):
        flush()
        ev[i][0].record(stream)
        g.replay()
        ev[i][1].record(stream)
    torch.cuda.synchronize()
    barrier(dist)
    del g
    return max_over_ranks(sum(a.elapsed_time(b) for a, b in ev) / steps, dist)


def run_ours(args, rank, world, local, dist):
    import torch

    from paged_kv_cache_42_gb300 import binding
    from paged_kv_cache_42_gb300 import build as libbuild

    libbuild.build()
    torch.cuda.set_device(local)
    binding.init()
    binding.get_device_error(clear=True)
    binding.set_option("decode_tc", {"auto": 1, "cuda-core": 0, "tensor-core": 2}[args.split_kv])
    if args.tm_ctas_per_sm:
        binding.set_option("decode_tm_ctas_per_sm", args.tm_ctas_per_sm)
    if args.mixed_prefill_ctas:
        binding.set_option("mixed_prefill_ctas", args.mixed_prefill_ctas)
    props = torch.cuda.get_device_properties(local)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20) or (128 << 20))
    flush_buf = torch.empty(2 * l2, dtype=torch.uint8, device="cuda")
    clean_buf = torch.ones(2 * l2 // 4, dtype=torch.float32, device="cuda")

    def flush():
        # Write a buffer of twice the L2 size (evicts everything), then read
        # another of the same size so the L2 is left holding clean lines:
        # the timed step starts cold and pays no write-back of the flush.
        flush_buf.fill_(1)
        clean_buf.sum()

    peaks = measured_peaks()
    result = {}
    for idx in [args.config] + ([MIXED_CONFIG] if args.config != MIXED_CONFIG and not args.quick
                                else []):
        w = wl.make_config(idx, seed=42 + idx + 1000 * rank)
        casc = w.shared_prefix_blocks * 16 if (args.cascade and idx == args.config) else 0
        f8 = FP8_SCALES if (args.fp8 and idx == args.config) else None
        res = Resident(w, torch, binding, cascade_len=casc, fp8_scales=f8)
        sb = step_bytes(w, fp8=f8 is not None)
        steps = args.steps if idx == args.config else max(50, args.steps // 10)
        t = time_steps(res, steps, args.warmup, flush, torch, binding, dist,
                       clocks=ClockSampler(local) if idx == args.config else None)
        tk = time_kernels(res, steps, args.warmup, flush, torch, binding, dist)
        code, detail = binding.get_device_error(clear=True)
        if code:
            raise RuntimeError(f"device error {code} at {detail}")
        ms = max_over_ranks(t["ms_per_step"], dist)
        dec_ms = tk["decode_ms"]
        pre_ms = tk["prefill_ms"]
        entry = {"w": w, "sb": sb, "t": t, "ms": ms, "dec_ms": dec_ms, "pre_ms": pre_ms,
                 "res": res, "steps": steps, "signature": res.signature}
        entry["graph_ms"] = graph_steps(res, steps, args.warmup, flush, torch, dist)
        if idx == MIXED_CONFIG:  # the same step with the chunks and split-KV work in turn
            binding.set_option("mixed_overlap", 0)
            try:
                ts = time_steps(res, steps, args.warmup, flush, torch, binding, dist)
            finally:
                binding.set_option("mixed_overlap", 1)
            entry["serial_ms"] = max_over_ranks(ts["ms_per_step"], dist)
        if idx == args.config and not args.no_e2e:
            te = time_steps(res, max(20, steps // 4), args.warmup, flush, torch, binding, dist,
                            e2e=True)
            entry["e2e_ms"] = max_over_ranks(te["ms_per_step"], dist)
        result[idx] = entry
        if idx != args.config:
            del res
            entry["res"] = None
            torch.cuda.empty_cache()

    main = result[args.config]
    w, sb = main["w"], main["sb"]
    ms = main["ms"]
    kname, ksrc = split_kv_kernel(w, fp8=bool(args.fp8), cascade=bool(args.cascade),
                                  force=args.split_kv)
    value = world * sb["step"] / (ms * 1e-3) / 1e9
    achieved = sb["attention"] / (main["dec_ms"] * 1e-3) / 1e9
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": main["steps"],
        "warmup": args.warmup,
        "ms_per_step": round(ms, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "e4m3" if args.fp8 else "bf16",
        "data": "synthetic (seeded numpy PCG64, N(0,1) rounded to bf16)",
        "config": {"workload": f"{wl.CONFIG_NAMES[args.config]}: "
                               f"{wl.CONFIG_DESCRIPTIONS[args.config]}" +
                               (f" over an E4M3 KV cache (k_scale {FP8_SCALES[0]}, "
                                f"v_scale {FP8_SCALES[1]})" if args.fp8 else ""),
                   "num_reqs": w.num_reqs, "num_tokens": w.num_tokens,
                   "split_kv": args.split_kv,
                   "step_signature": main["signature"],
                   "l2": "flushed before every timed step (2x L2 written, then 2x L2 read)",
                   "parallelism": f"replicas x{world}"},
        "roofline": {
            "bound": "hbm", "kernel": kname,
            "achieved": round(achieved, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4), "peak_source": peaks["source"],
            "traffic": ncu_traffic(wl.CONFIG_NAMES[args.config] + ("-e4m3" if args.fp8 else ""), ksrc),
            "algorithmic_bytes_per_launch": sb["attention"],
            "kernel_ms": round(main["dec_ms"], 5)},
        "gpu_launches": int(main["t"]["launches"]),
        "cuda_graph": {"ms_per_step": round(main["graph_ms"], 5),
                       "value": round(world * sb["step"] / (main["graph_ms"] * 1e-3) / 1e9, 2),
                       "unit": "GB/s",
                       "what": "the same step's calls captured once in a CUDA graph and replayed"},
        "prefill_kernel_ms": round(main["pre_ms"], 5) if main["pre_ms"] > 0 else None,
        "clocks": main["t"]["clocks"],
    }
    if w.shared_prefix_blocks:
        line["roofline"]["achieved_unique"] = round(
            (sb["attention"] - sb["kv"] + sb["kv_unique"]) / (main["dec_ms"] * 1e-3) / 1e9, 1)
    if "e2e_ms" in main:
        res = main["res"]
        line["e2e"] = {"value": round(world * sb["step"] / (main["e2e_ms"] * 1e-3) / 1e9, 2),
                       "unit": "GB/s", "ms_per_step": round(main["e2e_ms"], 5),
                       "h2d_bytes_per_step": res.h2d_bytes, "d2h_bytes_per_step": res.d2h_bytes,
                       "path": "inputs: one copy from a pinned pack; output: stored by the "
                               "kernels into pinned host memory (pa_mapped_pointer)"}
    if MIXED_CONFIG in result and MIXED_CONFIG != args.config:
        m = result[MIXED_CONFIG]
        mw = m["w"]
        line["mixed_batch"] = {
            "workload": f"{wl.CONFIG_NAMES[MIXED_CONFIG]}: {wl.CONFIG_DESCRIPTIONS[MIXED_CONFIG]}",
            "value": round(world * mw.num_tokens / (m["ms"] * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": round(m["ms"], 5), "steps": m["steps"],
            "step_signature": m["signature"],
            "serial_ms_per_step": round(m["serial_ms"], 5),
            "overlap": "prefill chunks on a few SMs beside the split-KV work (the planner's "
                       "split); serial_ms_per_step: the two in turn on every SM",
            "cuda_graph_ms_per_step": round(m["graph_ms"], 5),
            "cuda_graph_value": round(world * mw.num_tokens / (m["graph_ms"] * 1e-3), 1),
            "attention_kernel_ms": round(m["dec_ms"], 5),
            "prefill_kernel_ms": round(m["pre_ms"], 5),
            "kernel_ms_note": "kernels timed one after the other on every SM (overlap off)",
            "prefill_tflops": round(prefill_flops(mw) / (m["pre_ms"] * 1e-3) / 1e12, 1)
            if m["pre_ms"] > 0 else None,
            "kv_bytes": m["sb"]["kv"], "prefill_causal_flops": prefill_flops(mw)}
    if not args.quick and args.config != PREFIX_CONFIG:
        line["prefix_share"] = prefix_share_timing(args, flush, torch, binding, dist, rank, world)
    if not args.quick and args.config != LONG_CONFIG:
        line["long_context"] = long_context_timing(args, flush, torch, binding, dist, rank, world,
                                                   peaks)
    if not args.quick:
        line["kv_fp8"] = fp8_timing(args, flush, torch, binding, dist, rank, world, peaks)
    line["pages_context"] = PAGES_CONTEXT
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w, args.cpu_seconds)
    if rank == 0 and not args.quick:
        line["host_scheduler"] = host_scheduler_timing()
        line["host_scheduler"]["xxh64"] = host_scheduler_timing(hash_algo="xxh64", brief=True)
    return line


def host_scheduler_timing(steps: int = 200, hash_algo: str = "sha256", brief: bool = False) -> dict:
    """Time the library's host scheduler step (pa_sched_step) forming the
    mixed-batch shape: 512 decoding requests with the mixed workload's
    context lengths plus 3 long prompts prefilled in 512-token chunks under
    a 2048-token budget, prefix caching on (block hash: hash_algo). Only the
    C call is timed."""
    from paged_kv_cache_42_gb300 import host

    ctx, _, _ = wl.config_lengths(MIXED_CONFIG)
    rng = np.random.Generator(np.random.PCG64(7))
    pool = host.BlockPool(num_blocks=90000, block_size=16, hash_algo=hash_algo)
    s = host.Scheduler(pool, token_budget=2048, max_model_len=4096, long_prefill_threshold=512,
                       max_reqs=1024, retained_block_tables=True)
    for i, c in enumerate(ctx[:512]):
        s.add_request(i, rng.integers(0, 32000, int(c)))

    def after(out):
        nonlocal next_id
        for rid in out["req_ids"]:
            st = s.request_state(int(rid))
            if st["num_computed"] == st["num_tokens"]:
                if rid >= 512:
                    s.finish(int(rid))
                    s.add_request(next_id, rng.integers(0, 32000, 3500))
                    next_id += 1
                else:
                    s.append_token(int(rid), int(rng.integers(0, 32000)))

    next_id = 512
    while True:  # bring all 512 requests to decoding
        out = s.step()
        after(out)
        if s.num_waiting() == 0 and out["num_tokens"] == 512:
            break
    for _ in range(3):
        s.add_request(next_id, rng.integers(0, 32000, 3500))
        next_id += 1
    times, shapes = [], set()
    for _ in range(steps):
        out = s.step()
        times.append(s.last_step_seconds)
        shapes.add((len(out["req_ids"]), out["num_tokens"]))
        after(out)
    t = np.asarray(times) * 1e6
    if brief:
        return {"us_per_step_median": round(float(np.median(t)), 1),
                "us_per_step_p90": round(float(np.percentile(t, 90)), 1),
                "what": "the same, with XXH64 block hashes (PA_HASH_XXH64)"}
    return {"us_per_step_median": round(float(np.median(t)), 1),
            "us_per_step_p90": round(float(np.percentile(t, 90)), 1), "steps": steps,
            "batch": "512 decodes + 3 prefill chunks of 512, 2048 tokens",
            "batch_shapes_seen": sorted(shapes)[:4],
            "what": "pa_sched_step on one host core: budget pass, block allocation, prefix-cache "
                    "registration (SHA-256), metadata arrays for the kernels (block tables "
                    "retained between steps)"}


# ---------------------------------------------------------------------------
# CPU oracle arms
# ---------------------------------------------------------------------------
def _oracle_sample(w: wl.Workload, reqs, threads):
    import oracle
    kc, vc = w.k_cache, w.v_cache
    oracle.write_kv(w.k_new, w.v_new, w.slot_mapping, kc, vc)
    oracle.attention(w.q, kc, vc, w.block_tables, w.seq_lens, w.query_start_loc, w.scale,
                     reqs=reqs, threads=threads)


def _sample_bytes(w: wl.Workload, reqs) -> int:
    sub = wl.subset_requests(w, reqs)
    return step_bytes(sub)["step"]


def cpu_baseline(w: wl.Workload, seconds: float) -> dict:
    """The oracle as it stands on the host cores, on whole requests of the
    workload taken in order until `seconds` of work is done."""
    threads = os.cpu_count() or 1
    done_bytes, t0, r, reqs_done = 0, time.perf_counter(), 0, 0
    while time.perf_counter() - t0 < seconds and reqs_done < 100000:
        batch = [(r + i) % w.num_reqs for i in range(min(8, w.num_reqs))]
        _oracle_sample(w, batch, threads)
        done_bytes += _sample_bytes(w, batch)
        r = (r + len(batch)) % w.num_reqs
        reqs_done += len(batch)
    el = time.perf_counter() - t0
    return {"value": round(done_bytes / el / 1e9, 4), "unit": "GB/s", "cores": threads,
            "kind": "oracle",
            "sample": f"{reqs_done} requests of {w.name} (8 at a time, in order) in {el:.1f} s, "
                      f"write + attention, float64"}


def run_reference(args, rank, world):
    if rank != 0:
        return None
    w = wl.make_config(args.config)
    threads = os.cpu_count() or 1
    times, sizes = [], []
    for i in range(args.warmup + args.steps):
        req = [i % w.num_reqs]
        t0 = time.perf_counter()
        _oracle_sample(w, req, threads)
        dt = time.perf_counter() - t0
        if i >= args.warmup:
            times.append(dt)
            sizes.append(_sample_bytes(w, req))
    tot = sum(times)
    value = sum(sizes) / tot / 1e9
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 5), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(1e3 * tot / len(times), 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": f"{wl.CONFIG_NAMES[args.config]}: "
                               f"{wl.CONFIG_DESCRIPTIONS[args.config]}",
                   "sample": "one request of the batch per step (write + attention)"},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": threads,
                         "kind": "oracle",
                         "sample": "one request of the workload per step, in order"},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--config", type=int, default=HEADLINE_CONFIG, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--quick", action="store_true", help="headline workload only")
    ap.add_argument("--fp8", action="store_true",
                    help="step the chosen workload with an E4M3 KV cache")
    ap.add_argument("--cascade", action="store_true",
                    help="step the chosen workload through pa_attention_cascade (its shared "
                         "prefix as the common prefix; the prefix-sharing workload has one)")
    ap.add_argument("--split-kv", choices=["auto", "cuda-core", "tensor-core"], default="auto",
                    help="split-KV kernel: the library's routing (default), or one forced "
                         "(pa_set_option PA_OPT_DECODE_TC 0 / 2)")
    ap.add_argument("--tm-ctas-per-sm", type=int, choices=[1, 2], default=None,
                    help="CTAs per SM of the token-major E4M3 split-KV kernel "
                         "(pa_set_option PA_OPT_DECODE_TM_CTAS_PER_SM; default: the library's)")
    ap.add_argument("--mixed-prefill-ctas", type=int, default=0,
                    help="SMs the prefill chunks take beside the split-KV work in a mixed "
                         "batch (pa_set_option PA_OPT_MIXED_PREFILL_CTAS; 0: the planner's)")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    rank, world, local, dist = dist_setup()
    if args.impl == "reference":
        line = run_reference(args, rank, world)
    else:
        line = run_ours(args, rank, world, local, dist)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if dist is not None:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
