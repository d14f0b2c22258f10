// C ABI of libpagedattn: argument validation, per-device set-up, the device
// error word, optional launch timers and dispatch to the kernels.
//
// Validation happens before any CUDA call, so a malformed call is rejected
// without touching (or needing) a GPU.
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <nvtx3/nvToolsExt.h>

#include <atomic>
#include <mutex>

#include "pa_api.h"
#include "pa_internal.h"

namespace pa {

// The device error word: [0] code (PA_DEVERR_*), [1] detail. One per device,
// in static device memory; kernels receive its address as an argument.
__device__ unsigned long long g_device_error[2];

namespace {

constexpr int kMaxDevices = 64;

// Per-device set-up, done once. The cached device address of the error word
// stays valid for the life of the CUDA context: the library does not support
// cudaDeviceReset of a device it has been used on.
struct DeviceState {
  std::atomic<bool> ready{false};
  int num_sms = 0;
  unsigned long long* err = nullptr;
};

std::mutex g_mutex;
DeviceState g_devices[kMaxDevices];
std::atomic<long long> g_launches{0};
std::atomic<int> g_self_plan{1};  // pa_set_option(PA_OPT_DECODE_SELF_PLAN, ...)
std::atomic<int> g_decode_tc{1};  // pa_set_option(PA_OPT_DECODE_TC, ...): 0 off, 1 auto, 2 on
std::atomic<int> g_max_workers{0};  // pa_set_option(PA_OPT_DECODE_MAX_WORKERS, ...): 0 = no cap
std::atomic<int> g_mixed_overlap{1};  // pa_set_option(PA_OPT_MIXED_OVERLAP, ...)
std::atomic<int> g_token_major{1};  // pa_set_option(PA_OPT_DECODE_TOKEN_MAJOR, ...)
std::atomic<int> g_cascade_overlap{1};  // pa_set_option(PA_OPT_CASCADE_OVERLAP, ...)
std::atomic<int> g_tm_ctas{2};  // pa_set_option(PA_OPT_DECODE_TM_CTAS_PER_SM, ...)
std::atomic<int> g_mixed_ctas{0};  // pa_set_option(PA_OPT_MIXED_PREFILL_CTAS, ...): 0 = planned
constexpr int kNumTimers = 6;  // write, plan, decode, prefill, cascade prefix, merge
cudaEvent_t g_timer_start[kNumTimers] = {};
cudaEvent_t g_timer_stop[kNumTimers] = {};

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

pa_status device_state(DeviceState** out) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  DeviceState& d = g_devices[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(g_mutex);
    if (!d.ready.load(std::memory_order_relaxed)) {
      int sms = 0;
      if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return PA_ERR_CUDA;
      void* err = nullptr;
      if (cudaGetSymbolAddress(&err, g_device_error) != cudaSuccess) return PA_ERR_CUDA;
      d.num_sms = sms;
      d.err = static_cast<unsigned long long*>(err);
      d.ready.store(true, std::memory_order_release);
    }
  }
  *out = &d;
  return PA_OK;
}

// An NVTX range around a call's launches (header-only NVTX: nothing happens
// unless a profiler is attached), named after the entry point.
struct NvtxRange {
  explicit NvtxRange(const char* name) { nvtxRangePushA(name); }
  ~NvtxRange() { nvtxRangePop(); }
};

struct TimerScope {
  int id;
  cudaStream_t s;
  TimerScope(int kernel, cudaStream_t stream) : id(kernel), s(stream) {
    if (g_timer_start[id]) cudaEventRecord(g_timer_start[id], s);
  }
  ~TimerScope() {
    if (g_timer_stop[id]) cudaEventRecord(g_timer_stop[id], s);
  }
};

bool supported_group(int g) { return g == 1 || g == 2 || g == 4 || g == 8; }

}  // namespace

pa_status check_attention_args(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               const int32_t* query_start_loc, float scale, const void* out,
                               int num_reqs, int num_tokens, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks,
                               int max_blocks_per_req, int max_query_len, int max_seq_len,
                               int prefix_len, int kv_fp8, float k_scale, float v_scale,
                               bool* nothing_to_do) {
  *nothing_to_do = false;
  if (kv_fp8 && !(k_scale > 0.f && k_scale < INFINITY && v_scale > 0.f && v_scale < INFINITY))
    return PA_ERR_INVALID_ARG;
  if (kv_fp8 && prefix_len > 0) return PA_ERR_UNSUPPORTED;  // no FP8 cascade
  if (num_reqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || num_blocks < 0 || max_blocks_per_req < 0 || max_query_len < 0 ||
      max_seq_len < 0)
    return PA_ERR_INVALID_ARG;
  if (num_q_heads % num_kv_heads != 0) return PA_ERR_INVALID_ARG;
  if (block_size != kBlockSize || (head_dim != 64 && head_dim != 128) ||
      !supported_group(num_q_heads / num_kv_heads))
    return PA_ERR_UNSUPPORTED;
  if (!(scale == scale)) return PA_ERR_INVALID_ARG;  // NaN scale
  if (num_reqs == 0 || num_tokens == 0) {
    *nothing_to_do = true;
    return PA_OK;
  }
  if (!q || !k_cache || !v_cache || !block_tables || !seq_lens || !query_start_loc || !out)
    return PA_ERR_INVALID_ARG;
  if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
      (reinterpret_cast<uintptr_t>(block_tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(seq_lens) & 3u) ||
      (reinterpret_cast<uintptr_t>(query_start_loc) & 3u))
    return PA_ERR_INVALID_ARG;
  // flattened work positions must fit a 32-bit int: tokens x Hkv x blocks per token
  const long long max_blocks = ((long long)max_seq_len + kBlockSize - 1) / kBlockSize;
  if ((long long)num_tokens * num_kv_heads * max_blocks >= (1LL << 31))
    return PA_ERR_UNSUPPORTED;
  // a cascade prefix is whole blocks, inside the tables, and leaves every
  // request at least one key of its own
  if (prefix_len > 0 && (prefix_len / kBlockSize > max_blocks_per_req || prefix_len >= max_seq_len))
    return PA_ERR_INVALID_ARG;
  return PA_OK;
}

}  // namespace pa

using namespace pa;

extern "C" {

int pa_version(void) { return 100; }

long long pa_launch_count(void) { return g_launches.load(); }

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID_ARG: return "PA_ERR_INVALID_ARG: invalid argument";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED: unsupported block_size / head_dim / group";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE: workspace missing or too small";
    case PA_ERR_CUDA: return "PA_ERR_CUDA: CUDA runtime or launch failure";
    case PA_ERR_BOUNDS: return "PA_ERR_BOUNDS: index outside its valid range";
    case PA_ERR_TIMEOUT: return "PA_ERR_TIMEOUT: a bounded device wait gave up";
    default: return "unknown pa_status";
  }
}

pa_status pa_init(void) {
  DeviceState* d = nullptr;
  return device_state(&d);
}

}  // extern "C"

namespace {

pa_status write_kv_impl(const void* k, const void* v, const int64_t* slot_mapping, void* k_cache,
                        void* v_cache, int kv_fp8, float k_scale, float v_scale, int num_tokens,
                        int num_kv_heads, int head_dim, int block_size, int num_blocks,
                        void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0)
    return PA_ERR_INVALID_ARG;
  if (kv_fp8 && !(k_scale > 0.f && k_scale < INFINITY && v_scale > 0.f && v_scale < INFINITY))
    return PA_ERR_INVALID_ARG;
  if (block_size != kBlockSize || head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  const NvtxRange range(kv_fp8 ? "pa_write_kv_fp8" : "pa_write_kv");
  if (num_tokens == 0) return PA_OK;
  if (!k || !v || !slot_mapping || !k_cache || !v_cache) return PA_ERR_INVALID_ARG;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) ||
      (reinterpret_cast<uintptr_t>(slot_mapping) & 7u))
    return PA_ERR_INVALID_ARG;
  DeviceState* d = nullptr;
  if (pa_status st = device_state(&d)) return st;
  WriteParams p;
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.slot_mapping = slot_mapping;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.kv_fp8 = kv_fp8;
  p.k_scale = k_scale;
  p.v_scale = v_scale;
  p.num_tokens = num_tokens;
  p.num_kv_heads = num_kv_heads;
  p.head_dim = head_dim;
  p.num_slots = (long long)num_blocks * kBlockSize;
  p.err = d->err;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  TimerScope timer(0, s);
  const cudaError_t e = launch_write_kv(p, s);
  g_launches.fetch_add(1);
  return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

pa_status pa_write_kv(const void* k, const void* v, const int64_t* slot_mapping, void* k_cache,
                      void* v_cache, int num_tokens, int num_kv_heads, int head_dim,
                      int block_size, int num_blocks, void* stream) {
  return write_kv_impl(k, v, slot_mapping, k_cache, v_cache, 0, 1.f, 1.f, num_tokens,
                       num_kv_heads, head_dim, block_size, num_blocks, stream);
}

pa_status pa_write_kv_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                          void* k_cache, void* v_cache, float k_scale, float v_scale,
                          int num_tokens, int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, void* stream) {
  return write_kv_impl(k, v, slot_mapping, k_cache, v_cache, 1, k_scale, v_scale, num_tokens,
                       num_kv_heads, head_dim, block_size, num_blocks, stream);
}

size_t pa_attention_workspace_size(int num_reqs, int num_tokens, int num_q_heads,
                                   int num_kv_heads, int head_dim) {
  if (num_reqs < 0 || num_tokens < 0 || num_q_heads <= 0 || num_kv_heads <= 0 ||
      head_dim <= 0 || num_q_heads % num_kv_heads != 0)
    return 0;
  return ws_layout(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim).total;
}

size_t pa_attention_cascade_workspace_size(int num_reqs, int num_tokens, int num_q_heads,
                                           int num_kv_heads, int head_dim) {
  const size_t base =
      pa_attention_workspace_size(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim);
  if (base == 0) return 0;
  return base + prefix_partials_bytes(num_tokens, num_q_heads, num_kv_heads, head_dim);
}

}  // extern "C"

namespace {

// pa_attention and pa_attention_cascade (prefix_len > 0).
pa_status attention_impl(const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, const int32_t* seq_lens,
                         const int32_t* query_start_loc, float scale, void* out, int num_reqs,
                         int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int num_blocks, int max_blocks_per_req,
                         int max_query_len, int max_seq_len, int prefix_len, int kv_fp8,
                         float k_scale, float v_scale, void* workspace,
                         size_t workspace_bytes, void* stream) {
  bool nothing = false;
  if (pa_status st = check_attention_args(
          q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out, num_reqs,
          num_tokens, num_q_heads, num_kv_heads, head_dim, block_size, num_blocks,
          max_blocks_per_req, max_query_len, max_seq_len, prefix_len, kv_fp8, k_scale, v_scale,
          &nothing))
    return st;
  if (nothing) return PA_OK;
  const WsLayout lay = ws_layout(num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim);
  const size_t need =
      lay.total + (prefix_len > 0
                       ? prefix_partials_bytes(num_tokens, num_q_heads, num_kv_heads, head_dim)
                       : 0);
  if (!workspace || workspace_bytes < need || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return PA_ERR_WORKSPACE;

  DeviceState* d = nullptr;
  if (pa_status st = device_state(&d)) return st;
  const NvtxRange range(prefix_len > 0 ? "pa_attention_cascade"
                                       : (kv_fp8 ? "pa_attention_fp8" : "pa_attention"));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  unsigned char* ws = static_cast<unsigned char*>(workspace);

  const int group = num_q_heads / num_kv_heads;
  // cascade: prefix key chunks, all non-empty (they divide the key tiles evenly)
  int chunks = 0;
  if (prefix_len > 0) {
    const int nkt = (prefix_len + 127) / 128;
    const int c = prefix_chunks(num_tokens, num_kv_heads, group, nkt);
    const int per = (nkt + c - 1) / c;
    chunks = (nkt + per - 1) / per;
  }
  float* const prefix_partials =
      prefix_len > 0 ? reinterpret_cast<float*>(ws + lay.total) : nullptr;

  PlanParams pp;
  pp.qsl = query_start_loc;
  pp.seq_lens = seq_lens;
  pp.block_tables = block_tables;
  pp.prefix_blocks = prefix_len / kBlockSize;
  // a decode-only batch (every span at most one token) plans itself inside
  // the split-KV kernel: no planner launch, and the kernel overlaps the KV write
  const int self_plan = (g_self_plan.load() && prefix_len == 0 && max_query_len <= 1 &&
                         num_reqs <= kSelfPlanMaxReqs) ? 1 : 0;
  pp.early_trigger = prefix_len > 0 ? 1 : 0;
  pp.num_reqs = num_reqs;
  pp.num_tokens = num_tokens;
  pp.num_kv_heads = num_kv_heads;
  pp.max_blocks_per_req = max_blocks_per_req;
  pp.max_query_len = max_query_len;
  pp.max_seq_len = max_seq_len;
  pp.group = group;
  // a cascade sends every span to the split-KV path
  pp.use_prefill = (prefix_len == 0 && max_query_len >= kPrefillMinQlen) ? 1 : 0;
  const int occ_cap =
      prefix_len > 0 ? PA_DEC_OCC_CAP_CASCADE : (kv_fp8 ? PA_DEC_OCC_CAP_FP8 : PA_DEC_OCC_CAP);
  // The tensor-core split-KV kernel takes the groups whose arithmetic per
  // cached byte outgrows the CUDA cores (by default G >= PA_DECODE_TC_MIN_GROUP),
  // except a cascade's suffix pass: its short suffixes leave each CTA a few
  // tiles per (token, kv head), and the CUDA-core kernel's many warps hide
  // the per-(token, kv head) epilogue better (measured 39 vs 76 us on the
  // prefix-sharing batch).
  const int tc_mode = g_decode_tc.load();
  const bool use_tc = tc_mode != 0 &&
                      decode_tc_supported(head_dim, group, kv_fp8 != 0, prefix_len / kBlockSize) &&
                      (tc_mode == 2 || (group >= PA_DECODE_TC_MIN_GROUP && prefix_len == 0));
  // A cascade on the CUDA-core suffix pass may run its prefix pass on a few
  // SMs (about two prefix items each) beside the suffix pass on the rest; the
  // merge pass then folds every (token, kv head).
  const int c_overlap = (g_cascade_overlap.load() && prefix_len > 0 && !use_tc) ? 1 : 0;
  int prefix_ctas = 0;
  if (c_overlap) {
    const int items = prefix_pairs(num_tokens, group) * num_kv_heads * chunks;
    prefix_ctas = (items + 1) / 2;
    if (prefix_ctas > d->num_sms / 4) prefix_ctas = d->num_sms / 4;
    if (prefix_ctas < 1) prefix_ctas = 1;
  }
  const int dec_sms = d->num_sms - prefix_ctas;  // SMs the split-KV grid fills
  // An E4M3 cache over eight KV heads takes the token-major tiles (one block
  // of every KV head per tile) on the tensor cores.
  const int tm_cps = g_tm_ctas.load();
  const bool use_tm =
      use_tc && kv_fp8 && g_token_major.load() &&
      decode_tm_supported(head_dim, group, num_kv_heads, decode_tm_workers(group, d->num_sms, tm_cps));
  const int launched = use_tm   ? decode_tm_workers(group, d->num_sms, tm_cps)
                       : use_tc ? decode_tc_workers(d->num_sms)
                                : decode_workers(head_dim, pp.group, kv_fp8 != 0, dec_sms, occ_cap);
  if (launched <= 0) return PA_ERR_CUDA;
  const int cap = g_max_workers.load();
  pp.num_workers = (cap > 0 && cap < launched) ? cap : launched;
  pp.token_major = use_tm ? 1 : 0;
  // A mixed batch on the tensor-core split-KV kernel (bf16) may run its
  // prefill chunks on a few SMs beside the split-KV work (the planner decides
  // how many, or none); the E4M3 path keeps its query-split pass between them.
  const int overlap = (g_mixed_overlap.load() && pp.use_prefill && use_tc && !kv_fp8) ? 1 : 0;
  pp.overlap = overlap;
  pp.prefill_ctas_override = g_mixed_ctas.load();
  pp.num_sms = d->num_sms;
  pp.position_bytes = 2 * kBlockSize * head_dim * 2;  // K and V of one 16-key block
  pp.header = reinterpret_cast<WsHeader*>(ws + lay.header_off);
  pp.units = reinterpret_cast<UnitInfo*>(ws + lay.units_off);
  pp.tiles = reinterpret_cast<PrefillTile*>(ws + lay.tiles_off);
  pp.raw = reinterpret_cast<int2*>(ws + lay.raw_off);
  pp.worker_unit = reinterpret_cast<int*>(ws + lay.workers_off);
  pp.err = d->err;
  if (!self_plan) {
    TimerScope timer(1, s);
    const cudaError_t e = launch_plan(pp, s);
    g_launches.fetch_add(1);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }

  if (pp.use_prefill || prefix_len > 0) {
    PrefillLaunch pl;
    pl.prefix_len = prefix_len;
    pl.prefix_chunks = chunks;
    pl.slot_floats = lay.slot_floats;
    pl.prefix_partials = prefix_partials;
    pl.kv_fp8 = kv_fp8;
    pl.v_scale = kv_fp8 ? v_scale : 1.f;
    pl.q = q;
    pl.k_cache = k_cache;
    pl.v_cache = v_cache;
    pl.qsl = query_start_loc;
    pl.seq_lens = seq_lens;
    pl.block_tables = block_tables;
    pl.out = static_cast<uint16_t*>(out);
    pl.header = pp.header;
    pl.tiles = pp.tiles;
    pl.num_tokens = num_tokens;
    pl.num_q_heads = num_q_heads;
    pl.num_kv_heads = num_kv_heads;
    pl.head_dim = head_dim;
    pl.num_blocks = num_blocks;
    pl.bt_stride = max_blocks_per_req;
    pl.scale_log2 = scale * 1.4426950408889634f * (kv_fp8 ? k_scale : 1.f);
    pl.overlap = prefix_len > 0 ? c_overlap : overlap;
    pl.prefix_ctas = prefix_ctas;
    pl.err = d->err;
    TimerScope timer(prefix_len > 0 ? 4 : 3, s);
    const cudaError_t e = launch_prefill(pl, d->num_sms, s);
    g_launches.fetch_add(1);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }

  DecodeParams dp;
  dp.q = static_cast<const uint16_t*>(q);
  dp.k_cache = k_cache;
  dp.v_cache = v_cache;
  dp.v_scale = kv_fp8 ? v_scale : 1.f;
  dp.block_tables = block_tables;
  dp.out = static_cast<uint16_t*>(out);
  dp.bt_stride = max_blocks_per_req;
  dp.num_q_heads = num_q_heads;
  dp.num_kv_heads = num_kv_heads;
  dp.num_blocks = num_blocks;
  // scores in base-2 units; an E4M3 cache's k_scale rides on q
  dp.scale_log2 = scale * 1.4426950408889634f * (kv_fp8 ? k_scale : 1.f);
  dp.header = pp.header;
  dp.units = pp.units;
  dp.worker_unit = num_tokens <= kPlanSmemTokens ? pp.worker_unit : nullptr;
  dp.partials = reinterpret_cast<float*>(ws + lay.partials_off);
  dp.slot_floats = lay.slot_floats;
  dp.key_start_blocks = prefix_len / kBlockSize;
  dp.prefix_partials = prefix_partials;
  dp.prefix_chunks = chunks;
  dp.num_tokens = num_tokens;
  dp.self_plan = self_plan;
  dp.num_reqs = num_reqs;
  dp.max_blocks_per_req = max_blocks_per_req;
  dp.max_query_len = max_query_len;
  dp.max_seq_len = max_seq_len;
  dp.qsl = query_start_loc;
  dp.seq_lens = seq_lens;
  dp.header_out = pp.header;
  dp.merge_tasks = reinterpret_cast<int4*>(ws + lay.tasks_off);
  dp.max_workers = cap > 0 ? cap : kMaxDecodeWorkers;
  dp.qsplit = ws + lay.qsplit_off;
  dp.qinv = reinterpret_cast<const float*>(ws + lay.qinv_off);
  dp.overlap = (overlap || c_overlap) ? 1 : 0;
  dp.fold_later = c_overlap;
  dp.err = d->err;
  if (use_tc && kv_fp8) {  // the E4M3 tensor-core kernel takes the queries split
    const cudaError_t e = launch_qsplit(dp, group, s);
    g_launches.fetch_add(1);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  int launched_workers = 0;
  {
    TimerScope timer(2, s);
    const cudaError_t e =
        use_tm   ? launch_decode_tm(dp, group, d->num_sms, tm_cps, s, &launched_workers)
        : use_tc ? launch_decode_tc(dp, group, kv_fp8 != 0, d->num_sms, s, &launched_workers)
                 : launch_decode(dp, head_dim, group, kv_fp8 != 0, dec_sms, occ_cap, s,
                                 &launched_workers);
    g_launches.fetch_add(1);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  // the slicing's worker count, as the split-KV kernel computes it
  const int workers = (cap > 0 && cap < launched_workers) ? cap : launched_workers;

  MergeParams mp;
  mp.header = pp.header;
  mp.tasks = dp.merge_tasks;
  mp.partials = dp.partials;
  mp.slot_floats = lay.slot_floats;
  mp.num_workers = workers;
  mp.workers_from_header = overlap;
  mp.token_major = pp.token_major;
  mp.num_q_heads = num_q_heads;
  mp.num_kv_heads = num_kv_heads;
  mp.num_tokens = num_tokens;
  mp.key_start_blocks = dp.key_start_blocks;
  mp.prefix_partials = prefix_partials;
  mp.prefix_chunks = chunks;
  mp.v_scale = dp.v_scale;
  mp.out = dp.out;
  mp.all_units = c_overlap;
  mp.units = pp.units;
  if (workers > 1 || c_overlap) {
    TimerScope timer(5, s);
    const cudaError_t e = launch_merge(mp, head_dim, group, s);
    g_launches.fetch_add(1);
    if (e != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // namespace

extern "C" {

pa_status pa_attention(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* seq_lens,
                       const int32_t* query_start_loc, float scale, void* out, int num_reqs,
                       int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, int max_blocks_per_req,
                       int max_query_len, int max_seq_len, void* workspace,
                       size_t workspace_bytes, void* stream) {
  return attention_impl(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out,
                        num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, max_blocks_per_req, max_query_len, max_seq_len, 0, 0, 1.f,
                        1.f, workspace, workspace_bytes, stream);
}

pa_status pa_attention_fp8(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* seq_lens,
                           const int32_t* query_start_loc, float scale, float k_scale,
                           float v_scale, void* out, int num_reqs, int num_tokens,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, int max_blocks_per_req, int max_query_len,
                           int max_seq_len, void* workspace, size_t workspace_bytes,
                           void* stream) {
  return attention_impl(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out,
                        num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, max_blocks_per_req, max_query_len, max_seq_len, 0, 1,
                        k_scale, v_scale, workspace, workspace_bytes, stream);
}

pa_status pa_attention_cascade(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               const int32_t* query_start_loc, float scale, void* out,
                               int num_reqs, int num_tokens, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks,
                               int max_blocks_per_req, int max_query_len, int max_seq_len,
                               int common_prefix_len, void* workspace, size_t workspace_bytes,
                               void* stream) {
  if (common_prefix_len <= 0 || common_prefix_len % kBlockSize != 0) return PA_ERR_INVALID_ARG;
  return attention_impl(q, k_cache, v_cache, block_tables, seq_lens, query_start_loc, scale, out,
                        num_reqs, num_tokens, num_q_heads, num_kv_heads, head_dim, block_size,
                        num_blocks, max_blocks_per_req, max_query_len, max_seq_len,
                        common_prefix_len, 0, 1.f, 1.f, workspace, workspace_bytes, stream);
}

pa_status pa_mapped_pointer(const void* host_ptr, void** device_ptr) {
  if (host_ptr == nullptr || device_ptr == nullptr) return PA_ERR_INVALID_ARG;
  cudaPointerAttributes a;
  if (cudaPointerGetAttributes(&a, host_ptr) != cudaSuccess) {
    cudaGetLastError();  // clear the error the query recorded
    return PA_ERR_INVALID_ARG;
  }
  if (a.type != cudaMemoryTypeHost) return PA_ERR_INVALID_ARG;
  void* d = nullptr;
  if (cudaHostGetDevicePointer(&d, const_cast<void*>(host_ptr), 0) != cudaSuccess || !d) {
    cudaGetLastError();
    return PA_ERR_CUDA;
  }
  *device_ptr = d;
  return PA_OK;
}

pa_status pa_get_device_error(int* code, long long* detail, int clear) {
  DeviceState* d = nullptr;
  if (pa_status st = device_state(&d)) return st;
  unsigned long long w[2] = {0, 0};
  if (cudaMemcpy(w, d->err, sizeof w, cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  if (code) *code = (int)w[0];
  if (detail) *detail = (long long)w[1];
  if (clear) {
    const unsigned long long z[2] = {0, 0};
    if (cudaMemcpy(d->err, z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

pa_status pa_set_option(int option, int value) {
  switch (option) {
    case PA_OPT_DECODE_SELF_PLAN:
      g_self_plan.store(value ? 1 : 0);
      return PA_OK;
    case PA_OPT_DECODE_TC:
      if (value < 0 || value > 2) return PA_ERR_INVALID_ARG;
      g_decode_tc.store(value);
      return PA_OK;
    case PA_OPT_CASCADE_OVERLAP:
      g_cascade_overlap.store(value ? 1 : 0);
      return PA_OK;
    case PA_OPT_DECODE_TOKEN_MAJOR:
      g_token_major.store(value ? 1 : 0);
      return PA_OK;
    case PA_OPT_DECODE_TM_CTAS_PER_SM:
      if (value != 1 && value != 2) return PA_ERR_INVALID_ARG;
      g_tm_ctas.store(value);
      return PA_OK;
    case PA_OPT_MIXED_PREFILL_CTAS:
      if (value < 0) return PA_ERR_INVALID_ARG;
      g_mixed_ctas.store(value);
      return PA_OK;
    case PA_OPT_MIXED_OVERLAP:
      g_mixed_overlap.store(value ? 1 : 0);
      return PA_OK;
    case PA_OPT_DECODE_MAX_WORKERS:
      if (value < 0) return PA_ERR_INVALID_ARG;
      g_max_workers.store(value);
      return PA_OK;
  }
  return PA_ERR_INVALID_ARG;
}

pa_status pa_set_kernel_timer(int kernel_id, void* start_event, void* stop_event) {
  if (kernel_id < 0 || kernel_id >= kNumTimers) return PA_ERR_INVALID_ARG;
  if ((start_event == nullptr) != (stop_event == nullptr)) return PA_ERR_INVALID_ARG;
  g_timer_start[kernel_id] = static_cast<cudaEvent_t>(start_event);
  g_timer_stop[kernel_id] = static_cast<cudaEvent_t>(stop_event);
  return PA_OK;
}

}  // extern "C"
