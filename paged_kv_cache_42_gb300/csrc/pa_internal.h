// Internal declarations shared by the translation units of libpagedattn.
// Host and device code; no torch, no CUDA graph state.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "pa_api.h"

namespace pa {

constexpr int kBlockSize = 16;
// Upper bound on the number of split-KV decode workers (warps) of one launch.
// The workspace reserves one partial-result slot per (token, kv head) plus one
// per worker, so it is part of the workspace size formula.
constexpr int kMaxDecodeWorkers = 4096;
// The planner keeps per-token scratch in shared memory up to this many tokens.
constexpr int kPlanSmemTokens = 4096;
// A decode-only batch (every span at most one token) of up to this many
// requests is planned by the split-KV kernel itself, in shared memory, so
// that kernel need not wait for the planner or the KV write before streaming.
constexpr int kSelfPlanMaxReqs = 512;

// Split-KV workers used for W flattened positions when `all` are launched:
// at least PA_DEC_MIN_POS positions each (the planner and the split-KV kernel
// must agree).
#ifndef PA_DEC_MIN_POS
#define PA_DEC_MIN_POS 8
#endif
__host__ __device__ inline int plan_workers(int W, int all) {
  int n = W / PA_DEC_MIN_POS;
  return n < 1 ? 1 : (n > all ? all : n);
}
// Worker w of NW takes positions [worker_begin(w), worker_begin(w + 1)) of
// the W flattened positions; worker_of(x) is the worker that takes x. The
// split-KV kernel and the merge pass must slice alike.
__host__ __device__ inline int worker_begin(int w, int W, int NW) {
  return (int)((long long)w * W / NW);
}
__host__ __device__ inline int worker_of(int x, int W, int NW) {
  return (int)(((long long)(x + 1) * NW - 1) / W);
}

// One entry per token that has keys to attend to, in token order (the
// planner compacts away tokens with no work). `base` is the first position
// of the token's (kv head, block) sequence in the flattened decode work list.
struct UnitInfo {
  int tok;   // row of q / out
  int req;   // request (row of block_tables)
  int len;   // number of keys this token attends to (causal limit + 1)
  int base;  // flattened position of (kv head 0, block 0)
};
static_assert(sizeof(UnitInfo) == 16, "UnitInfo is loaded as one 16-byte vector");

struct WsHeader {
  int num_units;      // K: tokens with work on the split-KV path
  int num_positions;  // W: sum over units of Hkv * ceil(len / 16)
  int num_tiles;      // prefill-chunk tiles for the tensor-core path
  // Overlapped mixed batch (PlanParams::overlap): CTAs of the prefill-chunk
  // grid that take items (the rest retire at once), and split-KV workers.
  // Otherwise prefill_ctas is the whole grid's share and decode_workers the
  // launch's worker count.
  int prefill_ctas;
  int decode_workers;
  int pad[59];
};

// Overlapped mixed batch: the planner gives the prefill-chunk items P SMs
// and the split-KV work the other S - P, when the two then end together
// sooner than one after the other. Costs, measured on GB300 at head_dim 128:
// one prefill step (two 128-row tiles against 128 keys) holds an SM for
// about kPrefillStepUs; the split-KV kernel streams about kDecodeSmBytesPerUs
// per SM until the copy peak (kHbmBytesPerUs) caps it.
constexpr float kPrefillStepUs = 2.4f;
constexpr float kDecodeSmBytesPerUs = 47.0e3f;
constexpr float kHbmBytesPerUs = 6.6e6f;
constexpr float kOverlapMargin = 0.85f;  // prefill share planned to end this early

// Requests with at least this many new tokens go to the tensor-core
// prefill-chunk kernel; shorter ones (decodes, short verify spans) to the
// split-KV kernel.
#ifndef PA_PREFILL_MIN_QLEN
#define PA_PREFILL_MIN_QLEN 16
#endif
constexpr int kPrefillMinQlen = PA_PREFILL_MIN_QLEN;

// One prefill work item: two 128-row tiles of request `req`, kv head `kv`,
// chunk tokens j0 .. j0 + 2*128/G - 1, attending to nkv 128-key tiles.
struct PrefillTile {
  int req, kv, j0, nkv;
};
static_assert(sizeof(PrefillTile) == 16, "tiles are 16 bytes");
static_assert(sizeof(WsHeader) == 256, "header occupies the first 256 bytes");

// Workspace carve-up, identical on host and device.
struct WsLayout {
  size_t header_off, units_off, tiles_off, raw_off, workers_off, tasks_off, partials_off;
  // E4M3 caches on the tensor-core split-KV kernel: each query row scaled by a
  // power of two and split into two E4M3 terms (hi, lo: 2 x head_dim bytes),
  // and the inverse scales, 8 floats per (token, kv head)
  size_t qsplit_off, qinv_off, total;
  int slot_floats;  // floats per partial-result slot
};

__host__ __device__ inline size_t pa_align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline WsLayout ws_layout(int num_reqs, int num_tokens, int num_q_heads,
                                              int num_kv_heads, int head_dim) {
  WsLayout l;
  const int G = num_q_heads / num_kv_heads;
  l.slot_floats = 16 + G * head_dim;  // [m x G][l x G] padded to 16 floats, then o[G][D]
  l.header_off = 0;
  l.units_off = pa_align256(sizeof(WsHeader));
  l.tiles_off = l.units_off + pa_align256(sizeof(UnitInfo) * (size_t)(num_tokens + 1));
  // a chunk of qlen tokens makes ceil(qlen / (128 / G)) <= qlen / 16 + 1 tiles per kv head
  const size_t max_tiles = (size_t)num_kv_heads * ((size_t)num_tokens / 16 + (size_t)num_reqs + 1);
  l.raw_off = l.tiles_off + pa_align256(sizeof(PrefillTile) * max_tiles);
  l.workers_off = l.raw_off + pa_align256(8 * (size_t)num_tokens);
  l.tasks_off = l.workers_off + pa_align256(sizeof(int) * (size_t)kMaxDecodeWorkers);
  l.partials_off = l.tasks_off + pa_align256(sizeof(int4) * (size_t)kMaxDecodeWorkers);
  const size_t slots = (size_t)num_tokens * num_kv_heads + kMaxDecodeWorkers;
  l.qsplit_off = l.partials_off + pa_align256(sizeof(float) * (size_t)l.slot_floats * slots);
  l.qinv_off = l.qsplit_off + pa_align256((size_t)num_tokens * num_q_heads * 2 * head_dim);
  l.total = l.qinv_off + pa_align256(sizeof(float) * 8 * (size_t)num_tokens * num_kv_heads);
  return l;
}

// Cascade prefix pass: work items are (pair of 128-row tiles, kv head, key
// chunk); the prefix keys are split into as many chunks as bring the item
// count to about this many, at most kMaxPrefixChunks. More chunks shorten the
// prefix pass but give the split-KV kernel more partials to fold per token
// (on the 128-token prefix-sharing batch: 24 items, two chunks, measured
// 64.1 us per step against 65.0 at 40 and 64.8 at 64).
#ifndef PA_PREFIX_TARGET_ITEMS
#define PA_PREFIX_TARGET_ITEMS 24
#endif
constexpr int kPrefixTargetItems = PA_PREFIX_TARGET_ITEMS;
constexpr int kMaxPrefixChunks = 16;

__host__ __device__ inline int prefix_pairs(int num_tokens, int group) {
  const int tok_per_pair = 2 * (128 / group);
  return (num_tokens + tok_per_pair - 1) / tok_per_pair;
}
// Key chunks for a prefix of `key_tiles` 128-key tiles (0: the bound used to
// size the workspace, before the prefix length is known).
__host__ __device__ inline int prefix_chunks(int num_tokens, int num_kv_heads, int group,
                                             int key_tiles) {
  const int per_chunk = prefix_pairs(num_tokens, group) * num_kv_heads;
  int c = (kPrefixTargetItems + per_chunk - 1) / per_chunk;
  if (c > kMaxPrefixChunks) c = kMaxPrefixChunks;
  if (key_tiles > 0 && c > key_tiles) c = key_tiles;
  return c < 1 ? 1 : c;
}

// Bytes of prefix partials a cascade call needs beyond the ws_layout total:
// one partial slot per (chunk, token, kv head).
__host__ __device__ inline size_t prefix_partials_bytes(int num_tokens, int num_q_heads,
                                                        int num_kv_heads, int head_dim) {
  const int G = num_q_heads / num_kv_heads;
  const size_t slot = sizeof(float) * (size_t)(16 + G * head_dim);
  return pa_align256(slot * (size_t)prefix_chunks(num_tokens, num_kv_heads, G, 0) *
                     (size_t)num_tokens * (size_t)num_kv_heads);
}

struct PlanParams {
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_tables;  // read only for the cascade prefix check
  int prefix_blocks;            // cascade: blocks of the common prefix; 0 otherwise
  int early_trigger;            // release the next grid at the top (it needs no plan at first)
  int num_reqs, num_tokens, num_kv_heads, max_blocks_per_req, max_query_len, max_seq_len;
  int group;        // G = Hq / Hkv
  int use_prefill;  // route requests with qlen >= kPrefillMinQlen to the tensor-core kernel
  int num_workers;  // split-KV workers the decode launch provides
  // overlapped mixed batch allowed: the planner may split the SMs between the
  // prefill-chunk and split-KV grids (num_sms of them; position_bytes of
  // K and V per split-KV position)
  int overlap, num_sms, position_bytes;
  int prefill_ctas_override;  // > 0: the prefill-chunk grid's share, instead of the cost model
  int token_major;  // positions per token are its blocks (all kv heads at once)
  WsHeader* header;
  UnitInfo* units;
  PrefillTile* tiles;
  int2* raw;        // per-token scratch when the batch is too large for shared memory
  int* worker_unit; // first unit of each split-KV worker (only when the batch fits)
  unsigned long long* err;
};

struct PrefillLaunch {
  // cascade prefix pass (prefix_len > 0): no planner tiles; items are
  // (pair, kv head, key chunk) over request 0's first prefix_len keys and the
  // output is fp32 partials, one slot per (chunk, token, kv head)
  int prefix_len, prefix_chunks, slot_floats;
  float* prefix_partials;
  // E4M3 caches: k_cache / v_cache hold codes; k_scale is already folded into
  // scale_log2, v_scale multiplies the output
  int kv_fp8;
  float v_scale;
  const void* q;
  const void* k_cache;
  const void* v_cache;
  const int32_t* qsl;
  const int32_t* seq_lens;
  const int32_t* block_tables;
  uint16_t* out;
  const WsHeader* header;
  const PrefillTile* tiles;
  int num_tokens, num_q_heads, num_kv_heads, head_dim, num_blocks, bt_stride;
  float scale_log2;
  // overlapped mixed batch: header->prefill_ctas CTAs take the items and the
  // grid releases the split-KV grid as soon as it has read that count.
  // Overlapped cascade (prefix pass): prefix_ctas CTAs take the items, and the
  // grid releases the suffix split-KV grid once the planner has completed.
  int overlap, prefix_ctas;
  unsigned long long* err;
};

struct DecodeParams {
  const uint16_t* q;
  const void* k_cache;  // bf16, or E4M3 codes in the f8 instantiation
  const void* v_cache;
  float v_scale;        // output multiplier: the E4M3 V scale, 1 for bf16
  const int32_t* block_tables;
  uint16_t* out;
  int bt_stride, num_q_heads, num_kv_heads, num_blocks;
  float scale_log2;  // scale * log2(e): scores are kept in base-2 exponent units
  const WsHeader* header;
  const UnitInfo* units;
  const int* worker_unit;  // null: each worker searches for its first unit
  float* partials;
  int slot_floats;
  // cascade: keys start after the common prefix, whose partials are merged in
  int key_start_blocks;          // 0 without a cascade
  const float* prefix_partials;  // null without a cascade
  int prefix_chunks, num_tokens;
  // self-planned decode-only batch: the kernel builds its unit table from these
  // and its first CTA publishes the position count (header_out) for the merge pass
  int self_plan, num_reqs, max_blocks_per_req, max_query_len, max_seq_len;
  const int32_t* qsl;
  const int32_t* seq_lens;
  WsHeader* header_out;
  // merge task of the slice boundary before each worker (see MergeParams)
  int4* merge_tasks;
  // workers the slicing uses: at most the launched ones (a smaller value
  // leaves the rest idle and gives every worker a longer slice)
  int max_workers;
  // E4M3 caches on the tensor-core kernel: the split query rows and inverse
  // scales (WsLayout::qsplit_off, qinv_off), written by launch_qsplit
  const unsigned char* qsplit;
  const float* qinv;
  // overlapped mixed batch / cascade: this grid starts while the tensor-core
  // grid before it (prefill chunks / cascade prefix pass) still runs (the
  // planner, its predecessor's predecessor, is complete); the grid completes
  // only after that grid. Mixed batch: the worker count comes from the header.
  int overlap;
  // overlapped cascade: every (token, kv head) leaves partials, whole ones
  // too; the merge pass folds them with the prefix partials (MergeParams::all_units)
  int fold_later;
  unsigned long long* err;
};

// Merge pass: every (token, kv head) whose key blocks were split over more
// than one split-KV worker is merged from the workers' partials (and, in a
// cascade, the prefix partials), after the split-KV grid. Each split-KV
// worker w > 0 leaves the task of the slice boundary before it in tasks[w]:
// {token, kv head, first worker, last worker} of the (token, kv head) that
// boundary splits, if w is the first worker after its first boundary, else
// token -1.
struct MergeParams {
  const WsHeader* header;
  const int4* tasks;
  const float* partials;
  int slot_floats;
  int num_workers;  // split-KV workers launched (the slicing's upper bound)
  int workers_from_header;  // overlapped mixed batch: header->decode_workers, if fewer
  // overlapped cascade: one CTA per (unit, kv head), merging that portion's
  // suffix partials (the workers holding it, from the unit table) and the
  // prefix chunks; grid units * Hkv
  int all_units;
  const UnitInfo* units;
  int token_major;          // token-major split-KV: a task {token, -, wf, wl} covers every
                            // kv head (a CTA per boundary, a warp per kv head), slot
                            // (token + w) * Hkv + kv head
  int num_q_heads, num_kv_heads, num_tokens;
  int key_start_blocks;
  const float* prefix_partials;
  int prefix_chunks;
  float v_scale;
  uint16_t* out;
};

struct WriteParams {
  const uint16_t* k;
  const uint16_t* v;
  const int64_t* slot_mapping;
  void* k_cache;  // bf16, or E4M3 codes when kv_fp8
  void* v_cache;
  int kv_fp8;
  float k_scale, v_scale;  // E4M3 caches only
  int num_tokens, num_kv_heads, head_dim;
  long long num_slots;
  unsigned long long* err;
};

// Device error word: [0] = code, [1] = detail. First error wins.
__device__ inline void report_error(unsigned long long* err, int code, long long detail) {
  if (atomicCAS(err, 0ull, (unsigned long long)code) == 0ull)
    atomicExch(err + 1, (unsigned long long)detail);
}

// Host-side checks of an attention call's arguments, everything but the
// workspace (shapes, supported sizes, pointers, alignment, index ranges), in
// the order pa_attention reports them. *nothing_to_do is set for an empty
// batch (no request or no token), which is not an error.
pa_status check_attention_args(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               const int32_t* query_start_loc, float scale, const void* out,
                               int num_reqs, int num_tokens, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks,
                               int max_blocks_per_req, int max_query_len, int max_seq_len,
                               int prefix_len, int kv_fp8, float k_scale, float v_scale,
                               bool* nothing_to_do);

// Launchers (return the launch's cudaError_t).
cudaError_t launch_write_kv(const WriteParams& p, cudaStream_t s);
cudaError_t launch_plan(const PlanParams& p, cudaStream_t s);
// head_dim / G select the instantiation; unsupported combinations return
// cudaErrorInvalidValue. occ_cap bounds the resident CTAs per SM (the grid is
// SMs x min(occupancy, occ_cap)).
// f8 selects the E4M3-cache instantiation.
cudaError_t launch_decode(const DecodeParams& p, int head_dim, int group, bool f8, int num_sms,
                          int occ_cap, cudaStream_t s, int* workers_out);
// The merge pass after a split-KV launch of num_workers workers (p.num_workers).
cudaError_t launch_merge(const MergeParams& p, int head_dim, int group, cudaStream_t s);
// Split-KV workers launch_decode will use on this device (0 on error).
int decode_workers(int head_dim, int group, bool f8, int num_sms, int occ_cap);

// Tensor-core split-KV decode (decode_tc.cu): one CTA per SM is one worker.
// Supported for head_dim 128, over a bf16 cache (a cascade's suffix pass
// included) or an E4M3 cache; it takes the same plan, partial slots and merge
// tasks as launch_decode.
bool decode_tc_supported(int head_dim, int group, bool f8, int key_start_blocks);
int decode_tc_workers(int num_sms);
cudaError_t launch_decode_tc(const DecodeParams& p, int group, bool f8, int num_sms,
                             cudaStream_t s, int* workers_out);
// E4M3 caches: split every query row for the tensor-core kernel (into
// p.qsplit / p.qinv), as a programmatic dependent of the preceding grid that
// completes only after it.
cudaError_t launch_qsplit(const DecodeParams& p, int group, cudaStream_t s);
// Token-major tensor-core split-KV decode over an E4M3 cache (decode_tm.cu):
// eight KV heads, head_dim 128. Its positions are (token, block) - the plan
// built with PlanParams::token_major - and its partial of (token, kv head)
// from worker w sits in slot (token + w) * 8 + kv head (MergeParams::token_major).
// It runs ctas_per_sm (1 or 2; 2 only for G <= 4) CTAs per SM, one worker
// each: decode_tm_workers of them.
int decode_tm_workers(int group, int num_sms, int ctas_per_sm);
bool decode_tm_supported(int head_dim, int group, int num_kv_heads, int workers);
cudaError_t launch_decode_tm(const DecodeParams& p, int group, int num_sms, int ctas_per_sm,
                             cudaStream_t s, int* workers_out);

// 2-D tiled tensor map (CUtensorMap, passed as void*) over a row-major bf16
// matrix of `rows` rows of `inner` elements, `row_stride_bytes` apart, with a
// {box_inner, box_rows} box and 128-byte swizzle. False if the driver's
// encoder is unavailable or rejects the arguments.
bool encode_tmap_bf16_2d(void* tmap, const void* ptr, uint64_t inner, uint64_t rows,
                         uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_rows);
// Tiled tensor map of `rank` (<= 5) dimensions over bf16 data: dims[0] is
// contiguous; strides_bytes[i] is the byte stride of dimension i + 1 (any
// order: a dimension may step inside another's extent); 128-byte swizzle.
bool encode_tmap_bf16(void* tmap, int rank, const void* ptr, const uint64_t* dims,
                      const uint64_t* strides_bytes, const uint32_t* box);
// The same over byte data (E4M3 codes).
bool encode_tmap_u8(void* tmap, int rank, const void* ptr, const uint64_t* dims,
                    const uint64_t* strides_bytes, const uint32_t* box);

// Resident split-KV CTAs per SM: two suit long per-token key ranges (each
// worker's slice stays long); the short suffixes of a cascade call run better
// with a third, which hides more latency.
#ifndef PA_DEC_OCC_CAP
#define PA_DEC_OCC_CAP 2
#endif
#ifndef PA_DEC_OCC_CAP_CASCADE
#define PA_DEC_OCC_CAP_CASCADE 3
#endif
// Smallest GQA group the tensor-core split-KV kernel takes in automatic mode.
// From 4 query heads per KV head it is at least as fast per step as the
// CUDA-core kernel (equal on the Llama-8B decode batch, faster on the mixed,
// prefix-sharing and long-context batches); below, the CUDA cores are not
// short of arithmetic.
#ifndef PA_DECODE_TC_MIN_GROUP
#define PA_DECODE_TC_MIN_GROUP 4
#endif
#ifndef PA_DEC_OCC_CAP_FP8
#define PA_DEC_OCC_CAP_FP8 3  // E4M3 calls: smaller rings, a third CTA where registers allow
#endif
cudaError_t launch_prefill(const PrefillLaunch& a, int num_sms, cudaStream_t s);

}  // namespace pa
