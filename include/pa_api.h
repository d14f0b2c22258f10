/*
 * pa_api.h - C ABI of libpagedattn: attention over a paged KV cache on
 * NVIDIA GB300 (sm_103a).
 *
 * Two operations make up the path:
 *
 *   pa_write_kv   scatters each new token's K and V rows into its physical
 *                 cache slot through a slot mapping ("vLLM v1 Deep Dive: How
 *                 LLM(...) and the Server Boot and Generate", Part 3, "Aside -
 *                 KV cache and prefix caching": a slot is
 *                 block_id * block_size + offset and a scatter kernel writes
 *                 the freshly computed K/V there; "vLLM: An Exhaustive
 *                 Technical Study for Kernel Engineers", 2.1, "Reaching the
 *                 kernel").
 *
 *   pa_attention  runs attention for a unified mixed batch in one call:
 *                 prefill-chunk query spans attend causally over [their cached
 *                 prefix + their own new tokens], single-token decodes attend
 *                 over all of their blocks, every request reading K/V through
 *                 its own block table (same Aside, the block_table paragraph;
 *                 same page, Part 3, "Step 4c - Mixed batches" for
 *                 query_start_loc; "vLLM: An Exhaustive Technical Study for
 *                 Kernel Engineers", 2.4, "The seam" and "The backend
 *                 abstraction").
 *
 * Conventions shared by every call
 *  - All tensor arguments are DEVICE pointers owned by the caller. The library
 *    never allocates, frees or synchronises inside pa_write_kv/pa_attention;
 *    work is enqueued on `stream` (a cudaStream_t, or NULL for the legacy
 *    default stream) and the call returns at once.
 *  - Element type of q, k, v, k_cache, v_cache and out: bfloat16, passed as
 *    raw 16-bit storage. Index tensors: slot_mapping int64, the rest int32.
 *  - Layouts (row-major, contiguous):
 *      q, out            [num_tokens][num_q_heads][head_dim]
 *      k, v              [num_tokens][num_kv_heads][head_dim]
 *      k_cache, v_cache  [num_blocks][num_kv_heads][block_size][head_dim]
 *                        (one (block, kv head) is a contiguous block_size x
 *                        head_dim tile: the head-major "HND" block layout,
 *                        which "vLLM: An Exhaustive Technical Study for Kernel
 *                        Engineers", 2.6, names as the default for non-MLA
 *                        models)
 *      block_tables      [num_reqs][max_blocks_per_req]
 *      seq_lens          [num_reqs]
 *      query_start_loc   [num_reqs + 1], query_start_loc[0] == 0, non-decreasing
 *  - Supported shapes: block_size == 16; head_dim 64 or 128;
 *    num_q_heads / num_kv_heads (the GQA group) in {1, 2, 4, 8}. Other values
 *    return PA_ERR_UNSUPPORTED before anything is launched.
 *  - Every device pointer must be 16-byte aligned (PA_ERR_INVALID_ARG).
 *  - Errors that need the data to detect (a slot or block id outside the pool,
 *    seq_len shorter than the query span) are caught by the kernels: the bad
 *    item is skipped and a device error word is set, to be read with
 *    pa_get_device_error. Nothing traps and nothing waits unboundedly; a
 *    bounded wait that gives up reports PA_ERR_TIMEOUT the same way.
 *  - The first call on a device performs a one-time set-up (device property
 *    query and the address of the device error word); make one call, or
 *    pa_init, before capturing a stream into a CUDA graph.
 */
#ifndef PA_API_H
#define PA_API_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID_ARG = -1, /* null pointer, negative size, misaligned pointer, bad shape */
  PA_ERR_UNSUPPORTED = -2, /* block_size, head_dim or GQA group outside the supported set */
  PA_ERR_WORKSPACE = -3,   /* workspace null or smaller than pa_attention_workspace_size */
  PA_ERR_CUDA = -4,        /* a CUDA runtime call or a launch failed */
  PA_ERR_BOUNDS = -5,      /* (device error word) an index was outside its valid range */
  PA_ERR_TIMEOUT = -6      /* (device error word) a bounded wait in a kernel gave up */
} pa_status;

/* Device error word codes (pa_get_device_error `code`). */
#define PA_DEVERR_NONE 0
#define PA_DEVERR_SLOT 1         /* pa_write_kv: slot_mapping[t] >= num_blocks * block_size */
#define PA_DEVERR_BLOCK_ID 2     /* pa_attention: a block table entry outside [0, num_blocks) */
#define PA_DEVERR_LENGTHS 3      /* pa_attention: seq_len < query span, or too many blocks */
#define PA_DEVERR_QSL 4          /* pa_attention: query_start_loc not within [0, num_tokens] */
#define PA_DEVERR_WAIT_TIMEOUT 5 /* a kernel's bounded wait on a copy gave up */
#define PA_DEVERR_PREFIX 6       /* pa_attention_cascade: a request's table does not start
                                    with request 0's common-prefix blocks */

/*
 * One-time per-device set-up for the current device (see the conventions).
 * Idempotent; the other calls do it on first use.
 */
pa_status pa_init(void);

/*
 * Scatter new K/V rows into the paged caches.
 *   k, v           [num_tokens][num_kv_heads][head_dim] bf16, read only
 *   slot_mapping   [num_tokens] int64; token t goes to block
 *                  slot_mapping[t] / block_size, row slot_mapping[t] % block_size.
 *                  A negative slot marks a padding token: it is skipped.
 *   k_cache, v_cache  written at the named slots only; every other slot keeps
 *                  its contents, bit for bit.
 * Copies are exact (bit patterns). Two tokens naming the same slot is the
 * caller's error; which one lands is unspecified. A slot >= num_blocks *
 * block_size is skipped and sets PA_DEVERR_SLOT.
 * head_dim here may be any multiple of 8 (the scatter is type-agnostic).
 */
pa_status pa_write_kv(const void* k, const void* v, const int64_t* slot_mapping,
                      void* k_cache, void* v_cache, int num_tokens, int num_kv_heads,
                      int head_dim, int block_size, int num_blocks, void* stream);

/*
 * Bytes of device workspace pa_attention needs for a batch of this size
 * (planner output and split-KV partial results). The value
 * depends only on the arguments, not on the device. Returns 0 on bad
 * arguments.
 */
size_t pa_attention_workspace_size(int num_reqs, int num_tokens, int num_q_heads,
                                   int num_kv_heads, int head_dim);

/*
 * Attention for a mixed batch of decodes and prefill chunks.
 *   q                [num_tokens][num_q_heads][head_dim] bf16
 *   k_cache, v_cache the pool, already holding this step's new K/V
 *                    (call pa_write_kv first, on the same stream)
 *   block_tables     request r's logical block i is physical block
 *                    block_tables[r][i]; entries past ceil(seq_lens[r] / 16)
 *                    are never read
 *   seq_lens         total KV length of each request, new tokens included
 *   query_start_loc  request r's new tokens are rows
 *                    query_start_loc[r] .. query_start_loc[r+1]-1 of q/out;
 *                    with qlen = that count and ctx = seq_lens[r] - qlen, row
 *                    j attends to keys 0 .. ctx + j (causal, bottom-right
 *                    aligned; a decode is qlen 1 and sees every key)
 *   scale            multiplies q.k before the softmax (usually 1/sqrt(head_dim))
 *   out              [num_tokens][num_q_heads][head_dim] bf16; rows of
 *                    requests with qlen 0 and rows past query_start_loc[num_reqs]
 *                    are left untouched. Device memory, or pinned host memory
 *                    through the address pa_mapped_pointer gives: the kernels
 *                    then store the result across the host link as they
 *                    finish it, so no separate device-to-host copy follows.
 *   query head h reads KV head h / (num_q_heads / num_kv_heads)
 *   max_blocks_per_req  row stride of block_tables
 *   max_query_len, max_seq_len  host-side upper bounds the scheduler already
 *                    knows; they only size launches (max_query_len <= 1 skips
 *                    the prefill-chunk kernel). Values below the true maxima
 *                    are an error (PA_DEVERR_LENGTHS).
 *   workspace        device buffer of at least
 *                    pa_attention_workspace_size(...) bytes, 256-byte aligned,
 *                    no initial contents required; it must not be used by
 *                    another call that runs concurrently on the GPU.
 */
pa_status pa_attention(const void* q, const void* k_cache, const void* v_cache,
                       const int32_t* block_tables, const int32_t* seq_lens,
                       const int32_t* query_start_loc, float scale, void* out, int num_reqs,
                       int num_tokens, int num_q_heads, int num_kv_heads, int head_dim,
                       int block_size, int num_blocks, int max_blocks_per_req,
                       int max_query_len, int max_seq_len, void* workspace,
                       size_t workspace_bytes, void* stream);

/*
 * FP8 KV cache ("vLLM: An Exhaustive Technical Study for Kernel Engineers",
 * 2.8 Quantization & compute kernels: --kv-cache-dtype fp8 stores K and V as
 * E4M3 with one fp32 scale per tensor, k_scale and v_scale; FP8 halves the
 * bytes of a block). E4M3 here is the OCP 8-bit format the GPU implements:
 * 1 sign, 4 exponent bits (bias 7), 3 mantissa bits, no infinities, largest
 * finite 448.
 *
 * pa_write_kv_fp8: as pa_write_kv, but the caches hold one byte per element
 * ([num_blocks][num_kv_heads][block_size][head_dim] uint8) and each element
 * is stored as E4M3(x / scale): the quotient is a correctly rounded binary32
 * division, the conversion rounds to nearest even and saturates at +-448.
 * k_scale / v_scale must be finite and > 0 (PA_ERR_INVALID_ARG otherwise).
 */
pa_status pa_write_kv_fp8(const void* k, const void* v, const int64_t* slot_mapping,
                          void* k_cache, void* v_cache, float k_scale, float v_scale,
                          int num_tokens, int num_kv_heads, int head_dim, int block_size,
                          int num_blocks, void* stream);

/*
 * pa_attention_fp8: pa_attention over E4M3 caches written by pa_write_kv_fp8.
 * Keys are value(code) * k_scale and values value(code) * v_scale, and the
 * dequantisation is fused into both attention kernels, as for a bf16 cache:
 *  - prefill chunks (spans of 16 or more new tokens) run on the tensor-core
 *    kernel, whose converter warps widen each E4M3 tile exactly to bf16 in
 *    shared memory before the bf16 MMA;
 *  - every other span (decodes, short spans) runs on the CUDA-core split-KV
 *    kernel, which widens codes exactly to fp32.
 * k_scale is folded into the query scaling and v_scale into the output. The
 * workspace is pa_attention_workspace_size(...) bytes, as for pa_attention.
 * Errors as pa_attention, plus PA_ERR_INVALID_ARG for a scale that is not
 * finite and > 0.
 */
pa_status pa_attention_fp8(const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, const int32_t* seq_lens,
                           const int32_t* query_start_loc, float scale, float k_scale,
                           float v_scale, void* out, int num_reqs, int num_tokens,
                           int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                           int num_blocks, int max_blocks_per_req, int max_query_len,
                           int max_seq_len, void* workspace, size_t workspace_bytes,
                           void* stream);

/*
 * Cascade attention for a batch whose requests all share one common prefix
 * ("vLLM: An Exhaustive Technical Study for Kernel Engineers", 2.3 Automatic
 * prefix caching & KV reuse, cascade attention: when every request of a batch
 * shares one prefix, attention over the prefix is computed once for the whole
 * batch and merged with each request's attention over its own suffix by
 * log-sum-exp renormalisation; metadata common_prefix_len).
 *
 * The result equals pa_attention's on the same arguments (up to fp32 rounding
 * order). Arguments are pa_attention's plus:
 *   common_prefix_len  tokens of the shared prefix: a positive multiple of
 *                      block_size. Every request's first common_prefix_len /
 *                      block_size block-table entries must equal request 0's,
 *                      and every request's context (seq_len minus its new
 *                      tokens) must be at least common_prefix_len, so that
 *                      each new token sees the whole prefix.
 *   workspace          at least pa_attention_cascade_workspace_size(...) bytes.
 * The prefix pass runs on the tensor cores: for each KV head, the prefix keys
 * against the queries of every new token of the batch (all G heads), split
 * over key chunks, giving fp32 partials (max, sum, unnormalised output) in
 * the workspace. The split-KV kernel then attends each token to its own
 * suffix keys only and folds the prefix partials into its merge. Every span
 * is handled by the split-KV kernel (no prefill-chunk tiles).
 * Errors: host-side as pa_attention, plus PA_ERR_INVALID_ARG for a
 * common_prefix_len that is not a positive multiple of block_size. On the
 * device, a request whose context is shorter than the prefix sets
 * PA_DEVERR_LENGTHS and is skipped (its rows untouched); a request whose
 * table does not start with request 0's prefix blocks sets PA_DEVERR_PREFIX,
 * and its rows are computed with request 0's prefix (they are wrong; the
 * error word says so).
 */
size_t pa_attention_cascade_workspace_size(int num_reqs, int num_tokens, int num_q_heads,
                                           int num_kv_heads, int head_dim);

pa_status pa_attention_cascade(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               const int32_t* query_start_loc, float scale, void* out,
                               int num_reqs, int num_tokens, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks,
                               int max_blocks_per_req, int max_query_len, int max_seq_len,
                               int common_prefix_len, void* workspace, size_t workspace_bytes,
                               void* stream);

/*
 * pa_attention without a caller-provided workspace, for callers that cannot
 * allocate device memory (for example code running inside an allocator's own
 * callbacks, or under a host framework that owns all device memory and offers
 * no allocation hook). The pages describe no such entry point; it has no
 * counterpart there.
 *
 * Arguments are those of pa_attention minus workspace / workspace_bytes; the
 * caller still passes every input and output. The workspace is a fixed
 * scratch array of PA_NOALLOC_SCRATCH_BYTES compiled into the library: each
 * GPU that loads the library holds it until the process exits. The call
 * allocates nothing (no cudaMalloc, no cudaFree, no library allocator).
 *  - A batch whose pa_attention_workspace_size(...) exceeds
 *    PA_NOALLOC_SCRATCH_BYTES is rejected with PA_ERR_WORKSPACE before
 *    anything is launched.
 *  - Argument errors are reported as pa_attention reports them (the same
 *    codes, checked first), whatever the batch size; the size check follows.
 *  - The first call on a device looks up the scratch array's device address
 *    (with that device current). With lazy module loading (the CUDA default)
 *    that lookup is also when the driver places the array in device memory:
 *    an allocation the driver makes once, on that first call. So make the
 *    first call on each device outside any context that must not allocate,
 *    and before any stream capture; later calls allocate nothing.
 *  - Every call on a device shares the one scratch array, which keeps the
 *    last call's contents; the kernels re-initialise everything they read
 *    from it on each call. Calls whose work overlaps on the GPU (different
 *    streams, or different host threads without ordering) race on the
 *    scratch and give wrong results: serialise them.
 */
#define PA_NOALLOC_SCRATCH_BYTES ((size_t)64 << 20)

pa_status pa_attention_noalloc(const void* q, const void* k_cache, const void* v_cache,
                               const int32_t* block_tables, const int32_t* seq_lens,
                               const int32_t* query_start_loc, float scale, void* out,
                               int num_reqs, int num_tokens, int num_q_heads, int num_kv_heads,
                               int head_dim, int block_size, int num_blocks,
                               int max_blocks_per_req, int max_query_len, int max_seq_len,
                               void* stream);

/* Size of the fixed scratch array used by pa_attention_noalloc. */
size_t pa_noalloc_scratch_bytes(void);

/* Human-readable name of a pa_status value (static string). */
const char* pa_status_string(int status);

/*
 * Read the current device's error word: *code gets a PA_DEVERR_* value,
 * *detail the offending index (token, request or block position). With
 * clear != 0 the word is reset. Synchronises the device; not for the hot path.
 * Either output pointer may be NULL.
 * There is one error word per device, in the library's static device memory,
 * shared by every call on that device whatever its stream: the first error
 * recorded since the last clear wins, so calls running concurrently on
 * different streams cannot tell whose error it is, and a clear resets it for
 * all of them. (The word's address is cached at the first call on a device;
 * the library does not support cudaDeviceReset of a device it has used.)
 */
pa_status pa_get_device_error(int* code, long long* detail, int clear);

/*
 * Device address of pinned host memory (cudaHostAlloc / cudaHostRegister,
 * mapped into the device's address space): the address kernels use to reach
 * it, which `out` of the attention calls accepts. PA_ERR_INVALID_ARG when
 * host_ptr is not pinned host memory or device_ptr is NULL; PA_ERR_CUDA on a
 * runtime error. *device_ptr is set only on success.
 */
pa_status pa_mapped_pointer(const void* host_ptr, void** device_ptr);

/*
 * Instrumentation: record `start_event` / `stop_event` (cudaEvent_t handles
 * created by the caller) around every later launch of the given kernel on its
 * stream; pass NULL events to stop. Kernel ids: 0 write_kv, 1 planner,
 * 2 decode (split-KV), 3 prefill chunk, 4 cascade prefix pass, 5 split-KV
 * merge pass. Process-wide setting, not thread-safe.
 */
pa_status pa_set_kernel_timer(int kernel_id, void* start_event, void* stop_event);

/*
 * Process-wide options.
 *   PA_OPT_DECODE_SELF_PLAN (default 1): a batch whose spans are all at most
 *     one token (pure decode), with at most 512 requests and no cascade, is
 *     planned inside the split-KV kernel, and the planner is not launched.
 *     That kernel then starts streaming K/V without waiting for the preceding
 *     KV write; it waits for it (griddepcontrol.wait) only before reading a
 *     request's last block, which holds the newest token.
 *     The results are bit-identical with the option off (the planner path),
 *     which the tests compare. value 0 turns it off.
 * PA_ERR_INVALID_ARG for an unknown option. Not thread-safe.
 */
#define PA_OPT_DECODE_SELF_PLAN 1
/*
 *   PA_OPT_DECODE_TC (default 1): which kernel runs the split-KV work (the
 *     decodes and the spans shorter than 16 tokens) at head_dim 128. 0: the
 *     CUDA-core kernel always. 1: the tensor-core kernel for GQA groups of 4
 *     or 8 query heads per KV head, over a bf16 or an E4M3 cache, where the
 *     CUDA cores' arithmetic per cached byte, not HBM, would set the pace;
 *     the CUDA-core kernel otherwise and for a cascade's suffix pass. 2: the
 *     tensor-core kernel wherever it applies (every group; cascade suffixes
 *     over a bf16 cache). Both give results within the attention tolerances
 *     of the exact result; they are not bit-identical to each other (the
 *     tensor-core kernel rounds P to bf16, or over an E4M3 cache splits the
 *     queries and 256 P into two E4M3 terms each, for its products).
 *   PA_OPT_DECODE_MAX_WORKERS (default 0, no cap): at most this many
 *     split-KV workers share the flattened (token, kv head, block) work, so
 *     a long sequence is split over fewer parts (1: none). For tests of the
 *     split-count invariance; the default uses every worker the launch has.
 *   PA_OPT_MIXED_OVERLAP (default 1): in a call with prefill chunks and
 *     split-KV work on the tensor-core split-KV kernel (bf16 cache), the
 *     planner may give the chunks a few SMs and the split-KV work the rest,
 *     so that both run at once (the mixed batch of "vLLM v1 Deep Dive",
 *     Part 3, Step 4c, whose prefill and decode spans one forward serves
 *     together). It does so when its cost
 *     model (per-SM prefill and split-KV rates measured on GB300) puts the
 *     two ending together sooner than one after the other, and otherwise runs
 *     them in turn as with the option off. The chunks' results are
 *     bit-identical either way; the split-KV results stay within the
 *     attention tolerances (fewer workers slice the keys differently).
 *     value 0 turns it off.
 */
#define PA_OPT_DECODE_TC 2
#define PA_OPT_DECODE_MAX_WORKERS 3
#define PA_OPT_MIXED_OVERLAP 4
/*
 *   PA_OPT_DECODE_TOKEN_MAJOR (default 1): over an E4M3 cache with eight KV
 *     heads at head_dim 128, the tensor-core split-KV kernel takes one 16-key
 *     block of all eight KV heads per tile (one tensor copy each for K and V,
 *     each head's keys in one half-warp). 0: the per-(token, kv head) tiles
 *     of the other groupings. Both are within the attention tolerances of
 *     the exact result on the same codes; they are not bit-identical.
 */
#define PA_OPT_DECODE_TOKEN_MAJOR 5
/*
 *   PA_OPT_CASCADE_OVERLAP (default 1): in pa_attention_cascade, with the
 *     suffix pass on the CUDA-core split-KV kernel (the default routing), the
 *     prefix pass takes a few SMs (about two of its work items each) and the
 *     suffix pass the rest, both at once; every (token, kv head) then leaves
 *     fp32 partials and the merge pass folds suffix and prefix together.
 *     Results stay within the attention tolerances (the folding order
 *     differs). value 0: the prefix pass first, folded by the suffix pass.
 */
#define PA_OPT_CASCADE_OVERLAP 6
/*
 *   PA_OPT_DECODE_TM_CTAS_PER_SM (default 2; 1 or 2, anything else is
 *     PA_ERR_INVALID_ARG): CTAs per SM of the token-major E4M3 kernel. With 2
 *     (taken only at G = Hq / Hkv <= 4; G = 8 always runs one) each SM runs
 *     two CTAs of two copy stages each instead of one of four, so twice as
 *     many workers slice the keys; results stay within the attention
 *     tolerances.
 */
#define PA_OPT_DECODE_TM_CTAS_PER_SM 7
/*
 *   PA_OPT_MIXED_PREFILL_CTAS (default 0; negative is PA_ERR_INVALID_ARG):
 *     in an overlapped mixed batch (PA_OPT_MIXED_OVERLAP), how many SMs the
 *     prefill chunks take beside the split-KV work. 0: the planner's cost
 *     model decides, and may run the two in turn instead. n > 0: always
 *     overlap, with min(n, SMs / 2) SMs for the chunks. Results do not depend
 *     on it beyond the attention tolerances (the split-KV slicing changes).
 */
#define PA_OPT_MIXED_PREFILL_CTAS 8
pa_status pa_set_option(int option, int value);

/* Number of kernel launches the library has issued in this process. */
long long pa_launch_count(void);

/* Library ABI version (major * 10000 + minor * 100 + patch). */
int pa_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_API_H */
