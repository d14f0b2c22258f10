/*
 * pa_host.h - host-side runtime of libpagedattn: the pieces that produce the
 * metadata the attention kernels consume (block tables, slot mapping,
 * query_start_loc, seq_lens).
 *
 *  1. A physical block pool with reference counts, an LRU free queue and a
 *     chained-hash prefix cache ("Deep Dive - vLLM", "Block pool, prefix
 *     cache, and eviction"; "Inside the vLLM Engine", "The pool, the queue,
 *     and the hash"; "vLLM: An Exhaustive Technical Study for Kernel
 *     Engineers", 2.1 and 2.3):
 *      - every block has a fixed physical id, a reference count and, once
 *        full and registered, a 32-byte hash;
 *      - free blocks wait in a doubly linked queue and allocation pops its
 *        head; a released block whose count drops to zero goes to the tail
 *        if it holds a hash (a later prefix hit may still rescue it) and to
 *        the head if it does not; a request's blocks are released last
 *        block first;
 *      - a cached block keeps its hash while free and loses it only when it
 *        is popped for reuse; a prefix hit on a free cached block takes it
 *        back out of the queue.
 *  2. The chained block hash: SHA-256 (FIPS 180-4) over
 *        parent hash (32 bytes; 32 zero bytes for the first block)
 *        || block token ids (int32, little endian) || extra key bytes
 *     (adapter id, multimodal hashes, cache salt; the caller serialises
 *     them, tagged by source). The chaining and SHA-256 come from the pages;
 *     the byte serialisation is this library's own. A pool may select
 *     instead the faster, non-cryptographic XXH64 over the same bytes (the
 *     pages' "xxhash variant a flag away"; "Automatic Prefix Caching" on the
 *     selectable hash algorithm): its 64-bit value, little endian, fills the
 *     first 8 bytes of the 32-byte hash and the rest are zero. Distinct
 *     prefixes then collide with probability about n^2 / 2^65 over n cached
 *     blocks, the trade-off the pages attach to a fast hash.
 *  3. A token-budget scheduler step ("Deep Dive - vLLM", "The V1 scheduler:
 *     one token budget"; "vLLM v1 Deep Dive: How LLM(...) and the Server Boot
 *     and Generate", Part 3 "Step 3 - Scheduler iteration"; "vLLM: An
 *     Exhaustive Technical Study for Kernel Engineers", 2.2):
 *      - pass 1 walks the running requests in order, granting each
 *        min(tokens it still needs, long-prefill threshold, budget left,
 *        room under max_model_len); when its blocks cannot be allocated the
 *        last running request is preempted (blocks released, computed count
 *        reset, put back at the front of the waiting queue) until they can,
 *        or until the request itself was the one preempted;
 *      - pass 2 (skipped in a step that preempted) admits waiting requests
 *        in order while budget is left and fewer than max_running requests
 *        run: a request's computed count starts at its longest cached
 *        prefix (whole blocks, at most num_tokens - 1 tokens); without
 *        chunked prefill a request that does not fit the budget stops
 *        admission; a request whose blocks cannot be allocated stops it too;
 *      - every scheduled request's computed count then advances by its grant
 *        (planned state, before the GPU runs) and its newly full blocks are
 *        registered in the prefix cache.
 *
 * All functions are host-only and synchronous; none touches the GPU. The
 * pool allocates only in pa_pool_create. The scheduler allocates in its
 * create and add calls, and a step may grow storage it keeps (a request's
 * block and hash lists, its queues and per-step lists; amortised, reused
 * from step to step). Hashing and lookups allocate nothing. Objects are
 * not thread-safe. Negative return values are pa_status codes.
 */
#ifndef PA_HOST_H
#define PA_HOST_H

#include <stddef.h>
#include <stdint.h>

#include "pa_api.h"

#ifdef __cplusplus
extern "C" {
#endif

/* ---------------------------------------------------------------- pool -- */

typedef struct pa_block_pool pa_block_pool;

/* A pool of `num_blocks` blocks of `block_size` tokens. `ids` lists their
 * physical ids in the initial free-queue order (head first), all distinct
 * and >= 0; NULL means 0 .. num_blocks-1. Returns NULL on bad arguments or
 * allocation failure. The pool owns its bookkeeping; the caller frees it
 * with pa_pool_destroy (NULL is accepted). */
pa_block_pool* pa_pool_create(int num_blocks, int block_size, const int32_t* ids);
void pa_pool_destroy(pa_block_pool* pool);

int pa_pool_num_blocks(const pa_block_pool* pool);
int pa_pool_block_size(const pa_block_pool* pool);
int pa_pool_num_free(const pa_block_pool* pool);

/* Pop `n` blocks from the free-queue head into out_ids[0..n) with reference
 * count 1, dropping any hash they held. Fewer than n free blocks:
 * PA_ERR_BOUNDS and nothing changes. */
pa_status pa_pool_allocate(pa_block_pool* pool, int n, int32_t* out_ids);

/* Release one reference to each of ids[0..n), last id first. A block whose
 * count reaches zero joins the free queue (tail if it holds a hash, head if
 * not). An id not in the pool, or more releases than references:
 * PA_ERR_INVALID_ARG and nothing changes. */
pa_status pa_pool_free(pa_block_pool* pool, const int32_t* ids, int n);

/* Add one reference to each of ids[0..n) (prefix-cache hits); a block with
 * count 0 leaves the free queue. Unknown id: PA_ERR_INVALID_ARG, nothing
 * changes. */
pa_status pa_pool_touch(pa_block_pool* pool, const int32_t* ids, int n);

/* Register a live block (count > 0) that holds no hash under `hash`. If
 * another block already holds that hash, this block stays unregistered and
 * the call still returns PA_OK (the first block keeps the hash; block tables
 * are append-only, so no request is re-pointed). A free or unknown block, or
 * one that already holds a hash: PA_ERR_INVALID_ARG. */
pa_status pa_pool_cache_block(pa_block_pool* pool, int32_t id, const uint8_t hash[32]);

/* Block registered under `hash`, or -1. */
int32_t pa_pool_lookup(const pa_block_pool* pool, const uint8_t hash[32]);

/* Reference count of a block, -1 for an unknown id. */
int pa_pool_ref_count(const pa_block_pool* pool, int32_t id);
/* 1 if the block holds a hash, 0 if not, -1 for an unknown id. */
int pa_pool_is_cached(const pa_block_pool* pool, int32_t id);

/* Copy the free queue, head first, into out[0..max); returns its length
 * (which may exceed max). */
int pa_pool_free_queue(const pa_block_pool* pool, int32_t* out, int max);

/* Block hash algorithms (pa_pool_set_hash_algo, pa_block_hash_algo). */
#define PA_HASH_SHA256 0 /* default */
#define PA_HASH_XXH64 1

/* Select the pool's block hash algorithm: the one the scheduler drawing from
 * it and pa_pool_find_cached_prefix use. Allowed only while no block holds a
 * hash (digests of two algorithms never share a table); PA_ERR_INVALID_ARG
 * otherwise or for an unknown algorithm. */
pa_status pa_pool_set_hash_algo(pa_block_pool* pool, int algo);
/* The pool's algorithm, or -1 for a NULL pool. */
int pa_pool_hash_algo(const pa_block_pool* pool);

/* ---------------------------------------------------------------- hash -- */

/* Chained block hash of tokens[0..num_tokens) (see above) into out.
 * `parent` NULL means the first block; `extra` may be NULL when
 * extra_len == 0. */
void pa_block_hash(const uint8_t parent[32], const int32_t* tokens, int num_tokens,
                   const uint8_t* extra, int extra_len, uint8_t out[32]);

/* The same with the given algorithm (PA_HASH_*); PA_ERR_INVALID_ARG for an
 * unknown one, out untouched. */
pa_status pa_block_hash_algo(int algo, const uint8_t parent[32], const int32_t* tokens,
                             int num_tokens, const uint8_t* extra, int extra_len,
                             uint8_t out[32]);

/* Plain SHA-256 of len bytes (FIPS 180-4). */
void pa_sha256(const uint8_t* data, size_t len, uint8_t out[32]);
/* Plain XXH64 of len bytes with the given seed. */
uint64_t pa_xxh64(const uint8_t* data, size_t len, uint64_t seed);

/* The longest run of the prompt's full blocks registered in the pool,
 * chained from the first block and stopping at the first miss, limited to
 * num_tokens - 1 tokens so that one position is left to compute. Writes the
 * block ids to out_ids (at most max_blocks) and returns the number of cached
 * tokens (a multiple of the block size), or a negative pa_status. Changes
 * nothing in the pool. */
int pa_pool_find_cached_prefix(const pa_block_pool* pool, const int32_t* tokens,
                               int num_tokens, const uint8_t* extra, int extra_len,
                               int32_t* out_ids, int max_blocks);

/* Tokens a prompt of `prompt_length` can skip given `shared` tokens of
 * exactly matching prefix: whole blocks only, and at most prompt_length - 1
 * (the last position is recomputed for its logits). PA_ERR_INVALID_ARG
 * unless block_size > 0, prompt_length > 0 and 0 <= shared <= prompt_length.
 * ("Deep Dive - vLLM", "Block pool, prefix cache, and eviction".) */
pa_status pa_reusable_tokens(int shared, int prompt_length, int block_size, int* out);

/* ----------------------------------------------------------- scheduler -- */

typedef struct pa_scheduler pa_scheduler;

typedef struct pa_sched_config {
  int token_budget;           /* max_num_batched_tokens, > 0 */
  int max_running;            /* max_num_seqs; <= 0 means no limit */
  int long_prefill_threshold; /* per-request cap per step; <= 0 means none */
  int max_model_len;          /* > 0; a request never holds more tokens */
  int max_blocks_per_req;     /* block-table row stride, >= ceil(max_model_len / block_size) */
  int enable_prefix_caching;  /* nonzero: look up and register block hashes */
  int enable_chunked_prefill; /* nonzero: a waiting request may get part of its prompt */
} pa_sched_config;

/* Caller-owned output of one step. The caller sets the capacities and the
 * array pointers; pa_sched_step fills the arrays and the counts.
 * Requests appear in the order they were scheduled (running first, then
 * newly admitted); request i's tokens are [query_start_loc[i],
 * query_start_loc[i+1]). block_tables is [num_reqs][block_table_stride],
 * the stride being the widest scheduled request's block count (so a step
 * writes no more of the table than it uses; max_blocks_per_req with
 * block_tables_retained), with -1 past each request's blocks; its capacity
 * is max_reqs * max_blocks_per_req entries. */
typedef struct pa_sched_output {
  int max_reqs, max_tokens, max_preempted; /* capacities */
  int64_t* req_ids;         /* [max_reqs] */
  int32_t* num_scheduled;   /* [max_reqs] tokens granted */
  int32_t* num_computed;    /* [max_reqs] tokens computed before this step (context) */
  int32_t* query_start_loc; /* [max_reqs + 1] */
  int32_t* seq_lens;        /* [max_reqs] context + granted */
  int32_t* block_tables;    /* [num_reqs][block_table_stride], capacity max_reqs * max_blocks_per_req */
  int64_t* slot_mapping;    /* [max_tokens] block * block_size + offset */
  int32_t* positions;       /* [max_tokens] absolute position of each token */
  int32_t* input_tokens;    /* [max_tokens] token id at that position */
  int64_t* preempted_ids;   /* [max_preempted], may be NULL when max_preempted == 0 */
  /* filled by pa_sched_step */
  int num_reqs, num_tokens, num_preempted;
  int max_query_len, max_seq_len;
  int block_table_stride;   /* row stride of block_tables, >= 1 */
  int num_decode_reqs;      /* requests granted 1 token that is past their prompt */
  /* The step's profile signature ("vLLM v1 Deep Dive: How LLM(...) and the
   * Server Boot and Generate", Part 3, Step 4c: a trace names each forward
   * execute_context_A(a)_generation_B(b)): context requests are those whose
   * span starts inside their prompt (prefill, chunked or not), generation
   * requests those whose span starts past it (decode); with their tokens. */
  int num_context_reqs, num_context_tokens;
  int num_generation_reqs, num_generation_tokens;
  /* Set by the caller. Nonzero selects retained block tables: the row stride
   * is fixed at the configuration's max_blocks_per_req (so rows stay where
   * earlier steps put them), and the caller promises that block_tables is
   * the buffer this scheduler's previous successful step wrote, unmodified
   * since. The step then writes only what differs from what that step left:
   * the new blocks of a row whose request and block list carry over (at the
   * same row), every other row in full. The result is the same table as
   * writing every row at that stride. A buffer address or row stride other
   * than the previous step's means writing every row in full. */
  int block_tables_retained;
} pa_sched_output;

/* A scheduler drawing blocks from `pool`, which it does not own and which
 * must outlive it. NULL on bad arguments. */
pa_scheduler* pa_sched_create(pa_block_pool* pool, const pa_sched_config* cfg);
/* Releases the blocks of every request still held, then frees the object. */
void pa_sched_destroy(pa_scheduler* sched);

/* Queue a request at the back of the waiting queue. 1 <= prompt_len <=
 * max_model_len, req_id unused; `extra` (may be NULL) enters every block
 * hash of the request. */
pa_status pa_sched_add_request(pa_scheduler* sched, int64_t req_id, const int32_t* prompt,
                               int prompt_len, const uint8_t* extra, int extra_len);

/* Append a sampled token to a running request whose every token is
 * computed (it produced logits in the last step). PA_ERR_INVALID_ARG
 * otherwise, or when the request already holds max_model_len tokens. */
pa_status pa_sched_append_token(pa_scheduler* sched, int64_t req_id, int32_t token);

/* Remove a request, releasing its blocks last block first. */
pa_status pa_sched_finish(pa_scheduler* sched, int64_t req_id);

/* One scheduler step (see above). PA_ERR_WORKSPACE if an output capacity is
 * too small, in which case the scheduler state is unchanged. */
pa_status pa_sched_step(pa_scheduler* sched, pa_sched_output* out);

int pa_sched_num_running(const pa_scheduler* sched);
int pa_sched_num_waiting(const pa_scheduler* sched);

/* State of one request: computed tokens, total tokens, prompt length, blocks
 * held and whether it is running (1) or waiting (0). Unknown id:
 * PA_ERR_INVALID_ARG. Any output pointer may be NULL. */
pa_status pa_sched_request_state(const pa_scheduler* sched, int64_t req_id, int* num_computed,
                                 int* num_tokens, int* prompt_len, int* num_blocks,
                                 int* running);

/* Copy a request's block ids into out[0..max); returns how many it holds. */
int pa_sched_request_blocks(const pa_scheduler* sched, int64_t req_id, int32_t* out, int max);

#ifdef __cplusplus
}
#endif

#endif /* PA_HOST_H */
