// Physical block pool: reference counts, the LRU free queue and the
// hash -> block map of the prefix cache ("Deep Dive - vLLM", "Block pool,
// prefix cache, and eviction"; "Inside the vLLM Engine", "The pool, the
// queue, and the hash"; "vLLM: An Exhaustive Technical Study for Kernel
// Engineers", 2.3 "Automatic prefix caching & KV reuse").
//
// Blocks live in dense arrays indexed 0..n-1; the physical id is a label kept
// beside them (the pages' examples use ids such as 12, 41, 73, 90). The free
// queue is an intrusive doubly linked list over those indices, so allocation,
// release and a prefix hit on a free block are all O(1).
#include <new>

#include "host_internal.h"

using pa_host::Hash;

void pa_block_pool::push_back(int i) {
  prev[i] = tail;
  next[i] = -1;
  if (tail >= 0) next[tail] = i; else head = i;
  tail = i;
  in_free[i] = 1;
  ++num_free;
}

void pa_block_pool::push_front(int i) {
  next[i] = head;
  prev[i] = -1;
  if (head >= 0) prev[head] = i; else tail = i;
  head = i;
  in_free[i] = 1;
  ++num_free;
}

void pa_block_pool::unlink(int i) {
  if (prev[i] >= 0) next[prev[i]] = next[i]; else head = next[i];
  if (next[i] >= 0) prev[next[i]] = prev[i]; else tail = prev[i];
  prev[i] = next[i] = -1;
  in_free[i] = 0;
  --num_free;
}

int pa_block_pool::lookup(const Hash& h) const {
  const uint32_t tag = tag_of(h);
  for (size_t s = tag & mask;; s = (s + 1) & mask) {
    const Slot e = table[s];
    if (e.block < 0) return -1;
    if (e.tag == tag && hash[e.block] == h) return e.block;
  }
}

bool pa_block_pool::insert(const Hash& h, int i) {
  const uint32_t tag = tag_of(h);
  size_t s = tag & mask;
  for (; table[s].block >= 0; s = (s + 1) & mask)
    if (table[s].tag == tag && hash[table[s].block] == h) return false;  // first block keeps it
  table[s] = Slot{i, tag};
  hash[i] = h;
  has_hash[i] = 1;
  return true;
}

void pa_block_pool::drop_hash(int i) {
  if (!has_hash[i]) return;
  size_t hole = tag_of(hash[i]) & mask;
  while (table[hole].block != i) hole = (hole + 1) & mask;
  // Backward-shift deletion: walk the run after the hole and move back every
  // entry whose home slot does not lie strictly between the hole and it, so
  // no probe sequence crosses an empty slot before reaching its key.
  for (size_t t = (hole + 1) & mask; table[t].block >= 0; t = (t + 1) & mask) {
    const size_t home = table[t].tag & mask;
    if (((t - home) & mask) >= ((t - hole) & mask)) {
      table[hole] = table[t];
      hole = t;
    }
  }
  table[hole] = Slot{-1, 0};
  has_hash[i] = 0;
}

int pa_block_pool::pop_front_for_use() {
  const int i = head;
  unlink(i);
  drop_hash(i);  // the storage is about to be overwritten
  ref[i] = 1;
  return i;
}

void pa_block_pool::release(int i) {
  if (--ref[i] == 0) {
    if (has_hash[i]) push_back(i);  // may still be rescued by a prefix hit
    else push_front(i);             // nothing to keep: reuse it first
  }
}

void pa_block_pool::acquire(int i) {
  if (ref[i] == 0) unlink(i);
  ++ref[i];
}

extern "C" {

pa_block_pool* pa_pool_create(int num_blocks, int block_size, const int32_t* ids) {
  if (num_blocks < 0 || block_size <= 0) return nullptr;
  pa_block_pool* p = new (std::nothrow) pa_block_pool();
  if (!p) return nullptr;
  try {
    p->block_size = block_size;
    p->id.resize(num_blocks);
    p->ref.assign(num_blocks, 0);
    p->prev.assign(num_blocks, -1);
    p->next.assign(num_blocks, -1);
    p->in_free.assign(num_blocks, 0);
    p->has_hash.assign(num_blocks, 0);
    p->uses.assign(num_blocks, 0);
    p->hash.resize(num_blocks);
    size_t slots = 2;
    while (slots < 2 * (size_t)num_blocks) slots *= 2;
    p->table.assign(slots, pa_block_pool::Slot{-1, 0});
    p->mask = slots - 1;
    p->index.reserve(num_blocks);
    for (int i = 0; i < num_blocks; ++i) {
      const int32_t pid = ids ? ids[i] : i;
      if (pid < 0 || !p->index.emplace(pid, i).second) {  // negative or repeated id
        delete p;
        return nullptr;
      }
      p->id[i] = pid;
      p->push_back(i);
    }
  } catch (...) {
    delete p;
    return nullptr;
  }
  return p;
}

void pa_pool_destroy(pa_block_pool* pool) { delete pool; }

int pa_pool_num_blocks(const pa_block_pool* pool) { return pool ? (int)pool->id.size() : 0; }
int pa_pool_block_size(const pa_block_pool* pool) { return pool ? pool->block_size : 0; }
int pa_pool_num_free(const pa_block_pool* pool) { return pool ? pool->num_free : 0; }

pa_status pa_pool_allocate(pa_block_pool* pool, int n, int32_t* out_ids) {
  if (!pool || n < 0 || (n > 0 && !out_ids)) return PA_ERR_INVALID_ARG;
  if (n > pool->num_free) return PA_ERR_BOUNDS;
  for (int k = 0; k < n; ++k) out_ids[k] = pool->id[pool->pop_front_for_use()];
  return PA_OK;
}

pa_status pa_pool_free(pa_block_pool* pool, const int32_t* ids, int n) {
  if (!pool || n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID_ARG;
  // Validate everything first (an id may repeat, at most as often as the
  // block is referenced): nothing changes on error. The counts live in a
  // zeroed per-pool array and are put back to zero before returning.
  int k = 0;
  bool ok = true;
  for (; k < n; ++k) {
    const int i = pool->find(ids[k]);
    if (i < 0) {
      ok = false;
      break;
    }
    if (++pool->uses[i] > pool->ref[i]) {
      ++k;  // this one was counted
      ok = false;
      break;
    }
  }
  for (int j = 0; j < k; ++j) pool->uses[pool->find(ids[j])] = 0;
  if (!ok) return PA_ERR_INVALID_ARG;
  for (int j = n - 1; j >= 0; --j) pool->release(pool->find(ids[j]));
  return PA_OK;
}

pa_status pa_pool_touch(pa_block_pool* pool, const int32_t* ids, int n) {
  if (!pool || n < 0 || (n > 0 && !ids)) return PA_ERR_INVALID_ARG;
  for (int k = 0; k < n; ++k)
    if (pool->find(ids[k]) < 0) return PA_ERR_INVALID_ARG;
  for (int k = 0; k < n; ++k) pool->acquire(pool->find(ids[k]));
  return PA_OK;
}

pa_status pa_pool_cache_block(pa_block_pool* pool, int32_t id, const uint8_t hash[32]) {
  if (!pool || !hash) return PA_ERR_INVALID_ARG;
  const int i = pool->find(id);
  if (i < 0 || pool->ref[i] == 0 || pool->has_hash[i]) return PA_ERR_INVALID_ARG;
  Hash h;
  std::memcpy(h.data(), hash, 32);
  pool->insert(h, i);  // a digest already present stays with its first block
  return PA_OK;
}

int32_t pa_pool_lookup(const pa_block_pool* pool, const uint8_t hash[32]) {
  if (!pool || !hash) return -1;
  Hash h;
  std::memcpy(h.data(), hash, 32);
  const int i = pool->lookup(h);
  return i < 0 ? -1 : pool->id[i];
}

pa_status pa_pool_set_hash_algo(pa_block_pool* pool, int algo) {
  if (!pool || (algo != PA_HASH_SHA256 && algo != PA_HASH_XXH64)) return PA_ERR_INVALID_ARG;
  for (uint8_t h : pool->has_hash)
    if (h) return PA_ERR_INVALID_ARG;  // digests of one algorithm per table
  pool->hash_algo = algo;
  return PA_OK;
}

int pa_pool_hash_algo(const pa_block_pool* pool) { return pool ? pool->hash_algo : -1; }

int pa_pool_ref_count(const pa_block_pool* pool, int32_t id) {
  const int i = pool ? pool->find(id) : -1;
  return i < 0 ? -1 : pool->ref[i];
}

int pa_pool_is_cached(const pa_block_pool* pool, int32_t id) {
  const int i = pool ? pool->find(id) : -1;
  return i < 0 ? -1 : (int)pool->has_hash[i];
}

int pa_pool_free_queue(const pa_block_pool* pool, int32_t* out, int max) {
  if (!pool) return 0;
  int n = 0;
  for (int i = pool->head; i >= 0; i = pool->next[i], ++n)
    if (out && n < max) out[n] = pool->id[i];
  return n;
}

int pa_pool_find_cached_prefix(const pa_block_pool* pool, const int32_t* tokens, int num_tokens,
                               const uint8_t* extra, int extra_len, int32_t* out_ids,
                               int max_blocks) {
  if (!pool || num_tokens <= 0 || !tokens || extra_len < 0 || (extra_len > 0 && !extra) ||
      max_blocks < 0 || (max_blocks > 0 && !out_ids))
    return PA_ERR_INVALID_ARG;
  const int bs = pool->block_size;
  int limit = (num_tokens - 1) / bs;  // whole blocks within num_tokens - 1 tokens
  if (limit > max_blocks) limit = max_blocks;
  Hash parent;
  int hits = 0;
  for (int b = 0; b < limit; ++b) {
    parent = pa_host::block_hash(pool->hash_algo, b ? &parent : nullptr, tokens + (size_t)b * bs,
                                 bs, extra, extra_len);
    const int i = pool->lookup(parent);
    if (i < 0) break;  // a chained hash cannot match past a miss
    out_ids[hits++] = pool->id[i];
  }
  return hits * bs;
}

pa_status pa_reusable_tokens(int shared, int prompt_length, int block_size, int* out) {
  if (!out || block_size <= 0 || prompt_length <= 0 || shared < 0 || shared > prompt_length)
    return PA_ERR_INVALID_ARG;
  const int limit = shared < prompt_length - 1 ? shared : prompt_length - 1;
  *out = limit / block_size * block_size;
  return PA_OK;
}

}  // extern "C"
