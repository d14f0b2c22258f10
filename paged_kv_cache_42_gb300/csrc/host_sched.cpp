// Token-budget scheduler step and the batch metadata it emits ("Deep Dive -
// vLLM", "The V1 scheduler: one token budget"; "vLLM v1 Deep Dive: How
// LLM(...) and the Server Boot and Generate", Part 3 "Step 3 - Scheduler
// iteration"; "vLLM: An Exhaustive Technical Study for Kernel Engineers", 2.2
// "The V1 scheduler & continuous batching").
//
// There is no prefill/decode flag: each request has tokens (prompt plus
// sampled outputs) and a count of tokens whose KV is computed, and a step
// grants each scheduled request part of the difference under one budget.
// The step's output is exactly what pa_write_kv and pa_attention take:
// query_start_loc, seq_lens, block tables and the slot of every new token.
#include <algorithm>
#include <deque>
#include <memory>
#include <new>

#include "host_internal.h"

using pa_host::Hash;

namespace {

// The fields a step reads for every request come first (the first two
// cache lines of the 64-byte aligned object); the hashes and extra keys,
// touched only when a block fills or a request arrives, last.
struct alignas(64) Req {
  int64_t id = 0;
  std::vector<int32_t> tokens;  // prompt, then sampled tokens
  std::vector<int> blocks;      // pool indices, logical block order
  std::vector<int32_t> ids;     // the same blocks' physical ids (block-table rows)
  int num_computed = 0;
  int prompt_len = 0;
  int num_registered = 0;       // leading blocks already registered or hit
  // copies of tokens.back() and ids.back(), which a decode's metadata needs
  // every step (read here, they cost no access to either array)
  int32_t last_token = 0, last_id = -1;
  // identity of the block list: the request (serial, never reused) and how
  // often its blocks were released; within one (serial, epoch) the list only
  // grows at its end
  uint32_t epoch = 0;
  uint64_t serial = 0;
  bool running = false;
  std::vector<Hash> hashes;     // chained hashes of the first full blocks
  int hashes_algo = PA_HASH_SHA256;  // the algorithm they were taken with
  std::vector<uint8_t> extra;   // extra hash keys
};

// What a block-table row was last written from.
struct RowSrc {
  uint64_t serial;
  uint32_t epoch;
  int nb;  // blocks written; -1 after them
};

}  // namespace

struct pa_scheduler {
  pa_block_pool* pool = nullptr;
  pa_sched_config cfg{};
  std::unordered_map<int64_t, std::unique_ptr<Req>> reqs;
  std::vector<Req*> running;
  std::deque<Req*> waiting;
  uint64_t next_serial = 1;
  // What the last step left in the caller's block table: its address and
  // stride, and per row the block list it was written from.
  const int32_t* bt_ptr = nullptr;
  int bt_stride = 0;
  std::vector<RowSrc> bt_rows;
  // a step's scheduled list and one admission's prefix hits, kept between
  // steps so that their storage is reused
  std::vector<std::pair<Req*, int>> sched;
  std::vector<int> hits;

  int blocks_for(int tokens) const { return (tokens + pool->block_size - 1) / pool->block_size; }

  // Chained hashes of the request's first n full blocks (tokens only grow,
  // so hashes once computed stay valid, across preemption too - unless the
  // pool's algorithm changed, which it can only while no block holds one).
  void ensure_hashes(Req* r, int n) {
    const int bs = pool->block_size;
    if (r->hashes_algo != pool->hash_algo) {
      r->hashes.clear();
      r->hashes_algo = pool->hash_algo;
    }
    while ((int)r->hashes.size() < n) {
      const int b = (int)r->hashes.size();
      r->hashes.push_back(pa_host::block_hash(pool->hash_algo, b ? &r->hashes[b - 1] : nullptr,
                                              r->tokens.data() + (size_t)b * bs, bs,
                                              r->extra.data(), (int)r->extra.size()));
    }
  }

  void add_block(Req* r, int i) {
    r->blocks.push_back(i);
    r->ids.push_back(pool->id[i]);
    r->last_id = pool->id[i];
  }

  void release_blocks(Req* r) {
    for (auto it = r->blocks.rbegin(); it != r->blocks.rend(); ++it) pool->release(*it);
    r->blocks.clear();
    r->ids.clear();
    ++r->epoch;
    r->num_registered = 0;
  }

  // Recompute-style preemption: the KV is dropped (its full blocks stay in
  // the prefix cache while free) and the request waits at the front.
  void preempt(Req* r) {
    release_blocks(r);
    r->num_computed = 0;
    r->running = false;
    waiting.push_front(r);
  }

  void register_full_blocks(Req* r) {
    const int full = std::min(r->num_computed / pool->block_size, (int)r->blocks.size());
    if (full <= r->num_registered) return;
    ensure_hashes(r, full);
    for (int b = r->num_registered; b < full; ++b) {
      const int i = r->blocks[b];
      if (!pool->has_hash[i]) pool->insert(r->hashes[b], i);  // a present digest stays put
    }
    r->num_registered = full;
  }
};

extern "C" {

pa_scheduler* pa_sched_create(pa_block_pool* pool, const pa_sched_config* cfg) {
  if (!pool || !cfg || cfg->token_budget <= 0 || cfg->max_model_len <= 0) return nullptr;
  const long long need = ((long long)cfg->max_model_len + pool->block_size - 1) / pool->block_size;
  if (cfg->max_blocks_per_req < need) return nullptr;
  pa_scheduler* s = new (std::nothrow) pa_scheduler();
  if (!s) return nullptr;
  s->pool = pool;
  s->cfg = *cfg;
  return s;
}

void pa_sched_destroy(pa_scheduler* s) {
  if (!s) return;
  for (Req* r : s->running) s->release_blocks(r);
  delete s;
}

pa_status pa_sched_add_request(pa_scheduler* s, int64_t req_id, const int32_t* prompt,
                               int prompt_len, const uint8_t* extra, int extra_len) {
  if (!s || !prompt || prompt_len <= 0 || prompt_len > s->cfg.max_model_len || extra_len < 0 ||
      (extra_len > 0 && !extra) || s->reqs.count(req_id))
    return PA_ERR_INVALID_ARG;
  try {
    auto r = std::make_unique<Req>();
    r->id = req_id;
    r->serial = s->next_serial++;
    r->tokens.assign(prompt, prompt + prompt_len);
    r->last_token = prompt[prompt_len - 1];
    r->tokens.reserve(s->cfg.max_model_len);
    r->prompt_len = prompt_len;
    if (extra_len) r->extra.assign(extra, extra + extra_len);
    // The prompt's full blocks are hashed once, when the request arrives,
    // so a step only hashes blocks that its own tokens complete.
    if (s->cfg.enable_prefix_caching) s->ensure_hashes(r.get(), prompt_len / s->pool->block_size);
    s->waiting.push_back(r.get());
    s->reqs.emplace(req_id, std::move(r));
  } catch (...) {
    return PA_ERR_INVALID_ARG;
  }
  return PA_OK;
}

pa_status pa_sched_append_token(pa_scheduler* s, int64_t req_id, int32_t token) {
  if (!s) return PA_ERR_INVALID_ARG;
  auto it = s->reqs.find(req_id);
  if (it == s->reqs.end()) return PA_ERR_INVALID_ARG;
  Req* r = it->second.get();
  if (!r->running || r->num_computed != (int)r->tokens.size() ||
      (int)r->tokens.size() >= s->cfg.max_model_len)
    return PA_ERR_INVALID_ARG;
  r->tokens.push_back(token);
  r->last_token = token;
  return PA_OK;
}

pa_status pa_sched_finish(pa_scheduler* s, int64_t req_id) {
  if (!s) return PA_ERR_INVALID_ARG;
  auto it = s->reqs.find(req_id);
  if (it == s->reqs.end()) return PA_ERR_INVALID_ARG;
  Req* r = it->second.get();
  if (r->running) {
    s->running.erase(std::find(s->running.begin(), s->running.end(), r));
    s->release_blocks(r);
  } else {
    s->waiting.erase(std::find(s->waiting.begin(), s->waiting.end(), r));
  }
  s->reqs.erase(it);
  return PA_OK;
}

pa_status pa_sched_step(pa_scheduler* s, pa_sched_output* out) {
  if (!s || !out) return PA_ERR_INVALID_ARG;
  const pa_sched_config& c = s->cfg;
  pa_block_pool* pool = s->pool;
  const int bs = pool->block_size;
  // Capacities, checked before any state changes: at most token_budget
  // tokens, one request per granted token, one preemption per running one.
  const long long live = (long long)s->running.size() + (long long)s->waiting.size();
  if (out->max_tokens < c.token_budget || out->max_reqs < std::min<long long>(live, c.token_budget) ||
      out->max_preempted < (int)s->running.size())
    return PA_ERR_WORKSPACE;
  if (!out->req_ids || !out->num_scheduled || !out->num_computed || !out->query_start_loc ||
      !out->seq_lens || !out->block_tables || !out->slot_mapping || !out->positions ||
      !out->input_tokens || (out->max_preempted > 0 && !out->preempted_ids))
    return PA_ERR_INVALID_ARG;

  int budget = c.token_budget;
  std::vector<std::pair<Req*, int>>& sched = s->sched;
  sched.clear();
  int num_preempted = 0;

  // Pass 1: running requests, in order.
  for (size_t i = 0; i < s->running.size() && budget > 0;) {
    Req* r = s->running[i];
    int n = (int)r->tokens.size() - r->num_computed;
    if (c.long_prefill_threshold > 0 && n > c.long_prefill_threshold) n = c.long_prefill_threshold;
    n = std::min(n, budget);
    n = std::min(n, c.max_model_len - r->num_computed);
    if (n <= 0) {
      ++i;
      continue;
    }
    const int need = s->blocks_for(r->num_computed + n) - (int)r->blocks.size();
    bool self_preempted = false;
    while (need > pool->num_free) {
      Req* victim = s->running.back();
      s->running.pop_back();
      s->preempt(victim);
      out->preempted_ids[num_preempted++] = victim->id;
      if (victim == r) {
        self_preempted = true;
        break;
      }
    }
    if (self_preempted) break;
    for (int k = 0; k < need; ++k) s->add_block(r, pool->pop_front_for_use());
    sched.emplace_back(r, n);
    budget -= n;
    ++i;
  }

  // Pass 2: admit waiting requests (not in a step that had to preempt).
  while (num_preempted == 0 && !s->waiting.empty() && budget > 0) {
    if (c.max_running > 0 && (int)s->running.size() >= c.max_running) break;
    Req* r = s->waiting.front();
    std::vector<int>& hits = s->hits;
    hits.clear();
    if (c.enable_prefix_caching) {
      const int max_hit = ((int)r->tokens.size() - 1) / bs;
      s->ensure_hashes(r, max_hit);
      for (int b = 0; b < max_hit; ++b) {
        const int i = pool->lookup(r->hashes[b]);
        if (i < 0) break;
        hits.push_back(i);
      }
    }
    const int cached = (int)hits.size() * bs;
    int n = (int)r->tokens.size() - cached;
    if (c.long_prefill_threshold > 0 && n > c.long_prefill_threshold) n = c.long_prefill_threshold;
    if (!c.enable_chunked_prefill && n > budget) break;
    n = std::min(n, budget);
    const int need = s->blocks_for(cached + n) - (int)hits.size();
    int evictable = 0;  // free cached blocks that a hit takes out of the queue
    for (int h : hits) evictable += pool->ref[h] == 0;
    if (need + evictable > pool->num_free) break;
    for (int h : hits) {
      pool->acquire(h);
      s->add_block(r, h);
    }
    r->num_registered = (int)hits.size();
    for (int k = 0; k < need; ++k) s->add_block(r, pool->pop_front_for_use());
    r->num_computed = cached;
    r->running = true;
    s->waiting.pop_front();
    s->running.push_back(r);
    sched.emplace_back(r, n);
    budget -= n;
  }

  // Emit the batch metadata, then advance the planned state.
  int stride = 1;
  for (auto& e : sched) stride = std::max(stride, (int)e.first->blocks.size());
  if (out->block_tables_retained) stride = c.max_blocks_per_req;  // a fixed row layout
  const bool keep = out->block_tables_retained && s->bt_ptr == out->block_tables &&
                    s->bt_stride == stride;
  const size_t kept_rows = keep ? s->bt_rows.size() : 0;
  s->bt_rows.resize(sched.size());
  int t = 0, max_q = 0, max_s = 0, decodes = 0;
  int ctx_reqs = 0, ctx_toks = 0, gen_reqs = 0, gen_toks = 0;
  for (size_t k = 0; k < sched.size(); ++k) {
    Req* r = sched[k].first;
    const int n = sched[k].second, ctx = r->num_computed;
    out->req_ids[k] = r->id;
    out->num_scheduled[k] = n;
    out->num_computed[k] = ctx;
    out->query_start_loc[k] = t;
    out->seq_lens[k] = ctx + n;
    int32_t* row = out->block_tables + (size_t)k * stride;
    const int nb = (int)r->ids.size();
    RowSrc& src = s->bt_rows[k];
    if (k < kept_rows && src.serial == r->serial && src.epoch == r->epoch && src.nb <= nb) {
      // the same list, grown at its end: the row holds its first src.nb ids
      // and -1 after them
      std::memcpy(row + src.nb, r->ids.data() + src.nb, (size_t)(nb - src.nb) * sizeof(int32_t));
    } else {
      std::memcpy(row, r->ids.data(), (size_t)nb * sizeof(int32_t));
      std::memset(row + nb, 0xFF, (size_t)(stride - nb) * sizeof(int32_t));  // -1 past the blocks
    }
    src = RowSrc{r->serial, r->epoch, nb};
    if (n == 1 && ctx + 1 == (int)r->tokens.size()) {  // a decode: the newest token
      out->positions[t] = ctx;
      out->input_tokens[t] = r->last_token;
      out->slot_mapping[t] = (int64_t)r->last_id * bs + ctx % bs;  // its block is the last
    } else {
      for (int j = 0; j < n; ++j) {
        const int p = ctx + j;
        out->positions[t + j] = p;
        out->input_tokens[t + j] = r->tokens[p];
        out->slot_mapping[t + j] = (int64_t)r->ids[p / bs] * bs + p % bs;
      }
    }
    t += n;
    max_q = std::max(max_q, n);
    max_s = std::max(max_s, ctx + n);
    decodes += (n == 1 && ctx >= r->prompt_len);
    if (ctx < r->prompt_len) {
      ++ctx_reqs;
      ctx_toks += n;
    } else {
      ++gen_reqs;
      gen_toks += n;
    }
  }
  out->query_start_loc[sched.size()] = t;
  out->num_reqs = (int)sched.size();
  out->num_tokens = t;
  out->num_preempted = num_preempted;
  out->max_query_len = max_q;
  out->max_seq_len = max_s;
  out->block_table_stride = stride;
  out->num_decode_reqs = decodes;
  out->num_context_reqs = ctx_reqs;
  out->num_context_tokens = ctx_toks;
  out->num_generation_reqs = gen_reqs;
  out->num_generation_tokens = gen_toks;
  s->bt_ptr = out->block_tables;
  s->bt_stride = stride;
  for (auto& e : sched) {
    e.first->num_computed += e.second;
    if (c.enable_prefix_caching) s->register_full_blocks(e.first);
  }
  return PA_OK;
}

int pa_sched_num_running(const pa_scheduler* s) { return s ? (int)s->running.size() : 0; }
int pa_sched_num_waiting(const pa_scheduler* s) { return s ? (int)s->waiting.size() : 0; }

pa_status pa_sched_request_state(const pa_scheduler* s, int64_t req_id, int* num_computed,
                                 int* num_tokens, int* prompt_len, int* num_blocks,
                                 int* running) {
  if (!s) return PA_ERR_INVALID_ARG;
  auto it = s->reqs.find(req_id);
  if (it == s->reqs.end()) return PA_ERR_INVALID_ARG;
  const Req* r = it->second.get();
  if (num_computed) *num_computed = r->num_computed;
  if (num_tokens) *num_tokens = (int)r->tokens.size();
  if (prompt_len) *prompt_len = r->prompt_len;
  if (num_blocks) *num_blocks = (int)r->blocks.size();
  if (running) *running = r->running ? 1 : 0;
  return PA_OK;
}

int pa_sched_request_blocks(const pa_scheduler* s, int64_t req_id, int32_t* out, int max) {
  if (!s) return PA_ERR_INVALID_ARG;
  auto it = s->reqs.find(req_id);
  if (it == s->reqs.end()) return PA_ERR_INVALID_ARG;
  const Req* r = it->second.get();
  for (int b = 0; b < (int)r->ids.size() && b < max; ++b)
    if (out) out[b] = r->ids[b];
  return (int)r->blocks.size();
}

}  // extern "C"
