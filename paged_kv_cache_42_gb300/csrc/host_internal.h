// Host-side runtime internals shared by the pool, hash and scheduler sources.
#pragma once

#include <array>
#include <cstddef>
#include <cstdint>
#include <cstring>
#include <unordered_map>
#include <vector>

#include "pa_host.h"

namespace pa_host {

using Hash = std::array<uint8_t, 32>;

struct HashKey {
  size_t operator()(const Hash& h) const {
    size_t v;
    std::memcpy(&v, h.data(), sizeof v);  // the digest is already uniform
    return v;
  }
};

// SHA-256 (FIPS 180-4), streaming.
class Sha256 {
 public:
  Sha256();
  void update(const uint8_t* data, size_t len);
  void final(uint8_t out[32]);

 private:
  void compress(const uint8_t block[64]);
  const uint32_t* k_;  // round constants
  uint32_t h_[8];
  uint8_t buf_[64];
  size_t buf_len_ = 0;
  uint64_t total_ = 0;
};

// Chained block hash: SHA-256(parent || tokens as int32 LE || extra).
Hash block_hash(const Hash* parent, const int32_t* tokens, int n, const uint8_t* extra,
                int extra_len);

}  // namespace pa_host

// The pool: blocks addressed by a dense index; the physical id is a label.
struct pa_block_pool {
  int block_size = 0;
  std::vector<int32_t> id;  // index -> physical id
  std::unordered_map<int32_t, int> index;
  std::vector<int> ref, prev, next;
  std::vector<uint8_t> in_free, has_hash;
  std::vector<pa_host::Hash> hash;
  std::unordered_map<pa_host::Hash, int, pa_host::HashKey> by_hash;
  int head = -1, tail = -1, num_free = 0;

  int find(int32_t pid) const {
    auto it = index.find(pid);
    return it == index.end() ? -1 : it->second;
  }
  void push_back(int i);
  void push_front(int i);
  void unlink(int i);
  void drop_hash(int i);
  // Internal forms used by the scheduler (indices, no validation).
  int pop_front_for_use();  // allocate one block: ref 1, hash dropped
  void release(int i);      // one reference; count 0 -> free queue
  void acquire(int i);      // one reference; leaves the free queue
};
