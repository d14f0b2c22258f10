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

// XXH64 (host_xxh64.cpp), streaming: whole 32-byte stripes go through the
// four accumulators as they arrive, a partial one is carried.
class Xxh64 {
 public:
  explicit Xxh64(uint64_t seed);
  void update(const uint8_t* data, size_t len);
  uint64_t digest() const;

 private:
  uint64_t v_[4];
  uint8_t buf_[32];
  size_t buf_len_ = 0;
  uint64_t total_ = 0;
  uint64_t seed_;
};
uint64_t xxh64(const uint8_t* p, size_t n, uint64_t seed);

// Chained block hash over parent || tokens as int32 LE || extra: SHA-256
// (PA_HASH_SHA256), or XXH64 in the first 8 bytes, little endian, and zeros
// after them (PA_HASH_XXH64).
Hash block_hash(int algo, const Hash* parent, const int32_t* tokens, int n,
                const uint8_t* extra, int extra_len);

}  // namespace pa_host

// The pool: blocks addressed by a dense index; the physical id is a label.
struct pa_block_pool {
  int block_size = 0;
  std::vector<int32_t> id;  // index -> physical id
  std::unordered_map<int32_t, int> index;
  std::vector<int> ref, prev, next;
  std::vector<uint8_t> in_free, has_hash;
  std::vector<int> uses;  // all zero between calls: pa_pool_free's per-block count
  std::vector<pa_host::Hash> hash;
  // The prefix cache's hash -> block map: open addressing with linear probing
  // over a power-of-two table at least twice the block count (so a probe
  // always reaches an empty slot). A slot holds a block index (-1: empty) and
  // the low 32 bits of its digest's first word, which give the home slot and
  // screen a probe before it reads the block's full digest. has_hash[i] is
  // set exactly while block i is in the table. No allocation after creation.
  struct Slot {
    int32_t block;
    uint32_t tag;
  };
  std::vector<Slot> table;
  size_t mask = 0;
  int head = -1, tail = -1, num_free = 0;
  int hash_algo = PA_HASH_SHA256;  // of every digest in the table

  int find(int32_t pid) const {
    auto it = index.find(pid);
    return it == index.end() ? -1 : it->second;
  }
  void push_back(int i);
  void push_front(int i);
  void unlink(int i);
  static uint32_t tag_of(const pa_host::Hash& h) { return (uint32_t)pa_host::HashKey()(h); }
  int lookup(const pa_host::Hash& h) const;   // block index holding h, or -1
  bool insert(const pa_host::Hash& h, int i);  // false (nothing changed) if h is present
  void drop_hash(int i);                       // take block i's digest out, if it has one
  // Internal forms used by the scheduler (indices, no validation).
  int pop_front_for_use();  // allocate one block: ref 1, hash dropped
  void release(int i);      // one reference; count 0 -> free queue
  void acquire(int i);      // one reference; leaves the free queue
};
