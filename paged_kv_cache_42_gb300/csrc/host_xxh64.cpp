// XXH64, the 64-bit member of the xxHash family (Yann Collet), written from
// the algorithm's published description: the fast non-cryptographic option
// for the prefix cache's chained block hash ("Deep Dive - vLLM", "Block pool,
// prefix cache, and eviction": a faster xxhash variant is a flag away;
// "Automatic Prefix Caching": the hash algorithm is selectable).
//
// Outline. Five 64-bit odd constants P1..P5. An input of at least 32 bytes
// runs four accumulators over its 32-byte stripes (lane k of a stripe feeds
// accumulator k through the round acc = rotl(acc + lane * P2, 31) * P1),
// then folds them into one value and merges each accumulator in again;
// shorter inputs start from seed + P5. The length is added, the remaining
// 8-byte words, one 4-byte word and single bytes are mixed in, and a final
// avalanche of shifts and multiplies spreads every input bit over the
// result. Words are read little endian, whatever the host's byte order.
#include <cstring>

#include "host_internal.h"

namespace pa_host {
namespace {

constexpr uint64_t P1 = 0x9E3779B185EBCA87ull;
constexpr uint64_t P2 = 0xC2B2AE3D27D4EB4Full;
constexpr uint64_t P3 = 0x165667B19E3779F9ull;
constexpr uint64_t P4 = 0x85EBCA77C2B2AE63ull;
constexpr uint64_t P5 = 0x27D4EB2F165667C5ull;

inline uint64_t rotl(uint64_t x, int r) { return (x << r) | (x >> (64 - r)); }

inline uint64_t le64(const uint8_t* p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}

inline uint32_t le32(const uint8_t* p) {
  return (uint32_t)p[0] | (uint32_t)p[1] << 8 | (uint32_t)p[2] << 16 | (uint32_t)p[3] << 24;
}

inline uint64_t round(uint64_t acc, uint64_t lane) { return rotl(acc + lane * P2, 31) * P1; }

inline uint64_t merge(uint64_t h, uint64_t acc) { return (h ^ round(0, acc)) * P1 + P4; }

}  // namespace

Xxh64::Xxh64(uint64_t seed) : seed_(seed) {
  v_[0] = seed + P1 + P2;
  v_[1] = seed + P2;
  v_[2] = seed;
  v_[3] = seed - P1;
}

void Xxh64::update(const uint8_t* p, size_t n) {
  total_ += n;
  if (buf_len_ + n < 32) {  // not a whole stripe yet
    if (n) std::memcpy(buf_ + buf_len_, p, n);
    buf_len_ += n;
    return;
  }
  if (buf_len_) {  // complete the carried stripe
    const size_t take = 32 - buf_len_;
    std::memcpy(buf_ + buf_len_, p, take);
    for (int k = 0; k < 4; ++k) v_[k] = round(v_[k], le64(buf_ + 8 * k));
    p += take;
    n -= take;
    buf_len_ = 0;
  }
  for (; n >= 32; p += 32, n -= 32)
    for (int k = 0; k < 4; ++k) v_[k] = round(v_[k], le64(p + 8 * k));
  if (n) std::memcpy(buf_, p, n);
  buf_len_ = n;
}

uint64_t Xxh64::digest() const {
  uint64_t h;
  if (total_ >= 32) {
    h = rotl(v_[0], 1) + rotl(v_[1], 7) + rotl(v_[2], 12) + rotl(v_[3], 18);
    for (int k = 0; k < 4; ++k) h = merge(h, v_[k]);
  } else {
    h = seed_ + P5;
  }
  h += total_;
  const uint8_t* p = buf_;
  const uint8_t* const end = buf_ + buf_len_;
  for (; end - p >= 8; p += 8) h = rotl(h ^ round(0, le64(p)), 27) * P1 + P4;
  if (end - p >= 4) {
    h = rotl(h ^ (uint64_t)le32(p) * P1, 23) * P2 + P3;
    p += 4;
  }
  for (; p < end; ++p) h = rotl(h ^ (uint64_t)*p * P5, 11) * P1;
  h ^= h >> 33;
  h *= P2;
  h ^= h >> 29;
  h *= P3;
  h ^= h >> 32;
  return h;
}

uint64_t xxh64(const uint8_t* p, size_t n, uint64_t seed) {
  Xxh64 x(seed);
  x.update(p, n);
  return x.digest();
}

}  // namespace pa_host

extern "C" uint64_t pa_xxh64(const uint8_t* data, size_t len, uint64_t seed) {
  return pa_host::xxh64(len ? data : nullptr, len, seed);
}
