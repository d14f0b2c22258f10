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

uint64_t xxh64(const uint8_t* p, size_t n, uint64_t seed) {
  const uint8_t* const end = p + n;
  uint64_t h;
  if (n >= 32) {
    uint64_t v1 = seed + P1 + P2, v2 = seed + P2, v3 = seed, v4 = seed - P1;
    for (; end - p >= 32; p += 32) {
      v1 = round(v1, le64(p));
      v2 = round(v2, le64(p + 8));
      v3 = round(v3, le64(p + 16));
      v4 = round(v4, le64(p + 24));
    }
    h = rotl(v1, 1) + rotl(v2, 7) + rotl(v3, 12) + rotl(v4, 18);
    h = merge(h, v1);
    h = merge(h, v2);
    h = merge(h, v3);
    h = merge(h, v4);
  } else {
    h = seed + P5;
  }
  h += (uint64_t)n;
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

}  // namespace pa_host

extern "C" uint64_t pa_xxh64(const uint8_t* data, size_t len, uint64_t seed) {
  return pa_host::xxh64(len ? data : nullptr, len, seed);
}
