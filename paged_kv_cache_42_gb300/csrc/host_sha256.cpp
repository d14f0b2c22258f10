// SHA-256 written from its definition in FIPS 180-4 (Secure Hash Standard),
// sections 4.1.2 (functions), 4.2.2 (constants), 5.1.1 (padding), 5.3.3
// (initial hash value) and 6.2.2 (computation), and the chained block hash
// built on it ("Deep Dive - vLLM", "Block pool, prefix cache, and eviction":
// a block's hash covers its parent's hash, its tokens and the extra keys;
// SHA-256 is the documented default).
//
// The round constants and the initial hash value are the leading 32 bits of
// the fractional parts of the cube roots of the first 64 primes and of the
// square roots of the first 8 primes (FIPS 180-4, 4.2.2 and 5.3.3). They are
// derived here from that definition with exact integer roots rather than
// typed in: floor(frac(root(p)) * 2^32) = floor(root(p * 2^(32k))) mod 2^32.
#include <algorithm>

#include "host_internal.h"

namespace pa_host {
namespace {

typedef unsigned __int128 u128;

u128 icbrt(u128 n) {  // largest x with x^3 <= n, n < 2^108
  u128 lo = 0, hi = (u128)1 << 36;
  while (hi - lo > 1) {
    u128 m = (lo + hi) / 2;
    if (m * m * m <= n) lo = m; else hi = m;
  }
  return lo;
}

u128 isqrt(u128 n) {  // largest x with x^2 <= n, n < 2^72
  u128 lo = 0, hi = (u128)1 << 36;
  while (hi - lo > 1) {
    u128 m = (lo + hi) / 2;
    if (m * m <= n) lo = m; else hi = m;
  }
  return lo;
}

struct Constants {
  uint32_t k[64];
  uint32_t h0[8];
  Constants() {
    int primes[64], n = 0;
    for (int c = 2; n < 64; ++c) {
      bool prime = true;
      for (int d = 2; d * d <= c; ++d)
        if (c % d == 0) { prime = false; break; }
      if (prime) primes[n++] = c;
    }
    for (int i = 0; i < 64; ++i) k[i] = (uint32_t)icbrt((u128)primes[i] << 96);
    for (int i = 0; i < 8; ++i) h0[i] = (uint32_t)isqrt((u128)primes[i] << 64);
  }
};

const Constants& constants() {
  static const Constants c;  // thread-safe one-time initialisation
  return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }
inline uint32_t ch(uint32_t x, uint32_t y, uint32_t z) { return (x & y) ^ (~x & z); }
inline uint32_t maj(uint32_t x, uint32_t y, uint32_t z) { return (x & y) ^ (x & z) ^ (y & z); }
inline uint32_t big_sigma0(uint32_t x) { return rotr(x, 2) ^ rotr(x, 13) ^ rotr(x, 22); }
inline uint32_t big_sigma1(uint32_t x) { return rotr(x, 6) ^ rotr(x, 11) ^ rotr(x, 25); }
inline uint32_t small_sigma0(uint32_t x) { return rotr(x, 7) ^ rotr(x, 18) ^ (x >> 3); }
inline uint32_t small_sigma1(uint32_t x) { return rotr(x, 17) ^ rotr(x, 19) ^ (x >> 10); }

}  // namespace

Sha256::Sha256() : k_(constants().k) { std::memcpy(h_, constants().h0, sizeof h_); }

void Sha256::compress(const uint8_t block[64]) {
  const uint32_t* K = k_;
  uint32_t w[64];
  for (int t = 0; t < 16; ++t)
    w[t] = (uint32_t)block[4 * t] << 24 | (uint32_t)block[4 * t + 1] << 16 |
           (uint32_t)block[4 * t + 2] << 8 | (uint32_t)block[4 * t + 3];
  for (int t = 16; t < 64; ++t)
    w[t] = small_sigma1(w[t - 2]) + w[t - 7] + small_sigma0(w[t - 15]) + w[t - 16];
  uint32_t a = h_[0], b = h_[1], c = h_[2], d = h_[3], e = h_[4], f = h_[5], g = h_[6],
           h = h_[7];
  for (int t = 0; t < 64; ++t) {
    const uint32_t t1 = h + big_sigma1(e) + ch(e, f, g) + K[t] + w[t];
    const uint32_t t2 = big_sigma0(a) + maj(a, b, c);
    h = g; g = f; f = e; e = d + t1;
    d = c; c = b; b = a; a = t1 + t2;
  }
  h_[0] += a; h_[1] += b; h_[2] += c; h_[3] += d;
  h_[4] += e; h_[5] += f; h_[6] += g; h_[7] += h;
}

void Sha256::update(const uint8_t* data, size_t len) {
  total_ += len;
  while (len > 0) {
    const size_t take = std::min(len, (size_t)64 - buf_len_);
    std::memcpy(buf_ + buf_len_, data, take);
    buf_len_ += take;
    data += take;
    len -= take;
    if (buf_len_ == 64) {
      compress(buf_);
      buf_len_ = 0;
    }
  }
}

void Sha256::final(uint8_t out[32]) {
  const uint64_t bits = total_ * 8;
  // Padding: one 1 bit, zeros up to 56 bytes mod 64, then the bit length.
  uint8_t pad[72] = {0x80};
  const size_t zeros = (buf_len_ < 56) ? 56 - buf_len_ : 120 - buf_len_;
  for (int i = 0; i < 8; ++i) pad[zeros + i] = (uint8_t)(bits >> (56 - 8 * i));
  const uint64_t keep = total_;
  update(pad, zeros + 8);
  total_ = keep;
  for (int i = 0; i < 8; ++i) {
    out[4 * i] = (uint8_t)(h_[i] >> 24);
    out[4 * i + 1] = (uint8_t)(h_[i] >> 16);
    out[4 * i + 2] = (uint8_t)(h_[i] >> 8);
    out[4 * i + 3] = (uint8_t)h_[i];
  }
}

Hash block_hash(int algo, const Hash* parent, const int32_t* tokens, int n,
                const uint8_t* extra, int extra_len) {
  static const Hash zero{};
  const uint8_t* const par = (parent ? *parent : zero).data();
  if (extra_len <= 0) extra = nullptr;
  if (algo == PA_HASH_XXH64) {
    Xxh64 x(0);
    x.update(par, 32);
    uint8_t le[256];  // tokens as int32 little endian, in chunks of 64
    for (int i0 = 0; i0 < n; i0 += 64) {
      const int m = std::min(64, n - i0);
      for (int i = 0; i < m; ++i) {
        const uint32_t v = (uint32_t)tokens[i0 + i];
        le[4 * i] = (uint8_t)v;
        le[4 * i + 1] = (uint8_t)(v >> 8);
        le[4 * i + 2] = (uint8_t)(v >> 16);
        le[4 * i + 3] = (uint8_t)(v >> 24);
      }
      x.update(le, (size_t)4 * m);
    }
    if (extra) x.update(extra, (size_t)extra_len);
    const uint64_t h = x.digest();
    Hash out{};
    for (int i = 0; i < 8; ++i) out[i] = (uint8_t)(h >> (8 * i));
    return out;
  }
  Sha256 s;
  s.update(par, 32);
  uint8_t le[256];  // tokens as int32 little endian, in chunks of 64
  for (int i0 = 0; i0 < n; i0 += 64) {
    const int m = std::min(64, n - i0);
    for (int i = 0; i < m; ++i) {
      const uint32_t v = (uint32_t)tokens[i0 + i];
      le[4 * i] = (uint8_t)v;
      le[4 * i + 1] = (uint8_t)(v >> 8);
      le[4 * i + 2] = (uint8_t)(v >> 16);
      le[4 * i + 3] = (uint8_t)(v >> 24);
    }
    s.update(le, (size_t)4 * m);
  }
  if (extra) s.update(extra, (size_t)extra_len);
  Hash out;
  s.final(out.data());
  return out;
}

}  // namespace pa_host

extern "C" void pa_sha256(const uint8_t* data, size_t len, uint8_t out[32]) {
  pa_host::Sha256 s;
  if (data && len) s.update(data, len);
  s.final(out);
}

extern "C" pa_status pa_block_hash_algo(int algo, const uint8_t parent[32],
                                        const int32_t* tokens, int num_tokens,
                                        const uint8_t* extra, int extra_len, uint8_t out[32]) {
  if (algo != PA_HASH_SHA256 && algo != PA_HASH_XXH64) return PA_ERR_INVALID_ARG;
  pa_host::Hash p;
  if (parent) std::memcpy(p.data(), parent, 32);
  const pa_host::Hash h = pa_host::block_hash(algo, parent ? &p : nullptr, tokens,
                                              num_tokens > 0 ? num_tokens : 0, extra, extra_len);
  std::memcpy(out, h.data(), 32);
  return PA_OK;
}

extern "C" void pa_block_hash(const uint8_t parent[32], const int32_t* tokens, int num_tokens,
                              const uint8_t* extra, int extra_len, uint8_t out[32]) {
  pa_block_hash_algo(PA_HASH_SHA256, parent, tokens, num_tokens, extra, extra_len, out);
}
