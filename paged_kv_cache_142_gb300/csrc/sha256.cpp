// SHA-256 (FIPS 180-4, sections 4.1.2, 4.2.2, 5.1.1, 5.3.3 and 6.2), the
// default block-key hash of automatic prefix caching ("llm-kv-cache-02-
// serving-engine-kv", section 4 "프리픽스 캐시": a block's key hashes the
// previous block's key, the block's token ids and the request's extras; the
// default hash is sha256).
//
// The round constants K and the initial hash value H(0) are the first 32
// bits of the fractional parts of the cube roots of the first 64 primes and
// of the square roots of the first 8 primes (FIPS 180-4, 4.2.2 and 5.3.3);
// they are derived here with exact integer roots instead of being listed.
#include "sha256.h"

#include <cstring>

namespace pa {
namespace {

using u128 = unsigned __int128;

// floor(p^(1/k) * 2^32) mod 2^32 for k = 2 or 3, by bisection on integers
uint32_t frac_root_bits(uint32_t p, int k) {
  const u128 target = static_cast<u128>(p) << (32 * k);  // p * 2^(32k)
  uint64_t lo = 0, hi = uint64_t(1) << 40;                 // root < 2^40 for p < 2^8
  while (hi - lo > 1) {
    const uint64_t mid = lo + (hi - lo) / 2;
    u128 v = mid;
    for (int i = 1; i < k; ++i) v *= mid;
    if (v <= target) lo = mid;
    else hi = mid;
  }
  return static_cast<uint32_t>(lo);
}

struct Constants {
  uint32_t k[64];
  uint32_t h0[8];
  Constants() {
    int n = 0;
    for (uint32_t c = 2; n < 64; ++c) {
      bool prime = true;
      for (uint32_t d = 2; d * d <= c; ++d)
        if (c % d == 0) {
          prime = false;
          break;
        }
      if (!prime) continue;
      k[n] = frac_root_bits(c, 3);
      if (n < 8) h0[n] = frac_root_bits(c, 2);
      ++n;
    }
  }
};

const Constants& constants() {
  static const Constants c;
  return c;
}

inline uint32_t rotr(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

void compress(uint32_t h[8], const uint8_t block[64], const uint32_t* k) {
  uint32_t w[64];
  for (int t = 0; t < 16; ++t)
    w[t] = (uint32_t(block[4 * t]) << 24) | (uint32_t(block[4 * t + 1]) << 16) |
           (uint32_t(block[4 * t + 2]) << 8) | uint32_t(block[4 * t + 3]);
  for (int t = 16; t < 64; ++t) {
    const uint32_t s0 = rotr(w[t - 15], 7) ^ rotr(w[t - 15], 18) ^ (w[t - 15] >> 3);
    const uint32_t s1 = rotr(w[t - 2], 17) ^ rotr(w[t - 2], 19) ^ (w[t - 2] >> 10);
    w[t] = s1 + w[t - 7] + s0 + w[t - 16];
  }
  uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
  for (int t = 0; t < 64; ++t) {
    const uint32_t big1 = rotr(e, 6) ^ rotr(e, 11) ^ rotr(e, 25);
    const uint32_t ch = (e & f) ^ (~e & g);
    const uint32_t t1 = hh + big1 + ch + k[t] + w[t];
    const uint32_t big0 = rotr(a, 2) ^ rotr(a, 13) ^ rotr(a, 22);
    const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
    const uint32_t t2 = big0 + maj;
    hh = g;
    g = f;
    f = e;
    e = d + t1;
    d = c;
    c = b;
    b = a;
    a = t1 + t2;
  }
  h[0] += a;
  h[1] += b;
  h[2] += c;
  h[3] += d;
  h[4] += e;
  h[5] += f;
  h[6] += g;
  h[7] += hh;
}

}  // namespace

Sha256::Sha256() {
  const Constants& c = constants();
  std::memcpy(h_, c.h0, sizeof(h_));
}

void Sha256::update(const void* data, size_t n) {
  const Constants& c = constants();
  const uint8_t* p = static_cast<const uint8_t*>(data);
  bytes_ += n;
  while (n > 0) {
    const size_t take = (64 - fill_) < n ? (64 - fill_) : n;
    std::memcpy(buf_ + fill_, p, take);
    fill_ += take;
    p += take;
    n -= take;
    if (fill_ == 64) {
      compress(h_, buf_, c.k);
      fill_ = 0;
    }
  }
}

void Sha256::finish(uint8_t out[32]) {
  // padding: a 1 bit, zeros to 56 mod 64 bytes, the message length in bits (big-endian)
  const uint64_t bits = bytes_ * 8;
  uint8_t pad[72] = {0x80};  // the 1 bit, then zeros up to 56 mod 64, then the length
  const size_t zeros = (fill_ < 56 ? 56 - fill_ : 120 - fill_) - 1;
  for (int i = 0; i < 8; ++i) pad[1 + zeros + i] = static_cast<uint8_t>(bits >> (56 - 8 * i));
  update(pad, 1 + zeros + 8);
  for (int i = 0; i < 8; ++i) {
    out[4 * i] = static_cast<uint8_t>(h_[i] >> 24);
    out[4 * i + 1] = static_cast<uint8_t>(h_[i] >> 16);
    out[4 * i + 2] = static_cast<uint8_t>(h_[i] >> 8);
    out[4 * i + 3] = static_cast<uint8_t>(h_[i]);
  }
}

}  // namespace pa

extern "C" pa_status pa_sha256(const void* data, size_t num_bytes, uint8_t digest[32]) {
  if ((!data && num_bytes) || !digest) return PA_ERR_INVALID_ARG;
  pa::Sha256 s;
  s.update(data, num_bytes);
  s.finish(digest);
  return PA_OK;
}
