// Block digests for cache lookup, keyed per tenant (host code).
//
// ["HyperCache - Distributed KV-cache quantization and relative RoPE reuse",
//  "Core Design", item 1 "Dual-Mode Block Hashing": two deterministic 128-bit
//  BLAKE2b digests per token block, keyed by a per-tenant secret derived via
//  HMAC-SHA256, with a "public" namespace.]
//
// The two digests of block j (tokens as little-endian int32):
//   prefix  p_j = BLAKE2b-128(key K; p_{j-1} || tokens of block j), p_{-1} empty
//   content c_j = BLAKE2b-128(key K; tokens of block j)
// and K = HMAC-SHA256(master, "hc-tenant:" || tenant), or
// HMAC-SHA256(master, "hc-public") for the public namespace.
//
// BLAKE2b follows RFC 7693 (keyed, digest length 16), SHA-256 FIPS 180-4,
// HMAC RFC 2104.  Portable C++: no intrinsics, explicit little/big-endian
// byte handling.
#include <cstdint>
#include <cstring>

#include "hc.h"

namespace {

// ------------------------------------------------------------------ BLAKE2b
constexpr uint64_t kB2IV[8] = {0x6a09e667f3bcc908ULL, 0xbb67ae8584caa73bULL, 0x3c6ef372fe94f82bULL,
                               0xa54ff53a5f1d36f1ULL, 0x510e527fade682d1ULL, 0x9b05688c2b3e6c1fULL,
                               0x1f83d9abfb41bd6bULL, 0x5be0cd19137e2179ULL};
constexpr uint8_t kSigma[10][16] = {
    {0, 1, 2, 3, 4, 5, 6, 7, 8, 9, 10, 11, 12, 13, 14, 15},
    {14, 10, 4, 8, 9, 15, 13, 6, 1, 12, 0, 2, 11, 7, 5, 3},
    {11, 8, 12, 0, 5, 2, 15, 13, 10, 14, 3, 6, 7, 1, 9, 4},
    {7, 9, 3, 1, 13, 12, 11, 14, 2, 6, 5, 10, 4, 0, 15, 8},
    {9, 0, 5, 7, 2, 4, 10, 15, 14, 1, 11, 12, 6, 8, 3, 13},
    {2, 12, 6, 10, 0, 11, 8, 3, 4, 13, 7, 5, 15, 14, 1, 9},
    {12, 5, 1, 15, 14, 13, 4, 10, 0, 7, 6, 3, 9, 2, 8, 11},
    {13, 11, 7, 14, 12, 1, 3, 9, 5, 0, 15, 4, 8, 6, 2, 10},
    {6, 15, 14, 9, 11, 3, 0, 8, 12, 2, 13, 7, 1, 4, 10, 5},
    {10, 2, 8, 4, 7, 6, 1, 5, 15, 11, 9, 14, 3, 12, 13, 0}};

inline uint64_t rotr64(uint64_t x, int n) { return (x >> n) | (x << (64 - n)); }

inline uint64_t load_le64(const uint8_t* p) {
  uint64_t v = 0;
  for (int i = 7; i >= 0; --i) v = (v << 8) | p[i];
  return v;
}

struct Blake2b {
  uint64_t h[8];
  uint64_t t = 0;         // bytes compressed so far (inputs here stay far below 2^64)
  uint8_t buf[128];
  size_t fill = 0;        // bytes waiting in buf
  size_t out_len = 16;

  void compress(const uint8_t* block, bool last) {
    uint64_t m[16], v[16];
    for (int i = 0; i < 16; ++i) m[i] = load_le64(block + 8 * i);
    for (int i = 0; i < 8; ++i) {
      v[i] = h[i];
      v[i + 8] = kB2IV[i];
    }
    v[12] ^= t;  // low word of the byte counter; the high word stays 0
    if (last) v[14] = ~v[14];
    auto g = [&](int a, int b, int c, int d, uint64_t x, uint64_t y) {
      v[a] = v[a] + v[b] + x;
      v[d] = rotr64(v[d] ^ v[a], 32);
      v[c] = v[c] + v[d];
      v[b] = rotr64(v[b] ^ v[c], 24);
      v[a] = v[a] + v[b] + y;
      v[d] = rotr64(v[d] ^ v[a], 16);
      v[c] = v[c] + v[d];
      v[b] = rotr64(v[b] ^ v[c], 63);
    };
    for (int r = 0; r < 12; ++r) {
      const uint8_t* s = kSigma[r % 10];
      g(0, 4, 8, 12, m[s[0]], m[s[1]]);
      g(1, 5, 9, 13, m[s[2]], m[s[3]]);
      g(2, 6, 10, 14, m[s[4]], m[s[5]]);
      g(3, 7, 11, 15, m[s[6]], m[s[7]]);
      g(0, 5, 10, 15, m[s[8]], m[s[9]]);
      g(1, 6, 11, 12, m[s[10]], m[s[11]]);
      g(2, 7, 8, 13, m[s[12]], m[s[13]]);
      g(3, 4, 9, 14, m[s[14]], m[s[15]]);
    }
    for (int i = 0; i < 8; ++i) h[i] ^= v[i] ^ v[i + 8];
  }

  void init(const uint8_t* key, size_t key_len, size_t digest_len) {
    out_len = digest_len;
    for (int i = 0; i < 8; ++i) h[i] = kB2IV[i];
    h[0] ^= 0x01010000ULL ^ (static_cast<uint64_t>(key_len) << 8) ^ digest_len;
    t = 0;
    fill = 0;
    if (key_len) {
      std::memset(buf, 0, sizeof buf);
      std::memcpy(buf, key, key_len);
      fill = 128;  // the key block is the first data block
    }
  }

  void update(const uint8_t* data, size_t n) {
    while (n > 0) {
      if (fill == 128) {  // a full block is compressed only once more input follows
        t += 128;
        compress(buf, false);
        fill = 0;
      }
      const size_t take = n < 128 - fill ? n : 128 - fill;
      std::memcpy(buf + fill, data, take);
      fill += take;
      data += take;
      n -= take;
    }
  }

  void final(uint8_t* out) {
    t += fill;
    std::memset(buf + fill, 0, 128 - fill);
    compress(buf, true);
    for (size_t i = 0; i < out_len; ++i) out[i] = static_cast<uint8_t>(h[i / 8] >> (8 * (i % 8)));
  }
};

// ------------------------------------------------------------------ SHA-256
constexpr uint32_t kK256[64] = {
    0x428a2f98, 0x71374491, 0xb5c0fbcf, 0xe9b5dba5, 0x3956c25b, 0x59f111f1, 0x923f82a4, 0xab1c5ed5,
    0xd807aa98, 0x12835b01, 0x243185be, 0x550c7dc3, 0x72be5d74, 0x80deb1fe, 0x9bdc06a7, 0xc19bf174,
    0xe49b69c1, 0xefbe4786, 0x0fc19dc6, 0x240ca1cc, 0x2de92c6f, 0x4a7484aa, 0x5cb0a9dc, 0x76f988da,
    0x983e5152, 0xa831c66d, 0xb00327c8, 0xbf597fc7, 0xc6e00bf3, 0xd5a79147, 0x06ca6351, 0x14292967,
    0x27b70a85, 0x2e1b2138, 0x4d2c6dfc, 0x53380d13, 0x650a7354, 0x766a0abb, 0x81c2c92e, 0x92722c85,
    0xa2bfe8a1, 0xa81a664b, 0xc24b8b70, 0xc76c51a3, 0xd192e819, 0xd6990624, 0xf40e3585, 0x106aa070,
    0x19a4c116, 0x1e376c08, 0x2748774c, 0x34b0bcb5, 0x391c0cb3, 0x4ed8aa4a, 0x5b9cca4f, 0x682e6ff3,
    0x748f82ee, 0x78a5636f, 0x84c87814, 0x8cc70208, 0x90befffa, 0xa4506ceb, 0xbef9a3f7, 0xc67178f2};

inline uint32_t rotr32(uint32_t x, int n) { return (x >> n) | (x << (32 - n)); }

struct Sha256 {
  uint32_t h[8] = {0x6a09e667, 0xbb67ae85, 0x3c6ef372, 0xa54ff53a,
                   0x510e527f, 0x9b05688c, 0x1f83d9ab, 0x5be0cd19};
  uint8_t buf[64];
  size_t fill = 0;
  uint64_t total = 0;

  void block(const uint8_t* p) {
    uint32_t w[64];
    for (int i = 0; i < 16; ++i)
      w[i] = (uint32_t{p[4 * i]} << 24) | (uint32_t{p[4 * i + 1]} << 16) |
             (uint32_t{p[4 * i + 2]} << 8) | p[4 * i + 3];
    for (int i = 16; i < 64; ++i) {
      const uint32_t s0 = rotr32(w[i - 15], 7) ^ rotr32(w[i - 15], 18) ^ (w[i - 15] >> 3);
      const uint32_t s1 = rotr32(w[i - 2], 17) ^ rotr32(w[i - 2], 19) ^ (w[i - 2] >> 10);
      w[i] = w[i - 16] + s0 + w[i - 7] + s1;
    }
    uint32_t a = h[0], b = h[1], c = h[2], d = h[3], e = h[4], f = h[5], g = h[6], hh = h[7];
    for (int i = 0; i < 64; ++i) {
      const uint32_t S1 = rotr32(e, 6) ^ rotr32(e, 11) ^ rotr32(e, 25);
      const uint32_t ch = (e & f) ^ (~e & g);
      const uint32_t t1 = hh + S1 + ch + kK256[i] + w[i];
      const uint32_t S0 = rotr32(a, 2) ^ rotr32(a, 13) ^ rotr32(a, 22);
      const uint32_t maj = (a & b) ^ (a & c) ^ (b & c);
      const uint32_t t2 = S0 + maj;
      hh = g;
      g = f;
      f = e;
      e = d + t1;
      d = c;
      c = b;
      b = a;
      a = t1 + t2;
    }
    h[0] += a; h[1] += b; h[2] += c; h[3] += d;
    h[4] += e; h[5] += f; h[6] += g; h[7] += hh;
  }

  void update(const uint8_t* p, size_t n) {
    total += n;
    while (n > 0) {
      const size_t take = n < 64 - fill ? n : 64 - fill;
      std::memcpy(buf + fill, p, take);
      fill += take;
      p += take;
      n -= take;
      if (fill == 64) {
        block(buf);
        fill = 0;
      }
    }
  }

  void final(uint8_t out[32]) {
    const uint64_t bits = total * 8;
    const uint8_t one = 0x80, zero = 0;
    update(&one, 1);
    while (fill != 56) update(&zero, 1);
    uint8_t len[8];
    for (int i = 0; i < 8; ++i) len[i] = static_cast<uint8_t>(bits >> (56 - 8 * i));
    update(len, 8);
    for (int i = 0; i < 32; ++i) out[i] = static_cast<uint8_t>(h[i / 4] >> (24 - 8 * (i % 4)));
  }
};

void hmac_sha256(const uint8_t* key, size_t key_len, const uint8_t* msg, size_t msg_len,
                 uint8_t out[32]) {
  uint8_t k[64] = {0};
  if (key_len > 64) {
    Sha256 s;
    s.update(key, key_len);
    s.final(k);
  } else {
    std::memcpy(k, key, key_len);
  }
  uint8_t ipad[64], opad[64];
  for (int i = 0; i < 64; ++i) {
    ipad[i] = k[i] ^ 0x36;
    opad[i] = k[i] ^ 0x5c;
  }
  uint8_t inner[32];
  Sha256 a;
  a.update(ipad, 64);
  a.update(msg, msg_len);
  a.final(inner);
  Sha256 b;
  b.update(opad, 64);
  b.update(inner, 32);
  b.final(out);
}

}  // namespace

extern "C" {

int hc_tenant_key(const uint8_t* master, int32_t master_len, const char* tenant,
                  uint8_t* key_out) {
  if (!key_out || master_len < 0 || (master_len > 0 && !master)) return HC_ERR_INVALID_ARG;
  static const char kPublic[] = "hc-public";
  static const char kPrefix[] = "hc-tenant:";
  const size_t tlen = tenant ? std::strlen(tenant) : 0;
  if (tlen > 4096) return HC_ERR_INVALID_ARG;
  uint8_t msg[sizeof kPrefix - 1 + 4096];
  size_t n;
  if (tlen == 0) {
    n = sizeof kPublic - 1;
    std::memcpy(msg, kPublic, n);
  } else {
    n = sizeof kPrefix - 1;
    std::memcpy(msg, kPrefix, n);
    std::memcpy(msg + n, tenant, tlen);
    n += tlen;
  }
  hmac_sha256(master, static_cast<size_t>(master_len), msg, n, key_out);
  return HC_OK;
}

int hc_block_digests(const int32_t* tokens, int64_t n_tokens, int32_t block_size,
                     const uint8_t* key, int32_t key_len, uint8_t* prefix_digests,
                     uint8_t* content_digests) {
  if (n_tokens < 0 || block_size < 1 || key_len < 1 || key_len > 64 || !key)
    return HC_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!tokens || !prefix_digests || !content_digests)) return HC_ERR_INVALID_ARG;
  const int64_t n_blocks = (n_tokens + block_size - 1) / block_size;
  uint8_t le[4 * 1024];
  for (int64_t j = 0; j < n_blocks; ++j) {
    const int64_t t0 = j * block_size;
    const int64_t cnt = (n_tokens - t0) < block_size ? (n_tokens - t0) : block_size;
    Blake2b c, p;
    c.init(key, static_cast<size_t>(key_len), 16);
    p.init(key, static_cast<size_t>(key_len), 16);
    if (j > 0) p.update(prefix_digests + 16 * (j - 1), 16);
    for (int64_t i = 0; i < cnt; i += 1024) {  // tokens as little-endian int32, in chunks
      const int64_t m = (cnt - i) < 1024 ? (cnt - i) : 1024;
      for (int64_t q = 0; q < m; ++q) {
        const uint32_t v = static_cast<uint32_t>(tokens[t0 + i + q]);
        le[4 * q] = static_cast<uint8_t>(v);
        le[4 * q + 1] = static_cast<uint8_t>(v >> 8);
        le[4 * q + 2] = static_cast<uint8_t>(v >> 16);
        le[4 * q + 3] = static_cast<uint8_t>(v >> 24);
      }
      c.update(le, static_cast<size_t>(4 * m));
      p.update(le, static_cast<size_t>(4 * m));
    }
    c.final(content_digests + 16 * j);
    p.final(prefix_digests + 16 * j);
  }
  return HC_OK;
}

}  // extern "C"
