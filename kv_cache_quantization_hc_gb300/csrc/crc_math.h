// GF(2) arithmetic of CRC-32/ISO-HDLC, shared by the CRC kernel, the fused
// encode CRC and the host code that builds their constants.
//
// Polynomials mod P are held bit-reflected: bit 31 - i is the coefficient of
// x^i, so multiplying by x is a right shift that folds the x^31 coefficient
// back with the reflected polynomial 0xEDB88320.  After n message bytes a CRC
// register is  init * x^(8n) + (a term linear in the message)  mod P.
#pragma once

#include <cstdint>

namespace hc {

constexpr uint32_t kCrcPolyReflected = 0xEDB88320u;

__host__ __device__ inline uint32_t crc_times_x(uint32_t v) {
  return (v >> 1) ^ ((v & 1u) ? kCrcPolyReflected : 0u);
}

// a * b mod P.
__host__ __device__ inline uint32_t gf2_mul(uint32_t a, uint32_t b) {
  uint32_t p = 0;
  for (int i = 0; i < 32; ++i) {
    if ((a >> (31 - i)) & 1u) p ^= b;
    b = crc_times_x(b);
  }
  return p;
}

// x^e mod P.
inline uint32_t crc_x_pow_bits(uint64_t e) {
  uint32_t result = 0x80000000u;  // 1
  uint32_t base = 0x40000000u;    // x
  for (; e; e >>= 1) {
    if (e & 1) result = gf2_mul(result, base);
    base = gf2_mul(base, base);
  }
  return result;
}

// x^(8n) mod P.
inline uint32_t crc_x_pow_bytes(uint64_t n) { return crc_x_pow_bits(8 * n); }

}  // namespace hc
