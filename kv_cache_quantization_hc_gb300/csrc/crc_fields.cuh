// GF(2)-linear maps onto CRC-32 registers, applied by table lookups on 5-bit
// fields.  Shared by the CRC kernel and the encoder's fused slab CRC.
//
// Everything a CRC computation does to a register or a message word is
// linear over GF(2) (crc_math.h): the register after a 16-byte word is a
// linear function of the word's 128 bits (with the incoming register xor-ed
// into its first four bytes), moving a register past n zero bytes multiplies
// it by x^(8n), and so on.  A linear map from N input bits to 32 output bits
// is stored as one table per 5-bit field of its input (the last field may be
// shorter): entry e of field f is the image of the input e << 5f, and the
// image of any input is the xor of its fields' entries (the slicing idea of
// Kounavis and Berry, "Novel table lookup-based algorithms for
// high-performance CRC generation", IEEE Trans. Computers 57(11), 2008, cut
// into 5-bit instead of 8-bit pieces).
//
// Why 5 bits: a 32-entry table of 4-byte words covers the 32 shared-memory
// banks exactly once, so the 32 lookups of a warp never collide - lanes that
// read different entries hit different banks, and lanes that read the same
// entry share one read.  A byte-indexed table spans every bank eight times,
// and a warp's 32 data-dependent lookups then collide 3-4 ways, which costs
// more than the 1.6x more lookups of 5-bit fields.
#pragma once

#include <cstdint>

namespace hc {

template <int N>
struct FieldMap {
  static constexpr int kWords = N / 32;
  static constexpr int kFields = (N + 4) / 5;
  uint32_t f[kFields][32];
};

// Fill `m` from the images of the N single-bit inputs (images[q] for input
// bit q, a shared or global array all threads can read).  Run by all threads
// of the CTA; the caller synchronizes before the map is used.
template <int N>
__device__ __forceinline__ void fill_field_map(FieldMap<N>& m, const uint32_t* images) {
  for (int i = threadIdx.x; i < FieldMap<N>::kFields * 32; i += blockDim.x) {
    const int f = i >> 5, e = i & 31, q = 5 * f;
    const int len = N - q < 5 ? N - q : 5;
    uint32_t c = 0;
    for (int b = 0; b < len; ++b)
      if ((e >> b) & 1) c ^= images[q + b];
    m.f[f][e] = c;
  }
}

// Entry of field F for the input v (N/32 little-endian words).  The field's
// value times 4 is the byte offset of its entry.
//
// The kernels that use these maps are bound by the integer ALU pipe: a
// field costs a shift and a mask there before its lookup.  A field that lies
// inside one word above bit 2 is written as a mask in place followed by the
// high word of a product with 2^(34 - s), which the compiler forms with a
// different shift instruction; both CRC kernels measured 2-3% faster with
// it, and ncu still shows the FMA pipe idle and the ALU pipe busy, so the
// bound is unchanged.  (The shift as a multiply-high of the unmasked word,
// masked afterwards, measured 8-10% slower; a multiplier of 2^(34 - s) + 1,
// which gives the same high word but cannot become a shift, keeps a true
// multiply-high on the FMA pipe and measured 19% slower.)
__device__ __forceinline__ uint32_t mul_hi(uint32_t a, uint32_t b) {
  uint32_t h;
  asm("mul.hi.u32 %0, %1, %2;" : "=r"(h) : "r"(a), "r"(b));
  return h;
}

template <int N, int F>
__device__ __forceinline__ uint32_t field_entry(const FieldMap<N>& m,
                                                const uint32_t (&v)[FieldMap<N>::kWords]) {
  constexpr int o = 5 * F, wi = o / 32, s = o % 32;
  constexpr int len = N - o < 5 ? N - o : 5;
  constexpr uint32_t mask = ((1u << len) - 1u) << 2;
  uint32_t x;
  if constexpr (s + len > 32) {
    x = __funnelshift_r(v[wi], v[wi + 1], s - 2) & mask;  // a field across two words (s >= 28)
  } else if constexpr (s > 2) {
    x = mul_hi(v[wi] & (mask << (s - 2)), 1u << (34 - s));
  } else {
    x = (v[wi] << (2 - s)) & mask;
  }
  return *reinterpret_cast<const uint32_t*>(reinterpret_cast<const char*>(m.f[F]) + x);
}

template <int N, int F = 0>
__device__ __forceinline__ uint32_t apply_map(const FieldMap<N>& m,
                                              const uint32_t (&v)[FieldMap<N>::kWords]) {
  if constexpr (F == FieldMap<N>::kFields) {
    return 0u;
  } else {
    return field_entry<N, F>(m, v) ^ apply_map<N, F + 1>(m, v);
  }
}

__device__ __forceinline__ uint32_t apply_map(const FieldMap<32>& m, uint32_t v) {
  const uint32_t w[1] = {v};
  return apply_map<32>(m, w);
}

}  // namespace hc
