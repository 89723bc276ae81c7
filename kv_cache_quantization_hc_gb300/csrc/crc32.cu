// CRC-32 of encoded units, for tamper detection of stored or sent blocks.
// ["HyperCache - Distributed KV-cache quantization and relative RoPE reuse",
//  "Example output" part B, "INT4 (Grouped) L3 Disk (.hckv + CRC32)", and the
//  CRC32 tamper-detection tests it lists.]
//
// The variant is CRC-32/ISO-HDLC (zlib, PNG): polynomial 0x04C11DB7 processed
// bit-reflected, register initialised to 0xFFFFFFFF, final xor 0xFFFFFFFF.
//
// Polynomials mod P are held bit-reflected: bit 31 - i is the coefficient of
// x^i, so multiplying by x is a right shift that folds the x^31 coefficient
// back with the reflected polynomial 0xEDB88320.  After n message bytes the
// register is  init * x^(8n) + (a term linear in the message)  mod P, so a
// message can be cut into pieces whose registers (started at 0) are computed
// independently, moved to the end of the message by multiplying with
// x^(8 * bytes after the piece), and xor-ed.
//
// One warp per unit: lane k < 31 runs its piece of the a part, lane 31 the
// rest of a and all of b.  A lane consumes its piece 128 bytes at a time (eight
// 16-byte loads in flight), each 16-byte word in one step of the
// slicing-by-16 table method (Kounavis and Berry, "Novel table lookup-based
// algorithms for high-performance CRC generation", IEEE Trans. Computers
// 57(11), 2008): table k maps a byte to its register contribution when k
// zero bytes follow it.  The 16 tables (16 KiB) are built in shared memory by
// each CTA.
#include "crc_math.h"
#include "hc_internal.cuh"

namespace hc {
namespace {

constexpr uint32_t kPolyReflected = kCrcPolyReflected;
constexpr int kTables = 16;
inline uint32_t x_pow_bytes(uint64_t n) { return crc_x_pow_bytes(n); }

// One 16-byte word (bytes in memory order) into register r.
__device__ __forceinline__ uint32_t step16(const uint32_t (*T)[256], uint32_t r, uint4 w) {
  const uint32_t v = w.x ^ r;
  uint32_t c = T[15][v & 0xff] ^ T[14][(v >> 8) & 0xff] ^ T[13][(v >> 16) & 0xff] ^ T[12][v >> 24];
  c ^= T[11][w.y & 0xff] ^ T[10][(w.y >> 8) & 0xff] ^ T[9][(w.y >> 16) & 0xff] ^ T[8][w.y >> 24];
  c ^= T[7][w.z & 0xff] ^ T[6][(w.z >> 8) & 0xff] ^ T[5][(w.z >> 16) & 0xff] ^ T[4][w.z >> 24];
  c ^= T[3][w.w & 0xff] ^ T[2][(w.w >> 8) & 0xff] ^ T[1][(w.w >> 16) & 0xff] ^ T[0][w.w >> 24];
  return c;
}

__device__ __forceinline__ uint32_t step1(const uint32_t (*T)[256], uint32_t r, uint32_t byte) {
  return (r >> 8) ^ T[0][(r ^ byte) & 0xff];
}

__global__ void __launch_bounds__(kThreads) k_crc32(CrcParams p) {
  __shared__ uint32_t T[kTables][256];
  {
    const uint32_t t = threadIdx.x;  // kThreads == 256: one table entry per thread
    uint32_t c = t;
    for (int i = 0; i < 8; ++i) c = (c >> 1) ^ ((c & 1u) ? kPolyReflected : 0u);
    T[0][t] = c;
    __syncthreads();
    for (int k = 1; k < kTables; ++k) {
      c = (c >> 8) ^ T[0][c & 0xff];
      T[k][t] = c;
    }
    __syncthreads();
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t u = blockIdx.x * kWarps + warp;
  if (u >= p.n_units) return;
  const uint8_t* a = p.a + static_cast<int64_t>(u) * p.a_stride;
  const int64_t begin = lane * p.chunk;
  const int64_t end = lane < 31 ? begin + p.chunk : p.a_bytes;
  uint32_t r = 0;
  int64_t pos = begin;
  for (; pos + 128 <= end; pos += 128) {
    uint4 w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = __ldcs(reinterpret_cast<const uint4*>(a + pos) + i);
#pragma unroll
    for (int i = 0; i < 8; ++i) r = step16(T, r, w[i]);
  }
  for (; pos + 16 <= end; pos += 16) r = step16(T, r, __ldcs(reinterpret_cast<const uint4*>(a + pos)));
  for (; pos < end; ++pos) r = step1(T, r, a[pos]);
  if (lane == 31 && p.b_bytes > 0) {
    const uint8_t* b = p.b + static_cast<int64_t>(u) * p.b_stride;
    for (int64_t i = 0; i < p.b_bytes; ++i) r = step1(T, r, b[i]);
  }
  r = gf2_mul(r, p.lane_shift[lane]);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) r ^= __shfl_xor_sync(0xffffffffu, r, o);
  if (lane == 0) p.crc[u] = r ^ p.init_term;
}

}  // namespace

cudaError_t launch_crc32(const CrcParams& in, cudaStream_t s) {
  CrcParams p = in;
  p.chunk = (p.a_bytes / (32 * 128)) * 128;
  const uint64_t n = static_cast<uint64_t>(p.a_bytes + p.b_bytes);
  for (int k = 0; k < 32; ++k) {
    const uint64_t after = k < 31 ? n - static_cast<uint64_t>((k + 1) * p.chunk) : 0;
    p.lane_shift[k] = x_pow_bytes(after);
  }
  p.init_term = gf2_mul(0xFFFFFFFFu, x_pow_bytes(n)) ^ 0xFFFFFFFFu;
  const uint32_t grid = (p.n_units + kWarps - 1) / kWarps;
  k_crc32<<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hc
