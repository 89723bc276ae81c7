// CRC-32 of encoded units, for tamper detection of stored or sent blocks.
// ["HyperCache - Distributed KV-cache quantization and relative RoPE reuse",
//  "Example output" part B, "INT4 (Grouped) L3 Disk (.hckv + CRC32)", and the
//  CRC32 tamper-detection tests it lists.]
//
// The variant is CRC-32/ISO-HDLC (zlib, PNG): polynomial 0x04C11DB7 processed
// bit-reflected, register initialised to 0xFFFFFFFF, final xor 0xFFFFFFFF.
// The GF(2) arithmetic is in crc_math.h, the table-driven linear maps in
// crc_fields.cuh.
//
// A register that starts at 0 does not change over leading zero bytes, and
// after n message bytes it is  (a term linear in the message)  while the
// initial register contributes init * x^(8n) mod P.  So a message can be cut
// into pieces whose registers are computed independently and moved to the
// message's end by multiplying with x^(8 * bytes after the piece).
//
// One warp per unit, persistent CTAs.  A unit is two segments: the 16-byte
// words of a (16-byte aligned), then the ragged rest of a followed by b, read
// byte by byte and padded in front with zero bytes to whole 16-byte words
// (leading zeros leave a zero-started register unchanged).  A segment is cut
// into rows of 32 words, 512 bytes, and padded in front with zero words to a
// whole number of groups of kGroup rows.  Lane l takes word l of every row, so
// a warp's loads are 512 contiguous bytes.  Per group of rows a lane moves its
// register past the group (x^(8 * 512 * kGroup)) and adds each of its words'
// contributions, read from the map of that word's row position; the register
// then describes everything the lane has read, with every other lane's bytes
// taken as zero, positioned at the end of the lane's last word.  A butterfly
// over the lanes (the lower lane of each pair moves its register 16 * 2^j
// bytes on and adds its partner's) leaves lane 0 with the segment's register
// at the segment's end.  Lane 0 moves the first segment's register past the
// second segment and adds the second's, the initial register's term and the
// final xor.
//
// Why rows: the previous design gave each lane a contiguous piece of the unit,
// so a warp's 16-byte loads touched 32 lines 1 KiB apart; that layout, plus
// byte-indexed tables whose lookups collide, held the kernel to 2.0 TB/s.
#include <algorithm>
#include <cstring>
#include <mutex>

#include "crc_fields.cuh"
#include "crc_math.h"
#include "hc_internal.cuh"

namespace hc {
namespace {

// Tables of one CTA, filled from the host-computed images in CrcParams.
struct CrcShared {
  FieldMap<128> word[kCrcGroup];  // word at row position g of a group -> register at the group's end
  FieldMap<32> group;             // a register -> the register kGroup rows later
  FieldMap<32> level[5];          // a register -> the register 16 * 2^j bytes later
};

__device__ void build_maps(const CrcParams& p, CrcShared& s) {
  for (int g = 0; g < kCrcGroup; ++g) fill_field_map<128>(s.word[g], p.img_word[g]);
  fill_field_map<32>(s.group, p.img_group);
  for (int j = 0; j < 5; ++j) fill_field_map<32>(s.level[j], p.img_level[j]);
  __syncthreads();
}

__device__ __forceinline__ uint32_t lane_tree(const CrcShared& s, uint32_t r, int lane) {
#pragma unroll
  for (int j = 0; j < 5; ++j) {
    const uint32_t other = __shfl_xor_sync(0xffffffffu, r, 1 << j);
    const uint32_t moved = apply_map(s.level[j], r);
    r = ((lane >> j) & 1) ? r : (moved ^ other);
  }
  return r;
}

__device__ __forceinline__ uint32_t word_contrib(const FieldMap<128>& m, uint4 w) {
  const uint32_t v[4] = {w.x, w.y, w.z, w.w};
  return apply_map<128>(m, v);
}

// Segment 1: the n_words 16-byte words at `a`.  Only the first group can
// hold front padding; the rest read at a pointer that steps a group at a time.
__device__ __forceinline__ uint32_t aligned_segment(const CrcShared& s, const uint4* a,
                                                    int64_t n_words, int lane) {
  constexpr int kGroupWords = 32 * kCrcGroup;
  const int groups = static_cast<int>((n_words + kGroupWords - 1) / kGroupWords);
  const int64_t first = n_words - static_cast<int64_t>(groups) * kGroupWords + lane;  // > lane - 128
  uint32_t r = 0;
#pragma unroll
  for (int g = 0; g < kCrcGroup; ++g) {
    const int64_t k = first + g * 32;
    r ^= word_contrib(s.word[g], k >= 0 ? __ldcs(a + k) : make_uint4(0u, 0u, 0u, 0u));
  }
  const uint4* ptr = a + (first + kGroupWords);
#pragma unroll 2
  for (int gi = 1; gi < groups; ++gi, ptr += kGroupWords) {
    uint4 w[kCrcGroup];
#pragma unroll
    for (int g = 0; g < kCrcGroup; ++g) w[g] = __ldcs(ptr + g * 32);
    uint32_t c = apply_map(s.group, r);
#pragma unroll
    for (int g = 0; g < kCrcGroup; ++g) c ^= word_contrib(s.word[g], w[g]);
    r = c;
  }
  return lane_tree(s, r, lane);
}

// Segment 2: t bytes at `at`, then nb bytes at `b`, read byte by byte.
__device__ __forceinline__ uint32_t byte_segment(const CrcShared& s, const uint8_t* at, int64_t t,
                                                 const uint8_t* b, int64_t nb, int lane) {
  const int64_t len = t + nb;
  const int64_t n_words = (len + 15) / 16;
  const int64_t front = 16 * n_words - len;  // zero bytes in front
  const int64_t groups = (n_words + 32 * kCrcGroup - 1) / (32 * kCrcGroup);
  const int64_t first = n_words - groups * 32 * kCrcGroup + lane;
  uint32_t r = 0;
  for (int64_t gi = 0; gi < groups; ++gi) {
    uint32_t c = apply_map(s.group, r);
#pragma unroll
    for (int g = 0; g < kCrcGroup; ++g) {
      const int64_t k = first + (gi * kCrcGroup + g) * 32;
      uint32_t v[4] = {0u, 0u, 0u, 0u};
      if (k >= 0) {
        for (int i = 0; i < 16; ++i) {
          const int64_t m = 16 * k + i - front;  // byte of the segment
          const uint32_t byte = m < 0 ? 0u : (m < t ? at[m] : b[m - t]);
          v[i >> 2] |= byte << (8 * (i & 3));
        }
      }
      c ^= apply_map<128>(s.word[g], v);
    }
    r = c;
  }
  return lane_tree(s, r, lane);
}

__global__ void __launch_bounds__(kThreads) k_crc32(const __grid_constant__ CrcParams p) {
  __shared__ CrcShared maps;
  build_maps(p, maps);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t words = p.a_bytes >> 4, t = p.a_bytes & 15;
  for (uint32_t u = blockIdx.x * kWarps + warp; u < p.n_units; u += gridDim.x * kWarps) {
    const uint8_t* a = p.a + static_cast<int64_t>(u) * p.a_stride;
    uint32_t r1 = words ? aligned_segment(maps, reinterpret_cast<const uint4*>(a), words, lane) : 0u;
    uint32_t r2 = 0;
    if (t + p.b_bytes > 0) {
      const uint8_t* b = p.b_bytes > 0 ? p.b + static_cast<int64_t>(u) * p.b_stride : nullptr;
      r2 = byte_segment(maps, a + 16 * words, t, b, p.b_bytes, lane);
    }
    if (lane == 0) p.crc[u] = gf2_mul(r1, p.seg2_shift) ^ r2 ^ p.init_term;
  }
}

// The images of the maps' single-bit inputs; they depend on nothing but the
// polynomial and kCrcGroup, so they are computed once per process.
struct CrcImages {
  uint32_t word[kCrcGroup][128], group[32], level[5][32];
};

const CrcImages& crc_images() {
  static CrcImages img;
  static std::once_flag once;
  std::call_once(once, [] {
    // Message bit q of a 16-byte word (bit q % 8 of byte q / 8; the reflected
    // order processes bit 0 of byte 0 first) is the coefficient of
    // x^(127 - q), and x^32 more moves it into the register after the word.
    for (int g = 0; g < kCrcGroup; ++g) {
      const uint32_t later = crc_x_pow_bytes(512u * (kCrcGroup - 1 - g));
      for (int q = 0; q < 128; ++q) img.word[g][q] = gf2_mul(crc_x_pow_bits(159 - q), later);
    }
    // A register bit j (bit 31 - i holds x^i) times the shift.
    const uint32_t grp = crc_x_pow_bytes(512u * kCrcGroup);
    for (int j = 0; j < 32; ++j) img.group[j] = gf2_mul(1u << j, grp);
    for (int l = 0; l < 5; ++l) {
      const uint32_t sh = crc_x_pow_bytes(16u << l);
      for (int j = 0; j < 32; ++j) img.level[l][j] = gf2_mul(1u << j, sh);
    }
  });
  return img;
}

}  // namespace

cudaError_t launch_crc32(const CrcParams& in, cudaStream_t s) {
  CrcParams p = in;
  const CrcImages& img = crc_images();
  std::memcpy(p.img_word, img.word, sizeof img.word);
  std::memcpy(p.img_group, img.group, sizeof img.group);
  std::memcpy(p.img_level, img.level, sizeof img.level);
  const uint64_t n = static_cast<uint64_t>(p.a_bytes + p.b_bytes);
  p.seg2_shift = crc_x_pow_bytes(static_cast<uint64_t>((p.a_bytes & 15) + p.b_bytes));
  p.init_term = gf2_mul(0xFFFFFFFFu, crc_x_pow_bytes(n)) ^ 0xFFFFFFFFu;
  const int64_t ctas = (static_cast<int64_t>(p.n_units) + kWarps - 1) / kWarps;
  const uint32_t grid = static_cast<uint32_t>(
      std::min<int64_t>(ctas, static_cast<int64_t>(device_sm_count()) * kCrcCtasPerSm));
  k_crc32<<<grid, kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hc
