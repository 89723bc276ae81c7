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
// One warp per unit, persistent CTAs (k_crc32); few, large units are cut
// into chunks across warps (k_crc32_split, below).  A unit is two segments: the 16-byte
// words of a (16-byte aligned), then the ragged rest of a followed by b, read
// byte by byte and padded in front with zero bytes to whole 16-byte words
// (leading zeros leave a zero-started register unchanged).  Where a has no
// ragged rest and b is whole 16-byte words on 16-byte boundaries (the FP8
// wire's scales), the second segment is read as words too.  A segment is cut
// into rows of 32 words, 512 bytes, and padded in front with zero words to a
// whole number of groups of kCrcGroup rows.  Lane l takes word l of every row, so
// a warp's loads are 512 contiguous bytes.  Per group of rows a lane moves its
// register past the group (x^(8 * 512 * kCrcGroup)) and adds each of its words'
// contributions, read from the map of that word's row position; the register
// then describes everything the lane has read, with every other lane's bytes
// taken as zero, positioned at the end of the lane's last word, 16 (31 - l)
// bytes before its segment's end.  Each lane moves its first-segment register
// past the second segment (a map built from x^(8 * its bytes)) and adds its
// second-segment register; a butterfly over the lanes (the lower lane of each
// pair moves its register 16 * 2^j bytes on and adds its partner's) then
// leaves lane 0 with the unit's register, to which it adds the initial
// register's term and the final xor.
//
// Why rows: giving each lane a contiguous piece of the unit instead (as a first
// design did) makes a warp's 16-byte loads touch 32 lines 1 KiB apart; that
// layout, with byte-indexed tables whose lookups collide, held the kernel to
// 2.0 TB/s.
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
  FieldMap<32> group;             // a register -> the register kCrcGroup rows later
  FieldMap<32> level[5];          // a register -> the register 16 * 2^j bytes later
  FieldMap<32> seg2;              // a register -> the register after the second segment
};

__device__ void build_maps(const CrcParams& p, CrcShared& s) {
  for (int g = 0; g < kCrcGroup; ++g) fill_field_map<128>(s.word[g], p.img_word[g]);
  fill_field_map<32>(s.group, p.img_group);
  for (int j = 0; j < 5; ++j) fill_field_map<32>(s.level[j], p.img_level[j]);
  fill_field_map<32>(s.seg2, p.img_seg2);
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

// Whether row j of a segment's first group holds any word (rows wholly in
// the front padding contribute nothing and are skipped).  `first0` is the
// word index of lane 0's word in row 0, the same in every lane.
__device__ __forceinline__ bool row_has_words(int64_t first0, int j) {
  return first0 + 31 + 32 * j >= 0;
}

// The lane's register over groups [g0, g1) of a segment of 16-byte words at
// `a` (front-padded to whole groups), positioned at the end of its last word
// in group g1 - 1.  `first` is the word index of this lane's word in row 0
// of group 0 (negative in the padding).  Only group 0 can hold front
// padding; the rest read at a pointer that steps a group at a time.
__device__ __forceinline__ uint32_t group_range(const CrcShared& s, const uint4* a, int64_t first,
                                                int lane, int64_t g0, int64_t g1) {
  constexpr int kGroupWords = 32 * kCrcGroup;
  uint32_t r = 0;
  int64_t g = g0;
  if (g == 0 && g < g1) {
#pragma unroll
    for (int j = 0; j < kCrcGroup; ++j) {
      if (!row_has_words(first - lane, j)) continue;
      const int64_t k = first + j * 32;
      r ^= word_contrib(s.word[j], k >= 0 ? __ldcs(a + k) : make_uint4(0u, 0u, 0u, 0u));
    }
    ++g;
  }
  if (g >= g1) return r;
  const uint4* ptr = a + (first + g * kGroupWords);
  const int n = static_cast<int>(g1 - g);
#pragma unroll 2
  for (int gi = 0; gi < n; ++gi, ptr += kGroupWords) {
    uint4 w[kCrcGroup];
#pragma unroll
    for (int j = 0; j < kCrcGroup; ++j) w[j] = __ldcs(ptr + j * 32);
    uint32_t c = apply_map(s.group, r);
#pragma unroll
    for (int j = 0; j < kCrcGroup; ++j) c ^= word_contrib(s.word[j], w[j]);
    r = c;
  }
  return r;
}

__device__ __forceinline__ int64_t padded_groups(int64_t n_words) {
  return (n_words + 32 * kCrcGroup - 1) / (32 * kCrcGroup);
}

// A segment of n_words 16-byte words: the lane's register, at the end of its
// word in the segment's last row, 16 (31 - lane) bytes before the segment's end.
__device__ __forceinline__ uint32_t segment_words(const CrcShared& s, const uint4* a,
                                                  int64_t n_words, int lane) {
  const int64_t groups = padded_groups(n_words);
  const int64_t first = n_words - groups * 32 * kCrcGroup + lane;  // > lane - 128
  return group_range(s, a, first, lane, 0, groups);
}

// Segment 2: t bytes at `at`, then nb bytes at `b`, read byte by byte; the
// lane's register as for segment_words.
__device__ __forceinline__ uint32_t segment_bytes(const CrcShared& s, const uint8_t* at, int64_t t,
                                                  const uint8_t* b, int64_t nb, int lane) {
  const int64_t len = t + nb;
  const int64_t n_words = (len + 15) / 16;
  const int64_t front = 16 * n_words - len;  // zero bytes in front
  const int64_t groups = (n_words + 32 * kCrcGroup - 1) / (32 * kCrcGroup);
  const int64_t first = n_words - groups * 32 * kCrcGroup + lane;
  uint32_t r = 0;
  for (int64_t gi = 0; gi < groups; ++gi) {
    uint32_t c = gi ? apply_map(s.group, r) : 0u;
#pragma unroll
    for (int g = 0; g < kCrcGroup; ++g) {
      if (gi == 0 && !row_has_words(first - lane, g)) continue;
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
  return r;
}

// Segment 2 alone: lane 0 ends with its register at the segment's end.
__device__ __forceinline__ uint32_t second_segment(const CrcParams& p, const CrcShared& s,
                                                   const uint8_t* at, int64_t t, const uint8_t* b,
                                                   int lane) {
  return p.b_words ? segment_words(s, reinterpret_cast<const uint4*>(b), p.b_bytes >> 4, lane)
                   : segment_bytes(s, at, t, b, p.b_bytes, lane);
}

__global__ void __launch_bounds__(kThreads) k_crc32(const __grid_constant__ CrcParams p) {
  __shared__ CrcShared maps;
  build_maps(p, maps);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t words = p.a_bytes >> 4, t = p.a_bytes & 15;
  for (uint32_t u = blockIdx.x * kWarps + warp; u < p.n_units; u += gridDim.x * kWarps) {
    const uint8_t* a = p.a + static_cast<int64_t>(u) * p.a_stride;
    // Each lane's registers sit 16 (31 - lane) bytes before the end of their
    // segment; moving the first segment's past the second (seg2) puts both
    // at the same distance from the unit's end, so one butterfly joins them.
    uint32_t r = words ? segment_words(maps, reinterpret_cast<const uint4*>(a), words, lane) : 0u;
    if (t + p.b_bytes > 0) {
      const uint8_t* b = p.b_bytes > 0 ? p.b + static_cast<int64_t>(u) * p.b_stride : nullptr;
      r = apply_map(maps.seg2, r) ^
          (p.b_words ? segment_words(maps, reinterpret_cast<const uint4*>(b), p.b_bytes >> 4, lane)
                     : segment_bytes(maps, a + 16 * words, t, b, p.b_bytes, lane));
    }
    r = lane_tree(maps, r, lane);
    if (lane == 0) p.crc[u] = r ^ p.init_term;
  }
}

// Few, large units: each unit's segment 1 is cut into chunks of
// p.chunk_groups groups, one warp per chunk, and one more warp per unit takes
// segment 2.  A chunk's register is moved to the unit's end (past the rest of
// segment 1 and all of segment 2) and xor-ed into crc[u], which the host
// zeroed; the segment-2 warp adds the initial register's term and the final
// xor.  The xors commute, so the result does not depend on their order.
__global__ void __launch_bounds__(kThreads) k_crc32_split(const __grid_constant__ CrcParams p) {
  __shared__ CrcShared maps;
  build_maps(p, maps);
  const int lane = threadIdx.x & 31;
  const int64_t words = p.a_bytes >> 4, t = p.a_bytes & 15;
  const int64_t groups = padded_groups(words);
  const int64_t per_unit = p.chunks + 1;  // chunk warps, then the segment-2 warp
  const int64_t total = per_unit * p.n_units;
  for (int64_t item = static_cast<int64_t>(blockIdx.x) * kWarps + (threadIdx.x >> 5); item < total;
       item += static_cast<int64_t>(gridDim.x) * kWarps) {
    const int64_t u = item / per_unit, k = item % per_unit;
    const uint8_t* a = p.a + u * p.a_stride;
    uint32_t r;
    if (k < p.chunks) {
      const int64_t g0 = k * p.chunk_groups;
      const int64_t g1 = g0 + p.chunk_groups < groups ? g0 + p.chunk_groups : groups;
      const int64_t first = words - groups * 32 * kCrcGroup + lane;
      r = lane_tree(maps, group_range(maps, reinterpret_cast<const uint4*>(a), first, lane, g0, g1),
                    lane);
      if (lane == 0) {
        // x^(8 * 16 * 32 * kCrcGroup * (groups - g1)) from the host's powers of two
        uint32_t m = 0x80000000u;
        for (int64_t e = groups - g1, i = 0; e; e >>= 1, ++i)
          if (e & 1) m = gf2_mul(m, p.group_pow2[i]);
        r = gf2_mul(gf2_mul(r, m), p.seg2_shift);
      }
    } else {
      const uint8_t* b = p.b_bytes > 0 ? p.b + u * p.b_stride : nullptr;
      r = t + p.b_bytes > 0 ? lane_tree(maps, second_segment(p, maps, a + 16 * words, t, b, lane), lane)
                            : 0u;
      r ^= p.init_term;
    }
    if (lane == 0) atomicXor(p.crc + u, r);
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
  for (int j = 0; j < 32; ++j) p.img_seg2[j] = gf2_mul(1u << j, p.seg2_shift);
  p.b_words = (p.a_bytes & 15) == 0 && p.b_bytes > 0 && p.b_bytes % 16 == 0 &&
              reinterpret_cast<uintptr_t>(p.b) % 16 == 0 && (p.n_units == 1 || p.b_stride % 16 == 0);
  p.init_term = gf2_mul(0xFFFFFFFFu, crc_x_pow_bytes(n)) ^ 0xFFFFFFFFu;
  // One warp per unit: a persistent grid of twice the CTAs that fit
  // nominally (kCrcCtasPerSm per SM; at 40 registers 6 fit), which measured
  // 1.7% faster than once (3.91 against 3.85 TB/s) and 7% faster than one
  // CTA per 8 units; 4 times measured 3.80.
#ifndef HC_CRC_GRID_WAVES
#define HC_CRC_GRID_WAVES 2
#endif
  const int64_t resident = static_cast<int64_t>(device_sm_count()) * kCrcCtasPerSm;
  const int64_t groups = (p.a_bytes / 16 + 32 * kCrcGroup - 1) / (32 * kCrcGroup);
  if (static_cast<int64_t>(p.n_units) * 2 >= resident * kWarps || groups < 2 * kCrcMinChunkGroups) {
    // one warp per unit
    const int64_t ctas = (static_cast<int64_t>(p.n_units) + kWarps - 1) / kWarps;
    k_crc32<<<static_cast<uint32_t>(std::min<int64_t>(ctas, resident * HC_CRC_GRID_WAVES)), kThreads, 0,
              s>>>(p);
    return cudaGetLastError();
  }
  // few, large units: chunks of at least kCrcMinChunkGroups groups, about
  // two warps' worth per resident warp slot
  const int64_t want = std::max<int64_t>(1, 2 * resident * kWarps / p.n_units);
  p.chunk_groups = std::max<int64_t>(kCrcMinChunkGroups, (groups + want - 1) / want);
  p.chunks = (groups + p.chunk_groups - 1) / p.chunk_groups;
  for (int i = 0; i < 48; ++i)
    p.group_pow2[i] = crc_x_pow_bytes((16ull * 32 * kCrcGroup) << i);
  const cudaError_t e = cudaMemsetAsync(p.crc, 0, sizeof(uint32_t) * p.n_units, s);
  if (e != cudaSuccess) return e;
  const int64_t warps = (p.chunks + 1) * static_cast<int64_t>(p.n_units);
  const int64_t ctas = (warps + kWarps - 1) / kWarps;
  k_crc32_split<<<static_cast<uint32_t>(std::min<int64_t>(ctas, resident)), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hc
