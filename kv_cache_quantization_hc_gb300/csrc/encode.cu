// Evict/encode kernels: gather paged K/V blocks through the source block table
// and quantize them to the wire.
//
// FP8: one fp32 scale per (layer, block, kv, head) slab of B x d elements,
//      s = fp32(amax / 448), code = E4M3_rn_satfinite(fp32(x / s)).
// INT4: one scale per (layer, block, kv, head, token, group of g channels),
//      s = [fp16_rn](fp32(amax / 7)), code = clamp(rint(fp32(x / s)), -7, 7).
// ["HyperCache - Distributed KV-cache quantization and relative RoPE reuse",
//  "Core Design" compression paragraph; "Example output" part B.]
//
// Work decomposition.  One warp owns a 16-token sub-slab of one (layer,
// block, kv, head); each lane owns one 8-element chunk of a token row
// (16 bytes for fp16/bf16, 32 for fp32) per pass, 256/d rows per pass, d/16
// passes.  A CTA's warps take a "unit" of as many consecutive sub-slabs.
// Two launch shapes, chosen by measurement on GB300: one unit per CTA (16-bit
// INT4 in 4-warp CTAs; 16-bit FP8 with blocks over 16 tokens in CTAs of one
// slab's warps, at least 4), or persistent 8-warp CTAs, two per SM, stepping
// through the units with a three-deep
// pipeline per warp: the block table entry for unit i+2 is requested, the
// rows of unit i+1 are loaded (16-bit sources: into a second register
// buffer), and unit i is quantized and stored - so neither the table lookup
// nor the row loads sit on the critical path.  The FP8 slab amax needs all
// B/16 sub-slabs of a block;
// those warps are in the same CTA and combine through shared memory.  INT4
// groups lie inside a token row, so INT4 needs no cross-warp step.
//
// Quotients without a division per element.  The codes are defined through
// the IEEE quotient q* = fp32(x / s).
//
// 16-bit sources (FP8, and INT4 with fp16 scales): the product with a
// reciprocal of s, corrected once by its exact residual (Markstein), gives
// q* itself (FP8, correctly rounded reciprocal) or a value with the same
// rounded integer (INT4, approximate reciprocal).  Both are checked on every
// 16-bit (x, amax) pair against IEEE arithmetic (fp8x8_corrected,
// int4x8_corrected); scales outside the checked domain take the division.
//
// fp32 sources (and INT4 with fp32 scales): with r = fp32(1/s) and the
// bracketing multipliers r_lo = fp32(r (1 - 2^-20)), r_hi = fp32(r (1 + 2^-20)),
// the products q_lo = fp32(x r_lo) and q_hi = fp32(x r_hi) satisfy
// |q_lo| < |q*| < |q_hi| (three roundings of at most 2^-24 each cannot undo a
// 2^-20 relative offset; when x/s is so small that fp32 underflows, all three
// are far below the smallest code step and encode alike).  The quantizer is
// monotone in |q| for a fixed sign, so when q_lo and q_hi give the same code,
// that is the code of q*.  Where they differ, q* sits at (or within 2^-20 of)
// a rounding boundary: the main loop only flags the pass and stores the
// lower-bracket codes, and a deferred step per sub-slab revisits each lane's
// flagged passes and resolves just the disagreeing elements (an exact
// FMA-residual test, see fp8_resolve; IEEE division where that test does not
// apply), re-storing the 8 codes.  A scale below the smallest normal fp32
// takes the division path.
//
// Products are formed two at a time (FMUL2 / FFMA2).
//
// Reads use the streaming cache hint (each element is read once); codes are
// written with streaming stores.
#include <algorithm>
#include <type_traits>

#include "crc_fields.cuh"
#include "crc_math.h"
#include "encode_common.cuh"

namespace hc {
namespace {

template <int D>
struct EncodeGeom {
  static constexpr int kChunksPerRow = D / 8;
  static constexpr int kRowsPerPass = 32 / kChunksPerRow;
  static constexpr int kPasses = kRowsPerWarp / kRowsPerPass;
};

// Bracketing reciprocals of a scale (see the file comment).
struct Brackets {
  float2 lo, hi;
  bool ok;  // s is large enough for the bracket argument (and, INT4, no clamping)
};

__device__ __forceinline__ Brackets brackets(float s, float min_scale) {
  Brackets b;
  const float r = __frcp_rn(s);
  const float lo = r * (1.0f - 0x1p-20f), hi = r * (1.0f + 0x1p-20f);
  b.lo = make_float2(lo, lo);
  b.hi = make_float2(hi, hi);
  b.ok = s >= min_scale;
  return b;
}

__device__ __forceinline__ uint32_t fp8x1(float v) { return fp8x2(make_float2(v, 0.f)) & 0xffu; }

__device__ __noinline__ uint32_t fp8_div1(float x, float s) { return fp8x1(__fdiv_rn(x, s)); }

// Bit k set iff byte k of w is non-zero (k < 4): fold each byte onto its low
// bit, then gather the four bits with one multiply (no carries reach 24..27).
__device__ __forceinline__ uint32_t nonzero_bytes4(uint32_t w) {
  uint32_t t = w | (w >> 4);
  t |= t >> 2;
  t |= t >> 1;
  t &= 0x01010101u;
  return ((t * 0x01020408u) >> 24) & 0xfu;
}

// The code of q* = fp32(x/s) for an element whose bracket codes disagree.
// The brackets straddle exactly one E4M3 rounding boundary mu (they are 2^-19
// apart, boundaries at least 2^-4), so the answer is the lower code c_lo, the
// next code c_hi, or - when q* is mu itself - the even one of the two.  For
// |q| >= 2^-6 (the normal E4M3 range) mu has the form 1.xxx1 * 2^k, and the
// upper bracket product lies less than 2^4 fp32 ulps above it: clearing its
// mantissa below bit 19 gives mu.  The residual res = fma(-mu, s, |x|) =
// |x| - mu s is exact (its magnitude is below 2^-19 |x| and it has at most 29
// significant bits ending near x's lowest bit minus 5).  q* = mu exactly iff
// |x/s - mu| <= ulp(mu)/2, i.e. |res| <= s ulp(mu)/2 (mu has few significant
// bits, so an fp32 tie also rounds to it); otherwise the sign of res gives the
// side.  Quotients in the E4M3 subnormal range and scales below 2^-90 (where
// res or s ulp(mu)/2 could leave the normal range) use the IEEE division.
__device__ __forceinline__ uint32_t fp8_resolve(float xe, float s, float rhi, float s_half_ulp,
                                                bool resolvable, uint32_t lo_code) {
  const float ax = fabsf(xe);
  const float qh = ax * rhi;
  const uint32_t c_lo = lo_code & 0x7fu;
  const uint32_t c_hi = c_lo + 1u;
  if (resolvable && qh >= 0x1p-6f) {
    const float mu = __uint_as_float(__float_as_uint(qh) & 0xfff80000u);
    const float res = fmaf(-mu, s, ax);
    const float thr = __uint_as_float(__float_as_uint(mu) & 0x7f800000u) * s_half_ulp;
    const uint32_t code = fabsf(res) <= thr ? ((c_lo & 1u) ? c_hi : c_lo) : (res > 0.f ? c_hi : c_lo);
    return code | (__float_as_uint(xe) >> 31 << 7);
  }
  return fp8_div1(xe, s);
}

// 8 E4M3 codes of x[0..7] / s (see the file comment).
__device__ __forceinline__ uint2 fp8x8(const float2 (&x)[4], float s, const Brackets& br, uint2& diff) {
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    lo[e] = fp8x2(__fmul2_rn(x[e], br.lo));
    hi[e] = fp8x2(__fmul2_rn(x[e], br.hi));
  }
  const uint2 wl = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
  const uint2 wh = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
  diff = make_uint2(wl.x ^ wh.x, wl.y ^ wh.y);
  return wl;
}

// round_half_even(q) + 8 for |q| <= 7.5: adding 1.5 * 2^23 + 8 (an even
// integer, in the binade where the fp32 spacing is 1) rounds q to the
// nearest-even integer in one IEEE rounding and leaves rint(q) + 8, in
// [1, 15], as the whole low byte of the sum's bit pattern (the bits above it
// are those of 1.5 * 2^23).
constexpr float kRintMagic = 12582920.0f;

// The 4-bit two's complement codes from eight biased bytes b[e] = code_e + 8
// (in the low byte of each word), element 2k in the low half of byte k:
// byte k = (b[2k] + 16 b[2k+1]) ^ 0x88 - the two biased nibbles cannot carry
// into each other, and flipping bit 3 of code + 8 gives the code's nibble.
__device__ __forceinline__ uint32_t pack_nibbles(const uint32_t (&b)[8]) {
  uint32_t p[4];
#pragma unroll
  for (int k = 0; k < 4; ++k) p[k] = b[2 * k] + (b[2 * k + 1] << 4);
  return __byte_perm(__byte_perm(p[0], p[1], 0x0040), __byte_perm(p[2], p[3], 0x0040), 0x5410) ^
         0x88888888u;
}

// The hardware reciprocal approximation (at most 1 ulp of error).
__device__ __forceinline__ float rcp_approx(float s) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(s));
  return r;
}

__device__ __forceinline__ uint32_t int4_of(float q) {
  return static_cast<uint32_t>(min(7, max(-7, __float2int_rn(q)))) & 0xfu;
}

// INT4 codes for fp16 scales and 16-bit sources: the quotient corrected by its
// exact residual (Markstein, "Computation of elementary functions on the IBM
// RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990):
//   q1 = fp32(x r),  e = fma(-q1, s, x) (exact),  q = fma(e, r, q1),
// with r the hardware reciprocal approximation of s.  rint(q) equals
// rint(fp32(x / s)) for every pair of fp16 values and every pair of bf16
// values (x, amax) with |x| <= amax and a finite fp16 scale
// s = fp16(fp32(amax/7)) of at least 2^-14: the library's encoder is checked on
// all 16-bit pairs against IEEE arithmetic (tests/test_gpu_exhaustive16.py).
// On that domain |q| < 7.01, so no clamping is needed.
__device__ __forceinline__ uint32_t int4x8_corrected(const float2 (&x)[4], float s, float r) {
  const float2 ns2 = make_float2(-s, -s), r2 = make_float2(r, r);
  const float2 magic = make_float2(kRintMagic, kRintMagic);
  uint32_t b[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 q1 = __fmul2_rn(x[e], r2);
    const float2 res = __ffma2_rn(q1, ns2, x[e]);
    const float2 q = __fadd2_rn(__ffma2_rn(res, r2, q1), magic);
    b[2 * e] = __float_as_uint(q.x);
    b[2 * e + 1] = __float_as_uint(q.y);
  }
  return pack_nibbles(b);
}

// Where `need` has bit e set, the nibble of clamp(rint(fp32(x_e / s))); called
// by the whole warp, dividing only at positions some lane needs.
__device__ __noinline__ uint32_t int4x8_fix(float2 x0, float2 x1, float2 x2, float2 x3, float s,
                                            uint32_t out, uint32_t need) {
  const float x[8] = {x0.x, x0.y, x1.x, x1.y, x2.x, x2.y, x3.x, x3.y};
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const bool n = (need >> e) & 1u;
    if (__any_sync(0xffffffffu, n)) {
      if (n) out = (out & ~(0xfu << (4 * e))) | (int4_of(__fdiv_rn(x[e], s)) << (4 * e));
    }
  }
  return out;
}

// All 8 nibbles by IEEE division (fp16 scales below the verified domain).
__device__ __noinline__ uint32_t int4x8_divide(float2 x0, float2 x1, float2 x2, float2 x3, float s) {
  const float x[8] = {x0.x, x0.y, x1.x, x1.y, x2.x, x2.y, x3.x, x3.y};
  uint32_t out = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) out |= int4_of(__fdiv_rn(x[e], s)) << (4 * e);
  return out;
}

// INT4 codes from the two brackets (fp32 sources or fp32 scales), with the
// same warp-efficient fallback as FP8.  On the fast path |q| < 7.01.
__device__ __forceinline__ uint32_t int4x8_brackets(const float2 (&x)[4], float s, const Brackets& br,
                                                    bool valid) {
  const float2 magic = make_float2(kRintMagic, kRintMagic);
  uint32_t bl[8], bh[8];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 ql = __fadd2_rn(__fmul2_rn(x[e], br.lo), magic);
    const float2 qh = __fadd2_rn(__fmul2_rn(x[e], br.hi), magic);
    bl[2 * e] = __float_as_uint(ql.x);
    bl[2 * e + 1] = __float_as_uint(ql.y);
    bh[2 * e] = __float_as_uint(qh.x);
    bh[2 * e + 1] = __float_as_uint(qh.y);
  }
  uint32_t out = pack_nibbles(bl);
  const bool slow = valid && !br.ok;  // per lane: scale too small for the brackets
  uint32_t need = 0;  // bit e: element e needs the IEEE quotient
#pragma unroll
  for (int e = 0; e < 8; ++e) need |= static_cast<uint32_t>(valid && (slow || bl[e] != bh[e])) << e;
  if (__any_sync(0xffffffffu, need != 0u)) out = int4x8_fix(x[0], x[1], x[2], x[3], s, out, need);
  return out;
}

// The rows of a warp's sub-slab.  kZeroPad: rows past n_valid (and every row
// of an inactive warp or a bad slot) read as zeros.  Otherwise every row is
// loaded: a bad slot or an inactive warp reads slot 0, and rows past n_valid
// lie inside the slot, so all loads stay in bounds; the caller discards them.
template <typename SrcT, int D, bool kZeroPad>
__device__ __forceinline__ void load_rows(const EncodeParams& p, const Where& w, const SlotInfo& si,
                                          int chunk, int rr, Raw8<SrcT> (&raw)[EncodeGeom<D>::kPasses]) {
  using G = EncodeGeom<D>;
  const bool ok = w.active && slot_errors(p, si) == 0;
  const int row0 = static_cast<int>(w.sub) * kRowsPerWarp + rr;
  const int64_t row_stride = static_cast<int64_t>(p.H) * D;
  const SrcT* base = static_cast<const SrcT*>(w.kv ? p.v : p.k) +
                     static_cast<int64_t>(w.l) * p.layer_stride +
                     static_cast<int64_t>(ok ? si.slot : 0) * p.slot_stride + w.h * D + chunk * 8 +
                     row0 * row_stride;
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const SrcT* src = base + i * G::kRowsPerPass * row_stride;
    if constexpr (kZeroPad)
      raw[i] = (ok && row0 + i * G::kRowsPerPass < si.nv) ? load8_stream(src) : raw8_zero<SrcT>();
    else
      raw[i] = load8_stream(src);
  }
}

// ---------------------------------------------------------------- Fused CRC
// The FP8 encoder can also write the CRC-32/ISO-HDLC of every slab - its
// B x d code bytes, then its 4-byte fp32 scale - the unit hc_crc32 computes
// for a = codes (B d bytes apart), b = scales (4 bytes apart).  Everything a
// CRC does is linear over GF(2) (crc_math.h), and each linear map is applied
// by lookups on 5-bit fields of its input (crc_fields.cuh), whose tables a
// warp reads without bank collisions.  A lane's code pieces (8 bytes per
// pass) lie 256 bytes apart; the map of pass i takes a piece straight to its
// contribution at the end of the lane's last piece, so a pass costs 13
// lookups.  After the last pass the lanes' registers are combined.
// Persistent CTAs run 16-token blocks, whose slab is one sub-slab: each lane
// moves its own register past the rest of the slab and the scale's 4 bytes
// with a map of its own (kLaneShift, 7 lookups, tables laid out so that
// every lane reads only its own bank), lanes 0-6 add one field each of the
// scale's contribution, and shuffles add it all.  Flat CTAs, which fill
// their tables per unit, bring the registers to the end of the sub-slab with
// a butterfly over the lanes (crc_lane_tree, 35 lookups) on shared tables;
// the sub-slabs of a slab combine in shared memory (crc_sub), and the
// register is moved past the scale's 4 bytes, which are added.  Last come
// the initial register's term and the final xor.  The images of the maps'
// single-bit inputs come from the host (make_slab_crc_constants); each CTA
// fills its tables once.
template <int kPasses, bool kLaneShift>
struct SlabCrcMaps {
  FieldMap<64> pos[kPasses];  // pass i's 8 code bytes -> the lane's register at its last piece
  FieldMap<32> level[5];      // a register -> the register 8 * 2^j bytes later
  FieldMap<32> tail;          // a register -> the register after the 4 scale bytes
  FieldMap<32> scale;         // the scale's 4 bytes -> the register after them
  // lane l's register -> the register 8 (31 - l) + 4 bytes later, after the
  // slab's last code byte and its scale (persistent CTAs run 16-token
  // blocks, whose slab is one sub-slab): entry [f][e][l] for field f of
  // value e, so lane l reads bank l only
  uint32_t lane_shift[kLaneShift ? 7 : 1][kLaneShift ? 32 : 1][kLaneShift ? 32 : 1];
};

template <int kPasses, bool kLaneShift>
__device__ __forceinline__ void build_slab_crc_maps(const EncodeParams& p,
                                                    SlabCrcMaps<kPasses, kLaneShift>& m) {
  for (int i = 0; i < kPasses; ++i) fill_field_map<64>(m.pos[i], p.crc_img_pos[i]);
  for (int j = 0; j < 5; ++j) fill_field_map<32>(m.level[j], p.crc_img_level[j]);
  fill_field_map<32>(m.tail, p.crc_img_tail);
  fill_field_map<32>(m.scale, p.crc_img_scale);
  __syncthreads();
  if constexpr (kLaneShift) {
    // The shift by 8 (31 - l) bytes is the product of the level maps of the
    // set bits of 31 - l, and the tail map adds the scale's 4.  First the
    // images of single input bits (entries 1 << b; bits past 31 give 0),
    // then every other entry as the xor of the entries of its bits.
    for (int i = threadIdx.x; i < 7 * 5 * 32; i += blockDim.x) {
      const int f = i / 160, b = (i >> 5) % 5, l = i & 31, q = 5 * f + b;
      uint32_t v = q < 32 ? 1u << q : 0u;
#pragma unroll
      for (int j = 0; j < 5; ++j)
        if (((31 - l) >> j) & 1) v = apply_map(m.level[j], v);
      m.lane_shift[f][1 << b][l] = apply_map(m.tail, v);
    }
    __syncthreads();
    for (int i = threadIdx.x; i < 7 * 32 * 32; i += blockDim.x) {
      const int f = i >> 10, e = (i >> 5) & 31, l = i & 31;
      if (e != 0 && (e & (e - 1)) == 0) continue;  // a single bit: set above
      uint32_t v = 0;
#pragma unroll
      for (int b = 0; b < 5; ++b)
        if ((e >> b) & 1) v ^= m.lane_shift[f][1 << b][l];
      m.lane_shift[f][e][l] = v;
    }
    __syncthreads();
  }
}

__device__ __forceinline__ uint32_t crc_piece(const FieldMap<64>& m, uint2 c) {
  const uint32_t v[2] = {c.x, c.y};
  return apply_map<64>(m, v);
}

// The sum over the lanes of each lane's register moved past the lane's rest
// of the slab (the lane maps) plus `add`, in every lane.
__device__ __forceinline__ uint32_t crc_lane_shift(const uint32_t (&t)[7][32][32], uint32_t acc,
                                                   uint32_t add, int lane) {
  uint32_t r = add;
#pragma unroll
  for (int f = 0; f < 7; ++f) r ^= t[f][(acc >> (5 * f)) & 31u][lane];
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) r ^= __shfl_xor_sync(0xffffffffu, r, o);
  return r;
}

// The warp's register from each lane's (positioned at the end of the lane's
// last piece; lane l's pieces start at byte 8l of each 256-byte pass block):
// a butterfly in which the lower lane of each pair moves its value 8 * 2^j
// bytes on and adds its partner's.  Lane 0 ends with the value at the end of
// the sub-slab.
__device__ __forceinline__ uint32_t crc_lane_tree(const FieldMap<32> (&level)[5], uint32_t acc,
                                                  int lane) {
#pragma unroll
  for (int j = 0; j < 5; ++j) {
    const uint32_t other = __shfl_xor_sync(0xffffffffu, acc, 1 << j);
    const uint32_t moved = apply_map(level[j], acc);
    acc = ((lane >> j) & 1) ? acc : (moved ^ other);
  }
  return acc;
}

template <typename SrcT, int D, bool kCrc, typename Maps>
__device__ __forceinline__ void quantize_fp8(const EncodeParams& p, const Where& w,
                                             const SlotInfo& si, int chunk, int rr, int warp,
                                             int lane, float* s_amax, uint32_t* s_crc,
                                             const Maps* maps,
                                             const Raw8<SrcT> (&raw)[EncodeGeom<D>::kPasses]) {
  using G = EncodeGeom<D>;
  const int bad = w.active ? slot_errors(p, si) : 0;
  const bool ok = w.active && bad == 0;
  AbsMax<SrcT> am;
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) am.add(raw[i]);  // rows past n_valid hold zeros
  float amax = am.value();
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int wps = 1 << p.grid.wps_log2;
  if (wps > 1) {  // uniform over the CTA
    if (lane == 0) s_amax[warp] = amax;
    __syncthreads();
    const int first = warp - static_cast<int>(w.sub);
    amax = 0.f;
    for (int k = 0; k < wps; ++k) amax = fmaxf(amax, s_amax[first + k]);
  }
  if (bad && lane == 0) flag_error(p.err, bad);
  if (!ok) {
    if constexpr (kCrc) {
      if (wps > 1) __syncthreads();  // the slab combine below; uniform over the CTA
    }
    return;
  }

  const float s = __fdiv_rn(amax, 448.0f);
  uint8_t* out = p.codes + w.slab * static_cast<int64_t>(p.B) * D + chunk * 8;
  const int row0 = static_cast<int>(w.sub) * kRowsPerWarp + rr;
  if constexpr (sizeof(SrcT) == 2) {
    // Rows past n_valid hold zeros, whose codes are 0.  The branch is uniform
    // over the warp (one slab); scales below 2^-90 (bf16 slabs with amax below
    // about 2^-81) and s = 0 take the IEEE division.
    uint2* dst = reinterpret_cast<uint2*>(out + static_cast<int64_t>(row0) * D);
    constexpr int kPassStride = G::kRowsPerPass * D / 8;  // in uint2
    uint32_t acc = 0;  // fused CRC: this lane's pieces so far
    if (s >= 0x1p-90f) {
      const float r = __frcp_rn(s);
#pragma unroll
      for (int i = 0; i < G::kPasses; ++i) {
        const uint2 c = fp8x8_corrected(raw[i], s, r);
        __stcs(dst + i * kPassStride, c);
        if constexpr (kCrc) acc ^= crc_piece(maps->pos[i], c);
      }
    } else {
#pragma unroll
      for (int i = 0; i < G::kPasses; ++i) {
        const uint2 c = fp8x8_divide(raw[i], s);
        __stcs(dst + i * kPassStride, c);
        if constexpr (kCrc) acc ^= crc_piece(maps->pos[i], c);
      }
    }
    if (w.sub == 0 && lane == 0) static_cast<float*>(p.scales)[w.slab] = s;
    if constexpr (kCrc && sizeof(maps->lane_shift) > 4) {
      // Persistent CTAs run 16-token blocks only, so the sub-slab is the
      // slab: each lane's map moves its register past the scale's 4 bytes
      // too, lanes 0-6 add the scale's fields, and the shuffles add it all.
      const uint32_t sb = __float_as_uint(s);  // the scale's 4 bytes, little-endian
      const uint32_t scale_part = lane < 7 ? maps->scale.f[lane][(sb >> (5 * lane)) & 31u] : 0u;
      acc = crc_lane_shift(maps->lane_shift, acc, scale_part, lane);
      if (lane == 0) p.crc[w.slab] = acc ^ p.crc_init;
    } else if constexpr (kCrc) {
      acc = crc_lane_tree(maps->level, acc, lane);  // lane 0: the sub-slab's register
      if (wps > 1) {
        if (lane == 0) s_crc[warp] = acc;
        __syncthreads();
        if (w.sub == 0) {
          const int first = warp;
          acc = 0;
          for (int k = 0; k < wps; ++k) acc ^= gf2_mul(s_crc[first + k], p.crc_sub[k]);
        }
      }
      if (w.sub == 0 && lane == 0) {
        const uint32_t sb = __float_as_uint(s);  // the scale's 4 bytes, little-endian
        p.crc[w.slab] = apply_map(maps->tail, acc) ^ apply_map(maps->scale, sb) ^ p.crc_init;
      }
    }
    return;
  }
  // fp32 sources: the bracketed products with the deferred exact tie step.
  const Brackets br = brackets(s, 0x1p-126f);
  uint32_t pend = 0;  // bit i: in pass i the brackets disagree somewhere in this lane's chunk
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = row0 + i * G::kRowsPerPass;
    uint2 c = make_uint2(0u, 0u);
    if (t < si.nv && s != 0.f) {
      float2 x[4];
      raw8_to_float2(raw[i], x);
      uint2 df;
      c = fp8x8(x, s, br, df);
      pend |= static_cast<uint32_t>((df.x | df.y) != 0u || !br.ok) << i;
    }
    __stcs(reinterpret_cast<uint2*>(out + static_cast<int64_t>(t) * D), c);
  }
  // Deferred resolution: each lane walks its own flagged passes (usually none
  // or one), so the warp spends about one short divergent trip per sub-slab.
  const float s_half_ulp = s * 0x1p-24f;
  const bool resolvable = br.ok && s >= 0x1p-90f;
  while (pend != 0u) {
    const int i = __ffs(static_cast<int>(pend)) - 1;
    pend &= pend - 1u;
    Raw8<SrcT> r = raw[0];
#pragma unroll
    for (int k = 1; k < G::kPasses; ++k)
      if (i == k) r = raw[k];
    float2 x[4];
    raw8_to_float2(r, x);
    uint2 df;
    const uint2 c = fp8x8(x, s, br, df);
    uint32_t wd[2] = {c.x, c.y};
    uint32_t todo = br.ok ? (nonzero_bytes4(df.x) | (nonzero_bytes4(df.y) << 4)) : 0xffu;
    while (todo != 0u) {
      const int e = __ffs(static_cast<int>(todo)) - 1;
      todo &= todo - 1u;
      const float2 xp = e < 2 ? x[0] : e < 4 ? x[1] : e < 6 ? x[2] : x[3];
      const float xe = (e & 1) ? xp.y : xp.x;
      const uint32_t sh = 8 * (e & 3);
      const uint32_t lo_code = (e < 4 ? wd[0] : wd[1]) >> sh;
      const uint32_t code = br.ok ? fp8_resolve(xe, s, br.hi.x, s_half_ulp, resolvable, lo_code)
                                  : fp8_div1(xe, s);
      if (e < 4)
        wd[0] = (wd[0] & ~(0xffu << sh)) | (code << sh);
      else
        wd[1] = (wd[1] & ~(0xffu << sh)) | (code << sh);
    }
    const int t = row0 + i * G::kRowsPerPass;
    __stcs(reinterpret_cast<uint2*>(out + static_cast<int64_t>(t) * D), make_uint2(wd[0], wd[1]));
  }
  if (w.sub == 0 && lane == 0) static_cast<float*>(p.scales)[w.slab] = s;
}

// kGroupLog2: log2 of the group size when fixed at compile time, else 0.
// Rows past n_valid are loaded but never used: their scale is 0 and their
// codes are 0.
template <typename SrcT, int D, bool kScaleF16, int kGroupLog2>
__device__ __forceinline__ void quantize_int4(const EncodeParams& p, const Where& w,
                                              const SlotInfo& si, int chunk, int rr, int lane,
                                              const Raw8<SrcT> (&raw)[EncodeGeom<D>::kPasses]) {
  using G = EncodeGeom<D>;
  if (!w.active) return;
  const int bad = slot_errors(p, si);
  if (bad) {
    if (lane == 0) flag_error(p.err, bad);
    return;
  }
  const int group_log2 = kGroupLog2 ? kGroupLog2 : p.group_log2;
  const int lanes_per_group = 1 << (group_log2 - 3);  // 4, 8 or 16; groups never straddle rows
  const int groups_per_row = D >> group_log2;
  uint8_t* out = p.codes + w.slab * static_cast<int64_t>(p.B) * (D / 2) + chunk * 4;
  const int64_t scale_row0 = w.slab * static_cast<int64_t>(p.B) * groups_per_row;
  const int g = (chunk * 8) >> group_log2;
  const bool scale_writer = (chunk & (lanes_per_group - 1)) == 0;
  const int row0 = static_cast<int>(w.sub) * kRowsPerWarp + rr;
  uint32_t slow = 0;   // bit i: pass i's scale lies outside the corrected path's domain
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = row0 + i * G::kRowsPerPass;
    AbsMax<SrcT> am;
    am.add(raw[i]);
    float amax = am.value();
    // group max over lanes_per_group (4, 8 or 16) neighbouring lanes
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (lanes_per_group > 4) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    if (lanes_per_group > 8) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 8));
    const bool valid = t < si.nv;
    const float s32 = valid ? div7(amax) : 0.f;  // rows past n_valid: scale 0
    const __half s16 = __float2half_rn(s32);
    const float s = kScaleF16 ? __half2float(s16) : s32;
    float2 x[4];
    raw8_to_float2(raw[i], x);
    uint32_t packed;
    if constexpr (kScaleF16 && sizeof(SrcT) == 2) {
      packed = int4x8_corrected(x, s, rcp_approx(s));
      // outside the verified domain: s == 0 gives codes 0; other scales (fp16
      // subnormal, or +inf after an fp16 overflow, where x / s = 0) are
      // divided in the deferred step below
      const bool out_of_domain = !(s >= 0x1p-14f && s <= 65504.0f);
      if (out_of_domain) packed = 0u;
      slow |= static_cast<uint32_t>(out_of_domain && s != 0.f) << i;
    } else {
      packed = int4x8_brackets(x, s, brackets(s, kScaleF16 ? 0x1p-14f : 0x1p-126f), s != 0.f);
      if (s == 0.f) packed = 0;
    }
    __stcs(reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(t) * (D / 2)), packed);
    if (scale_writer) {
      const int64_t si_ = scale_row0 + static_cast<int64_t>(t) * groups_per_row + g;
      if (kScaleF16)
        static_cast<__half*>(p.scales)[si_] = s16;
      else
        static_cast<float*>(p.scales)[si_] = s;
    }
  }
  // Deferred IEEE division for rows whose scale is outside the verified
  // domain (tiny groups, or amax >= 458752 with fp16 scales); the scale is
  // read back from where the group's writer lane stored it.
  __syncwarp();
  while (slow != 0u) {
    const int i = __ffs(static_cast<int>(slow)) - 1;
    slow &= slow - 1u;
    Raw8<SrcT> r = raw[0];
#pragma unroll
    for (int k = 1; k < G::kPasses; ++k)
      if (i == k) r = raw[k];
    float2 x[4];
    raw8_to_float2(r, x);
    const int t = row0 + i * G::kRowsPerPass;
    const int64_t si_ = scale_row0 + static_cast<int64_t>(t) * groups_per_row + g;
    const float sc = kScaleF16 ? __half2float(static_cast<const __half*>(p.scales)[si_])
                               : static_cast<const float*>(p.scales)[si_];
    __stcs(reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(t) * (D / 2)),
           int4x8_divide(x[0], x[1], x[2], x[3], sc));
  }
}

// INT4 with fp16 scales from 16-bit sources, 16 channels per lane: half the
// group reductions, scale computations, and code and scale stores per
// element of the 8-channel layout.  A lane loads 32 contiguous bytes of a
// token row (two 16-byte loads), d/16 lanes cover a row, 512/d rows per pass.
// Warps are independent, one sub-slab each, in CTAs of 4 warps (8 per SM):
// a CTA's slot on the SM is freed only when its last warp ends, and smaller
// CTAs lose less to that wait (8-warp CTAs, 4 per SM, measured 1-2 points of
// the copy peak slower per ragged layer).
#ifndef HC_INT4_ENCODE_WARPS
#define HC_INT4_ENCODE_WARPS 4
#endif
#ifndef HC_ENCODE_WIDE_MIN_BLOCKS
#define HC_ENCODE_WIDE_MIN_BLOCKS 8
#endif
constexpr int kInt4EncodeWarps = HC_INT4_ENCODE_WARPS;
template <typename SrcT, int D, int kGroupLog2>
__global__ void __launch_bounds__(kInt4EncodeWarps * 32, HC_ENCODE_WIDE_MIN_BLOCKS)
    k_encode_int4_wide(EncodeParams p) {
  static_assert(sizeof(SrcT) == 2, "16-bit sources only");
  constexpr int kLanesPerRow = D / 16;
  constexpr int kRowsPerPass = 32 / kLanesPerRow;
  constexpr int kPasses = kRowsPerWarp / kRowsPerPass;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = lane % kLanesPerRow, rr = lane / kLanesPerRow;
  const Where w = locate(p.grid, blockIdx.x * kInt4EncodeWarps + warp);
  if (!w.active) return;
  const SlotInfo si = fetch_slot(p, w);
  const int bad = slot_errors(p, si);
  if (bad) {
    if (lane == 0) flag_error(p.err, bad);
    return;
  }
  const int row0 = static_cast<int>(w.sub) * kRowsPerWarp + rr;
  const int64_t row_stride = static_cast<int64_t>(p.H) * D;
  const SrcT* src = static_cast<const SrcT*>(w.kv ? p.v : p.k) +
                    static_cast<int64_t>(w.l) * p.layer_stride +
                    static_cast<int64_t>(si.slot) * p.slot_stride + w.h * D + chunk * 16 +
                    row0 * row_stride;
  // Every row of the slot is loaded; rows past n_valid get scale 0 and codes 0.
  Raw8<SrcT> raw[kPasses][2];
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    raw[i][0] = load8_stream(src + i * kRowsPerPass * row_stride);
    raw[i][1] = load8_stream(src + i * kRowsPerPass * row_stride + 8);
  }
  const int group_log2 = kGroupLog2 ? kGroupLog2 : p.group_log2;
  const int lanes_per_group = 1 << (group_log2 - 4);  // 2, 4 or 8
  const int groups_per_row = D >> group_log2;
  const int g = (chunk * 16) >> group_log2;
  const bool scale_writer = (chunk & (lanes_per_group - 1)) == 0;
  uint2* out = reinterpret_cast<uint2*>(p.codes + w.slab * static_cast<int64_t>(p.B) * (D / 2) +
                                        static_cast<int64_t>(row0) * (D / 2) + chunk * 8);
  __half* sc = static_cast<__half*>(p.scales) + w.slab * static_cast<int64_t>(p.B) * groups_per_row +
               static_cast<int64_t>(row0) * groups_per_row + g;
  uint32_t slow = 0;  // bit i: pass i's scale lies outside the corrected path's domain
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    AbsMax<SrcT> am;
    am.add(raw[i][0]);
    am.add(raw[i][1]);
    float amax = am.value();
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    if (lanes_per_group > 2) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    if (lanes_per_group > 4) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 4));
    const bool valid = row0 + i * kRowsPerPass < si.nv;
    const __half s16 = __float2half_rn(valid ? div7(amax) : 0.f);
    const float s = __half2float(s16);
    const float r = rcp_approx(s);
    float2 x0[4], x1[4];
    raw8_to_float2(raw[i][0], x0);
    raw8_to_float2(raw[i][1], x1);
    uint2 packed = make_uint2(int4x8_corrected(x0, s, r), int4x8_corrected(x1, s, r));
    // outside the verified domain: s == 0 gives codes 0; other scales are
    // divided in the deferred step below
    const bool out_of_domain = !(s >= 0x1p-14f && s <= 65504.0f);
    if (out_of_domain) packed = make_uint2(0u, 0u);
    slow |= static_cast<uint32_t>(out_of_domain && s != 0.f) << i;
    __stcs(out + i * kRowsPerPass * (D / 16), packed);
    if (scale_writer) sc[i * kRowsPerPass * groups_per_row] = s16;
  }
  // Deferred IEEE division (rows whose scale is outside the verified domain);
  // the rows are read again rather than kept in registers.
  __syncwarp();
  while (slow != 0u) {
    const int i = __ffs(static_cast<int>(slow)) - 1;
    slow &= slow - 1u;
    const Raw8<SrcT> r0 = load8_stream(src + i * kRowsPerPass * row_stride);
    const Raw8<SrcT> r1 = load8_stream(src + i * kRowsPerPass * row_stride + 8);
    float2 x0[4], x1[4];
    raw8_to_float2(r0, x0);
    raw8_to_float2(r1, x1);
    const float s = __half2float(sc[i * kRowsPerPass * groups_per_row]);
    __stcs(out + i * kRowsPerPass * (D / 16),
           make_uint2(int4x8_divide(x0[0], x0[1], x0[2], x0[3], s),
                      int4x8_divide(x1[0], x1[1], x1[2], x1[3], s)));
  }
}

// kWire: 0 = FP8, 1 = INT4 fp16 scales, 2 = INT4 fp32 scales.
// kFlat: one unit per CTA (launch_flat: CTAs of whole slabs, at least 4
// warps; 64 registers); otherwise persistent CTAs (2 per SM) with the
// per-warp double buffer for 16-bit sources.  Measured on GB300,
// the persistent pipeline is faster for FP8 with 16-token blocks, the flat
// launch for FP8 with larger blocks (whose units meet at a CTA barrier) and
// for INT4.
// kGroupLog2: INT4 group size fixed at compile time (5: g = 32), or 0.
// kCrc: the FP8 wire with the fused slab CRC (16-bit sources).
template <typename SrcT, int D, int kWire, bool kFlat, int kGroupLog2, bool kCrc = false>
__global__ void __launch_bounds__((kCrc && !kFlat) ? kFusedCrcWarps * 32 : kThreads,
                                  kFlat ? 4 : (kCrc ? kFusedCrcCtasPerSm : 2))
    k_encode(const __grid_constant__ EncodeParams p) {
  using G = EncodeGeom<D>;
  constexpr bool kDoubleBuffer = !kFlat && sizeof(SrcT) == 2 && !(kCrc && kFusedCrcCtasPerSm > 2);
  static_assert(!kCrc || (kWire == 0 && sizeof(SrcT) == 2), "fused CRC: FP8, 16-bit sources");
  constexpr int kMaxWarps = (kCrc && !kFlat) ? kFusedCrcWarps : kWarps;
  __shared__ float s_amax[2][kMaxWarps];
  __shared__ uint32_t s_crc[2][kMaxWarps];
  using Maps = SlabCrcMaps<G::kPasses, !kFlat>;
  __shared__ typename std::conditional<kCrc, Maps, char>::type crc_maps;
  const Maps* maps = nullptr;
  if constexpr (kCrc) {
    build_slab_crc_maps(p, crc_maps);
    maps = &crc_maps;
  }
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = lane % G::kChunksPerRow, rr = lane / G::kChunksPerRow;
  const uint32_t stride = gridDim.x;
  uint32_t c = blockIdx.x;
  // a CTA's unit is as many sub-slabs as it has warps (flat launches:
  // flat_warps(B), whole slabs); persistent CTAs step through the units
  const int unit_warps = static_cast<int>(blockDim.x >> 5);
  const uint32_t units = kFlat ? gridDim.x : (p.grid.total + unit_warps - 1) / unit_warps;
  if (!kFlat && c >= units) return;  // uniform over the CTA

  auto process = [&](const Where& w, const SlotInfo& si, const Raw8<SrcT>(&raw)[G::kPasses],
                     int parity) {
    if constexpr (kWire == 0)
      quantize_fp8<SrcT, D, kCrc>(p, w, si, chunk, rr, warp, lane, s_amax[parity], s_crc[parity],
                                  maps, raw);
    else
      quantize_int4<SrcT, D, kWire == 1, kGroupLog2>(p, w, si, chunk, rr, lane, raw);
  };
  constexpr bool kZeroPad = kWire == 0;

  Where w0 = locate(p.grid, c * unit_warps + warp);
  SlotInfo s0 = fetch_slot(p, w0);
  if constexpr (kFlat) {  // the grid has one CTA per unit
    Raw8<SrcT> cur[G::kPasses];
    load_rows<SrcT, D, kZeroPad>(p, w0, s0, chunk, rr, cur);
    process(w0, s0, cur, 0);
  } else if constexpr (kDoubleBuffer) {
    Where w1 = locate(p.grid, (c + stride) * unit_warps + warp);
    SlotInfo s1 = fetch_slot(p, w1);
    Raw8<SrcT> cur[G::kPasses];
    load_rows<SrcT, D, kZeroPad>(p, w0, s0, chunk, rr, cur);
    int parity = 0;
    for (; c < units; c += stride) {
      const Where w2 = locate(p.grid, (c + 2 * stride) * unit_warps + warp);
      const SlotInfo s2 = fetch_slot(p, w2);
      Raw8<SrcT> nxt[G::kPasses];
      load_rows<SrcT, D, kZeroPad>(p, w1, s1, chunk, rr, nxt);
      process(w0, s0, cur, parity);
      parity ^= 1;
      w0 = w1;
      s0 = s1;
      w1 = w2;
      s1 = s2;
#pragma unroll
      for (int i = 0; i < G::kPasses; ++i) cur[i] = nxt[i];
    }
  } else {
    int parity = 0;
    for (; c < units; c += stride) {
      const Where w1 = locate(p.grid, (c + stride) * unit_warps + warp);
      const SlotInfo s1 = fetch_slot(p, w1);
      Raw8<SrcT> cur[G::kPasses];
      load_rows<SrcT, D, kZeroPad>(p, w0, s0, chunk, rr, cur);
      process(w0, s0, cur, parity);
      parity ^= 1;
      w0 = w1;
      s0 = s1;
    }
  }
}

// Flat launches: CTAs of HC_ENCODE_FLAT_WARPS warps, or of one slab's warps
// where a slab is larger (a slab's warps combine through shared memory, so a
// CTA holds whole slabs).  Like the INT4 encode's, smaller CTAs wait less
// for their slowest warp before the slot is freed.
#ifndef HC_ENCODE_FLAT_WARPS
#define HC_ENCODE_FLAT_WARPS 4
#endif
inline int flat_warps(const EncodeParams& p) {
  return std::max(HC_ENCODE_FLAT_WARPS, 1 << p.grid.wps_log2);
}

// The fused CRC keeps 8-warp CTAs: each CTA fills its CRC tables first.
template <typename SrcT, int D, int kWire, int kGroupLog2, bool kCrc = false>
void launch_flat(const EncodeParams& p, cudaStream_t s) {
  const int w = kCrc ? kWarps : flat_warps(p);
  const uint32_t ctas = (p.grid.total + w - 1) / w;
  k_encode<SrcT, D, kWire, true, kGroupLog2, kCrc><<<ctas, 32 * w, 0, s>>>(p);
}

// Launch shape: 16-bit INT4, and 16-bit FP8 with blocks over 16 tokens, one
// unit per CTA; everything else persistent (fp32 sources hold twice the
// registers per row).
template <typename SrcT, int D, int kWire, int kGroupLog2>
void encode_launch(const EncodeParams& p, cudaStream_t s) {
  if constexpr (sizeof(SrcT) == 2 && kWire == 1) {
    const uint32_t ctas = (p.grid.total + kInt4EncodeWarps - 1) / kInt4EncodeWarps;
    k_encode_int4_wide<SrcT, D, kGroupLog2><<<ctas, kInt4EncodeWarps * 32, 0, s>>>(p);
  } else if constexpr (sizeof(SrcT) == 2 && kWire != 0) {
    launch_flat<SrcT, D, kWire, kGroupLog2>(p, s);
  } else {
    if constexpr (sizeof(SrcT) == 2) {
      if (p.B > kRowsPerWarp) {
        launch_flat<SrcT, D, kWire, kGroupLog2>(p, s);
        return;
      }
    }
    const uint32_t grid = static_cast<uint32_t>(
        std::min<int64_t>(p.grid.units, static_cast<int64_t>(device_sm_count()) * 2));
    k_encode<SrcT, D, kWire, false, kGroupLog2><<<grid, kThreads, 0, s>>>(p);
  }
}

template <typename SrcT, int D, int kWire>
cudaError_t encode_t(const EncodeParams& p, cudaStream_t s) {
  if constexpr (kWire != 0) {
    if (p.group_log2 == 5) {
      encode_launch<SrcT, D, kWire, 5>(p, s);
      return cudaGetLastError();
    }
  }
  encode_launch<SrcT, D, kWire, 0>(p, s);
  return cudaGetLastError();
}

template <int kWire>
cudaError_t encode_dispatch(int dtype, int d, const EncodeParams& p, cudaStream_t s) {
#define HC_ENCODE_CASE(T) \
  return d == 64 ? encode_t<T, 64, kWire>(p, s) : encode_t<T, 128, kWire>(p, s);
  switch (dtype) {
    case HC_F32: HC_ENCODE_CASE(float)
    case HC_F16: HC_ENCODE_CASE(__half)
    case HC_BF16: HC_ENCODE_CASE(__nv_bfloat16)
  }
#undef HC_ENCODE_CASE
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_encode_fp8(int dtype, int d, const EncodeParams& p, cudaStream_t s) {
  return encode_dispatch<0>(dtype, d, p, s);
}

void make_slab_crc_constants(int d, int block_size, EncodeParams* p) {
  const int passes = kRowsPerWarp * d / 256;  // 8-byte pieces per lane per sub-slab
  // A register bit j (bit 31 - i holds x^i) times x^e.
  auto reg_images = [](uint32_t* img, uint64_t bits) {
    const uint32_t m = crc_x_pow_bits(bits);
    for (int j = 0; j < 32; ++j) img[j] = gf2_mul(1u << j, m);
  };
  // Bit q of pass i's piece (bit q % 8 of byte q / 8, processed first for
  // q = 0) is the coefficient of x^(63 - q); x^32 moves it into the register
  // after the piece, and x^(8 * 256) per later pass to the lane's last piece.
  for (int i = 0; i < passes; ++i)
    for (int q = 0; q < 64; ++q)
      p->crc_img_pos[i][q] = crc_x_pow_bits(95 - q + 2048ull * (passes - 1 - i));
  for (int j = 0; j < 5; ++j) reg_images(p->crc_img_level[j], 64ull << j);
  reg_images(p->crc_img_tail, 32);
  for (int q = 0; q < 32; ++q) p->crc_img_scale[q] = crc_x_pow_bits(63 - q);
  const int64_t slab = static_cast<int64_t>(block_size) * d;
  for (int sub = 0; sub < 8; ++sub) {
    const int64_t after = slab - static_cast<int64_t>(kRowsPerWarp) * d * (sub + 1);
    p->crc_sub[sub] = after >= 0 ? crc_x_pow_bytes(static_cast<uint64_t>(after)) : 0u;
  }
  p->crc_init = gf2_mul(0xFFFFFFFFu, crc_x_pow_bytes(static_cast<uint64_t>(slab + 4))) ^ 0xFFFFFFFFu;
}

template <typename SrcT, int D>
cudaError_t encode_crc_t(const EncodeParams& p, cudaStream_t s) {
  // the persistent kernel's lane maps assume one sub-slab per slab
  if (p.B != kRowsPerWarp) {
    launch_flat<SrcT, D, 0, 0, true>(p, s);
  } else {
    const int64_t units = (static_cast<int64_t>(p.grid.total) + kFusedCrcWarps - 1) / kFusedCrcWarps;
    const uint32_t grid = static_cast<uint32_t>(
        std::min<int64_t>(units, static_cast<int64_t>(device_sm_count()) * kFusedCrcCtasPerSm));
    k_encode<SrcT, D, 0, false, 0, true><<<grid, kFusedCrcWarps * 32, 0, s>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_encode_fp8_crc(int dtype, int d, const EncodeParams& p, cudaStream_t s) {
  switch (dtype) {
    case HC_F16: return d == 64 ? encode_crc_t<__half, 64>(p, s) : encode_crc_t<__half, 128>(p, s);
    case HC_BF16:
      return d == 64 ? encode_crc_t<__nv_bfloat16, 64>(p, s) : encode_crc_t<__nv_bfloat16, 128>(p, s);
  }
  return cudaErrorInvalidValue;
}

cudaError_t launch_encode_int4(int dtype, int d, bool scale_f16, const EncodeParams& p,
                               cudaStream_t s) {
  return scale_f16 ? encode_dispatch<1>(dtype, d, p, s) : encode_dispatch<2>(dtype, d, p, s);
}

}  // namespace hc
