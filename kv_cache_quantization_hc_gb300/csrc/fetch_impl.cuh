// Fetch/decode kernel template: dequantize wire slabs, rotate every K pair by
// the block's delta-m, round to the paged dtype and scatter the valid token
// rows to the destination slot.
//
// [HyperCache - Distributed KV-cache quantization and relative RoPE reuse,
//  "Core Design" relative RoPE paragraph: post-RoPE keys cached at m_old are
//  rotated pair by pair by delta-m = m_new - m_old, since
//  R(m_new t) = R(delta-m t) R(m_old t); values are not rotated.
//  "Example output" part B: the fetched frame is dequantized and rotated on
//  the fly.]
//
// Work decomposition: one warp per 16-token sub-slab of one (layer, block,
// kv, head).  Lane q of a row owns channels [8q, 8q+8) ("low") and
// [d/2 + 8q, d/2 + 8q + 8) ("high"), so both pairing conventions keep every
// rotation pair inside one lane: half-split pairs low[e] with high[e];
// interleaved pairs (low[2e], low[2e+1]) and (high[2e], high[2e+1]).  d/16
// lanes cover a row, 512/d rows per pass.
//
// A CTA covers a unit of 4 consecutive sub-slabs; by default there is one
// unit per CTA and 7 CTAs per SM (the register budget is sized for that), as
// this write-heavy kernel gains more from resident warps than from software
// pipelining.  The same code runs persistent CTAs that step through units
// with a per-warp prefetch of the next unit when built with
// HC_FETCH_CTAS_PER_SM / HC_FETCH_DOUBLE_BUFFER (see hc_internal.cuh).
// Each store instruction writes 8 output elements per lane; neighbouring
// lanes write neighbouring 16-byte pieces of one token row, and the warps
// of a unit write neighbouring heads.  Stores are streaming (measured faster
// than write-back stores here).  Products are formed two at a time
// (FMUL2 / FFMA2).
#pragma once

#include <algorithm>

#include "hc_internal.cuh"

namespace hc {
namespace fetch_detail {

enum WireKind { kFp8 = 0, kInt4 = 1, kRaw = 2, kFp8Rows = 3 };

template <int D>
struct FetchGeom {
  static constexpr int kLanesPerRow = D / 16;
  static constexpr int kRowsPerPass = 32 / kLanesPerRow;
  static constexpr int kPasses = kRowsPerWarp / kRowsPerPass;
};

// Raw bytes one lane loads per row: low and high halves.
template <int W, typename OutT>
struct Codes;
template <typename OutT>
struct Codes<kFp8, OutT> {
  uint2 lo, hi;  // 8 E4M3 codes each
};
template <typename OutT>
struct Codes<kInt4, OutT> {
  uint32_t lo, hi;  // 8 nibbles each
  float s_lo, s_hi; // fp32 scales
  __half2 s2;       // fp16 scales (low, high half), widened at use
};
template <typename OutT>
struct Codes<kRaw, OutT> {
  Raw8<OutT> lo, hi;
};
template <typename OutT>
struct Codes<kFp8Rows, OutT> {
  uint2 lo, hi;  // 8 E4M3 codes each
  float s;       // the row's scale
};

// Everything one warp holds for one sub-slab before decoding it.
template <int W, typename OutT, int D>
struct Stage {
  Codes<W, OutT> cd[FetchGeom<D>::kPasses];
  float2 cs[4], sn[4];  // rotation table entries (K only): pairs as (cos, cos), (sin, sin)
  float s_slab;         // FP8 scale
};

struct Info {
  int32_t slot, nv, di;
};

__device__ __forceinline__ Info fetch_info(const FetchParams& p, const Where& w) {
  Info in{0, 0, 0};
  if (w.active) {
    in.slot = __ldg(p.dst_slots + w.j);
    in.nv = p.n_valid ? __ldg(p.n_valid + w.j) : p.B;
    in.di = __ldg(p.delta_idx + w.j);
  }
  return in;
}

__device__ __forceinline__ int info_errors(const FetchParams& p, const Info& in) {
  int bad = 0;
  if (in.slot < 0 || in.slot >= p.num_slots) bad |= HC_DEVERR_SLOT;
  if (in.nv < 1 || in.nv > p.B) bad |= HC_DEVERR_NVALID;
  if (in.di < 0 || in.di >= p.n_distinct) bad |= HC_DEVERR_DELTA;
  return bad;
}

__device__ __forceinline__ void fp8x8_to_float2(uint2 c, float s, float2 (&x)[4]) {
  const uint32_t w[2] = {c.x, c.y};
  const float2 s2 = make_float2(s, s);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t pr = static_cast<__nv_fp8x2_storage_t>(w[i >> 1] >> (16 * (i & 1)));
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
    __half2 h;
    memcpy(&h, &hr, 4);
    x[i] = __fmul2_rn(__half22float2(h), s2);  // exact widening, then one fp32 rounding
  }
}

// 8 nibbles -> 8 floats code * s.  Biasing every nibble by 8 makes it the
// unsigned value code + 8 in [1, 15]; placed in the low byte of the fp32
// pattern of 2^23 it reads as 2^23 + code + 8, so one subtraction of 2^23 + 8
// gives the code exactly, and one multiply by s gives code * s with one
// correct fp32 rounding, the value the oracle computes.  With an fp16 scale
// (11 significant bits) the product needs at most 14 bits and is exact; an
// fp32 scale can need 27, and then the multiply rounds it once.
__device__ __forceinline__ void int4x8_to_float2(uint32_t c, float s, float2 (&x)[4]) {
  const uint32_t b = c ^ 0x88888888u;
  const uint32_t even = b & 0x0f0f0f0fu;         // byte i: element 2i
  const uint32_t odd = (b >> 4) & 0x0f0f0f0fu;   // byte i: element 2i+1
  const float2 s2 = make_float2(s, s);
  const float2 off = make_float2(-8388616.0f, -8388616.0f);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float2 m = make_float2(__uint_as_float(__byte_perm(even, 0x4B000000u, 0x7540 + i)),
                                 __uint_as_float(__byte_perm(odd, 0x4B000000u, 0x7540 + i)));
    x[i] = __fmul2_rn(__fadd2_rn(m, off), s2);
  }
}

// The same for scales that are fp16 values (at most 11 significant bits),
// one fma per two elements: each biased code b = code + 8 in [1, 15] is put
// in mantissa bits 19..22 of 1.0, giving m = 1 + b/16 exactly, and
// x = fma(m, 16 s, -24 s) = (b - 8) s.  16 s and 24 s = 3 * 8 s are exact in
// fp32 (13 significant bits at most), and so is the result code * s (15 at
// most), so the fma's one rounding changes nothing.
__device__ __forceinline__ void int4x8_to_float2_f16s(uint32_t c, float s, float2 (&x)[4]) {
  // byte i of even / odd: 0x80 | (b << 3) for the low / high nibble of byte i
  // of c (the 0x80 is the low exponent bit of 1.0; xor 0x40 applies the bias)
  const uint32_t even = ((c << 3) & 0x78787878u) ^ 0xC0C0C0C0u;
  const uint32_t odd = ((c >> 1) & 0x78787878u) ^ 0xC0C0C0C0u;
  const float2 s16 = make_float2(16.0f * s, 16.0f * s);
  const float2 c24 = make_float2(-24.0f * s, -24.0f * s);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    // bytes [0, 0, byte i, 0x3F]: the fp32 pattern of 1 + b/16
    const float2 m = make_float2(__uint_as_float(__byte_perm(even, 0x3F000000u, 0x7044 + 0x100 * i)),
                                 __uint_as_float(__byte_perm(odd, 0x3F000000u, 0x7044 + 0x100 * i)));
    x[i] = __ffma2_rn(m, s16, c24);
  }
}

template <typename T>
__device__ __forceinline__ void raw8_to_f2(const Raw8<T>& r, float2 (&x)[4]) {
  raw8_to_float2(r, x);
}

// The wire rows of a sub-slab are loaded whatever the block table says: their
// addresses come from the sub-slab index alone (an inactive warp reads slab
// 0), padding rows exist on the wire, and rows that are not stored are
// discarded - so the loads need not wait for the table entries.  The rotation
// table row is read only for a valid block.
template <int W, typename OutT, int D, bool kHalfSplit, bool kScaleF16, int kGroupLog2>
__device__ __forceinline__ void load_codes(const FetchParams& p, const Where& w, int q, int r,
                                           Stage<W, OutT, D>& st) {
  using G = FetchGeom<D>;
  const int row0 = static_cast<int>(w.sub) * kRowsPerWarp + r;
  const int64_t rows = w.slab * static_cast<int64_t>(p.B) + row0;
  const int c_lo = 8 * q, c_hi = D / 2 + 8 * q;
  if (W == kFp8) st.s_slab = __ldg(static_cast<const float*>(p.scales) + w.slab);
  if constexpr (W == kFp8 || W == kFp8Rows) {
    const uint8_t* b = static_cast<const uint8_t*>(p.codes) + rows * D;
#pragma unroll
    for (int i = 0; i < G::kPasses; ++i) {
      st.cd[i].lo = __ldcs(reinterpret_cast<const uint2*>(b + i * G::kRowsPerPass * D + c_lo));
      st.cd[i].hi = __ldcs(reinterpret_cast<const uint2*>(b + i * G::kRowsPerPass * D + c_hi));
      if constexpr (W == kFp8Rows) {
        const int64_t si = rows + i * G::kRowsPerPass;
        st.cd[i].s = kScaleF16 ? __half2float(__ldg(static_cast<const __half*>(p.scales) + si))
                               : __ldg(static_cast<const float*>(p.scales) + si);
      }
    }
  } else if constexpr (W == kInt4) {
    const uint8_t* b = static_cast<const uint8_t*>(p.codes) + rows * (D / 2);
    const int group_log2 = kGroupLog2 ? kGroupLog2 : p.group_log2;
    const int gpr = D >> group_log2;  // groups per row
    const int64_t sb = rows * gpr;
    const int g_lo = c_lo >> group_log2, g_hi = c_hi >> group_log2;
#pragma unroll
    for (int i = 0; i < G::kPasses; ++i) {
      st.cd[i].lo = __ldcs(reinterpret_cast<const unsigned int*>(b + i * G::kRowsPerPass * (D / 2) + c_lo / 2));
      st.cd[i].hi = __ldcs(reinterpret_cast<const unsigned int*>(b + i * G::kRowsPerPass * (D / 2) + c_hi / 2));
      const int64_t si = sb + i * G::kRowsPerPass * gpr;
      if (kScaleF16) {
        const __half* S = static_cast<const __half*>(p.scales);
        st.cd[i].s2 = __halves2half2(__ldg(S + si + g_lo), __ldg(S + si + g_hi));
      } else {
        const float* S = static_cast<const float*>(p.scales);
        st.cd[i].s_lo = __ldg(S + si + g_lo);
        st.cd[i].s_hi = __ldg(S + si + g_hi);
      }
    }
  } else {
    const OutT* b = static_cast<const OutT*>(p.codes) + rows * D;
#pragma unroll
    for (int i = 0; i < G::kPasses; ++i) {
      st.cd[i].lo = load8_stream(b + i * G::kRowsPerPass * D + c_lo);
      st.cd[i].hi = load8_stream(b + i * G::kRowsPerPass * D + c_hi);
    }
  }
}

template <int W, typename OutT, int D, bool kHalfSplit>
__device__ __forceinline__ void load_table(const FetchParams& p, const Where& w, const Info& in,
                                           int q, Stage<W, OutT, D>& st) {
  const bool ok = w.active && info_errors(p, in) == 0;
  if (ok && w.kv == 0) {
    const float4* tab = reinterpret_cast<const float4*>(p.table + static_cast<int64_t>(in.di) * D);
    // float4 k of a table row holds pairs 2k and 2k+1 as (c, s, c, s)
    float4 t4[4];
    if (kHalfSplit) {
#pragma unroll
      for (int i = 0; i < 4; ++i) t4[i] = __ldg(tab + 4 * q + i);  // pairs 8q .. 8q+7
    } else {
      t4[0] = __ldg(tab + 2 * q);                                    // pairs 4q .. 4q+3
      t4[1] = __ldg(tab + 2 * q + 1);
      t4[2] = __ldg(tab + D / 8 + 2 * q);                            // pairs d/4+4q ..
      t4[3] = __ldg(tab + D / 8 + 2 * q + 1);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      st.cs[i] = make_float2(t4[i].x, t4[i].z);
      st.sn[i] = make_float2(t4[i].y, t4[i].w);
    }
  }
}

// (x1, x2) -> (x1 c - x2 s, x1 s + x2 c) for two pairs at once.
__device__ __forceinline__ void rotate2(float2& x1, float2& x2, float2 c, float2 s) {
  const float2 t = __fmul2_rn(x2, s);
  const float2 u = __fmul2_rn(x2, c);
  const float2 y1 = __ffma2_rn(x1, c, make_float2(-t.x, -t.y));
  const float2 y2 = __ffma2_rn(x1, s, u);
  x1 = y1;
  x2 = y2;
}

__device__ __forceinline__ void store8_f2(float* p, const float2 (&y)[4]) {
  __stcs(reinterpret_cast<float4*>(p), make_float4(y[0].x, y[0].y, y[1].x, y[1].y));
  __stcs(reinterpret_cast<float4*>(p) + 1, make_float4(y[2].x, y[2].y, y[3].x, y[3].y));
}
__device__ __forceinline__ void store8_f2(__half* p, const float2 (&y)[4]) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __float22half2_rn(y[i]);
    memcpy(&u[i], &h, 4);
  }
  __stcs(reinterpret_cast<uint4*>(p), make_uint4(u[0], u[1], u[2], u[3]));
}
__device__ __forceinline__ void store8_f2(__nv_bfloat16* p, const float2 (&y)[4]) {
  uint32_t u[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_bfloat162 h = __float22bfloat162_rn(y[i]);
    memcpy(&u[i], &h, 4);
  }
  __stcs(reinterpret_cast<uint4*>(p), make_uint4(u[0], u[1], u[2], u[3]));
}

template <int W, typename OutT, int D, bool kHalfSplit, bool kScaleF16>
__device__ __forceinline__ void process_stage(const FetchParams& p, const Where& w, const Info& in,
                                              int q, int r, int lane,
                                              const Stage<W, OutT, D>& st) {
  using G = FetchGeom<D>;
  if (!w.active) return;
  const int bad = info_errors(p, in);
  if (bad) {
    if (lane == 0) flag_error(p.err, bad);
    return;
  }
  const int row0 = static_cast<int>(w.sub) * kRowsPerWarp + r;
  const int c_lo = 8 * q, c_hi = D / 2 + 8 * q;
  OutT* dst = static_cast<OutT*>(w.kv == 0 ? p.k : p.v) +
              static_cast<int64_t>(w.l) * p.layer_stride +
              static_cast<int64_t>(in.slot) * p.slot_stride + w.h * D;
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = row0 + i * G::kRowsPerPass;
    if (t >= in.nv) continue;
    float2 lo[4], hi[4];
    if constexpr (W == kFp8) {
      fp8x8_to_float2(st.cd[i].lo, st.s_slab, lo);
      fp8x8_to_float2(st.cd[i].hi, st.s_slab, hi);
    } else if constexpr (W == kFp8Rows) {
      fp8x8_to_float2(st.cd[i].lo, st.cd[i].s, lo);
      fp8x8_to_float2(st.cd[i].hi, st.cd[i].s, hi);
    } else if constexpr (W == kInt4) {
      if constexpr (kScaleF16) {
        const float2 sf = __half22float2(st.cd[i].s2);  // exact widening
        int4x8_to_float2_f16s(st.cd[i].lo, sf.x, lo);
        int4x8_to_float2_f16s(st.cd[i].hi, sf.y, hi);
      } else {
        int4x8_to_float2(st.cd[i].lo, st.cd[i].s_lo, lo);
        int4x8_to_float2(st.cd[i].hi, st.cd[i].s_hi, hi);
      }
    } else {
      raw8_to_f2(st.cd[i].lo, lo);
      raw8_to_f2(st.cd[i].hi, hi);
    }
    if (w.kv == 0) {
      if (kHalfSplit) {
        // pairs (low[e], high[e]) with table entry 8q + e
#pragma unroll
        for (int k = 0; k < 4; ++k) rotate2(lo[k], hi[k], st.cs[k], st.sn[k]);
      } else {
        // pairs (low[2e], low[2e+1]) -> entry 4q + e; (high[2e], high[2e+1]) -> d/4 + 4q + e
#pragma unroll
        for (int k = 0; k < 2; ++k) {
          float2 a1 = make_float2(lo[2 * k].x, lo[2 * k + 1].x);
          float2 a2 = make_float2(lo[2 * k].y, lo[2 * k + 1].y);
          rotate2(a1, a2, st.cs[k], st.sn[k]);
          lo[2 * k] = make_float2(a1.x, a2.x);
          lo[2 * k + 1] = make_float2(a1.y, a2.y);
          float2 b1 = make_float2(hi[2 * k].x, hi[2 * k + 1].x);
          float2 b2 = make_float2(hi[2 * k].y, hi[2 * k + 1].y);
          rotate2(b1, b2, st.cs[2 + k], st.sn[2 + k]);
          hi[2 * k] = make_float2(b1.x, b2.x);
          hi[2 * k + 1] = make_float2(b1.y, b2.y);
        }
      }
    }
    OutT* o = dst + static_cast<int64_t>(t) * p.H * D;
    store8_f2(o + c_lo, lo);
    store8_f2(o + c_hi, hi);
  }
}

// kGroupLog2: INT4 group size fixed at compile time (5: g = 32), or 0.
// A unit is the kFetchWarps sub-slabs of one CTA, one per warp.
#ifndef HC_FETCH_WARPS
#define HC_FETCH_WARPS 4
#endif
constexpr int kFetchWarps = HC_FETCH_WARPS;

__host__ __device__ __forceinline__ uint32_t fetch_units(const SlabGrid& g) {
  return (g.total + kFetchWarps - 1) / kFetchWarps;
}

// The warp's sub-slab in unit c (inactive past the last unit; c may be up to
// three grids past it, which the 32-bit product must not wrap into range).
__device__ __forceinline__ Where unit_warp(const SlabGrid& g, uint32_t c, uint32_t units, int warp) {
  return locate(g, c < units ? c * kFetchWarps + warp : g.total);
}

template <typename OutT, int D, int W, bool kHalfSplit, bool kScaleF16, int kGroupLog2>
__global__ void __launch_bounds__(kFetchWarps * 32, HC_FETCH_MIN_BLOCKS) k_fetch(FetchParams p) {
  using St = Stage<W, OutT, D>;
  constexpr bool kDoubleBuffer = HC_FETCH_DOUBLE_BUFFER && W != kRaw;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = lane % FetchGeom<D>::kLanesPerRow, r = lane / FetchGeom<D>::kLanesPerRow;
  const uint32_t stride = gridDim.x, units = fetch_units(p.grid);
  uint32_t c = blockIdx.x;
  if (c >= units) return;
  Where w0 = locate(p.grid, c * kFetchWarps + warp);
  Info i0 = fetch_info(p, w0);
  if constexpr (kDoubleBuffer) {
    Where w1 = unit_warp(p.grid, c + stride, units, warp);
    Info i1 = fetch_info(p, w1);
    St cur;
    load_codes<W, OutT, D, kHalfSplit, kScaleF16, kGroupLog2>(p, w0, q, r, cur);
    load_table<W, OutT, D, kHalfSplit>(p, w0, i0, q, cur);
    for (; c < units; c += stride) {
      const Where w2 = unit_warp(p.grid, c + 2 * stride, units, warp);
      const Info i2 = fetch_info(p, w2);
      St nxt;
      load_codes<W, OutT, D, kHalfSplit, kScaleF16, kGroupLog2>(p, w1, q, r, nxt);
      load_table<W, OutT, D, kHalfSplit>(p, w1, i1, q, nxt);
      process_stage<W, OutT, D, kHalfSplit, kScaleF16>(p, w0, i0, q, r, lane, cur);
      w0 = w1;
      i0 = i1;
      w1 = w2;
      i1 = i2;
      cur = nxt;
    }
  } else {
    for (;;) {
      St cur;
      load_codes<W, OutT, D, kHalfSplit, kScaleF16, kGroupLog2>(p, w0, q, r, cur);
      load_table<W, OutT, D, kHalfSplit>(p, w0, i0, q, cur);
      process_stage<W, OutT, D, kHalfSplit, kScaleF16>(p, w0, i0, q, r, lane, cur);
      c += stride;
      if (c >= units) break;  // one unit per CTA: no next unit
      w0 = locate(p.grid, c * kFetchWarps + warp);
      i0 = fetch_info(p, w0);
    }
  }
}

// INT4 wire: K and V of the same (layer, block, head, sub-slab) in one warp.
// The two share one set of block-table loads, and the V sub-slab (which is
// not rotated) is decoded and stored while the K sub-slab's rotation-table row
// is in flight, so the warp no longer idles on the chain block table ->
// table row.  The two stages need about 88 registers.  Measured on GB300
// against the one-sub-slab-per-warp fetch at 4 CTAs/SM: ragged INT4
// per-layer calls B16 87.6% -> 90.7%, B64 90.1% -> 91.8% of the copy peak;
// for the FP8 wire the same pairing measured 2 points slower on the
// Llama-shaped fetch, so the FP8, row-scaled FP8 and RAW wires keep one
// sub-slab per warp.
// Warps are independent; CTAs of 4 warps, 5 per SM.  A CTA's slot is freed
// only when its last warp ends, and 8-warp CTAs (3 per SM) lost about 3
// points of the copy peak per ragged layer to that wait.
#ifndef HC_FETCH_KV_WARPS
#define HC_FETCH_KV_WARPS 4
#endif
#ifndef HC_FETCH_KV_MIN_BLOCKS
#define HC_FETCH_KV_MIN_BLOCKS 5
#endif
constexpr int kPairWarps = HC_FETCH_KV_WARPS;

template <typename OutT, int D, int W, bool kHalfSplit, bool kScaleF16, int kGroupLog2>
__global__ void __launch_bounds__(kPairWarps * 32, HC_FETCH_KV_MIN_BLOCKS) k_fetch_kv(FetchParams p) {
  using St = Stage<W, OutT, D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int q = lane % FetchGeom<D>::kLanesPerRow, r = lane / FetchGeom<D>::kLanesPerRow;
  // K sub-slab gk of the call; its flat index and its V partner's (the same
  // (layer, block) holds 2 H wps sub-slabs, K's first, then V's)
  const uint32_t half_total = p.grid.total / 2;
  const uint32_t gk = blockIdx.x * kPairWarps + warp;
  uint32_t fk = p.grid.total, fv = p.grid.total;  // out of range: an inactive warp
  if (gk < half_total) {
    const uint32_t per_lj = p.grid.per_lj.d, half = per_lj / 2;
    const uint32_t lj = p.grid.per_lj.div(2 * gk);
    fk = lj * per_lj + (gk - lj * half);
    fv = fk + half;
  }
  const Where wk = locate(p.grid, fk);
  const Where wv = locate(p.grid, fv);
  const Info in = fetch_info(p, wk);  // one block for both
  St ck, cv;
  load_codes<W, OutT, D, kHalfSplit, kScaleF16, kGroupLog2>(p, wk, q, r, ck);
  load_codes<W, OutT, D, kHalfSplit, kScaleF16, kGroupLog2>(p, wv, q, r, cv);
  load_table<W, OutT, D, kHalfSplit>(p, wk, in, q, ck);
  process_stage<W, OutT, D, kHalfSplit, kScaleF16>(p, wv, in, q, r, lane, cv);
  process_stage<W, OutT, D, kHalfSplit, kScaleF16>(p, wk, in, q, r, lane, ck);
}

template <typename OutT, int D, int W, bool kHalfSplit, bool kScaleF16>
cudaError_t launch_t(const FetchParams& p, cudaStream_t s) {
  if constexpr (W == kInt4) {
    const uint32_t grid = (p.grid.total / 2 + kPairWarps - 1) / kPairWarps;
    if (p.group_log2 == 5)
      k_fetch_kv<OutT, D, W, kHalfSplit, kScaleF16, 5><<<grid, kPairWarps * 32, 0, s>>>(p);
    else
      k_fetch_kv<OutT, D, W, kHalfSplit, kScaleF16, 0><<<grid, kPairWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
  } else {
    const uint32_t grid = static_cast<uint32_t>(std::min<int64_t>(
        fetch_units(p.grid), static_cast<int64_t>(device_sm_count()) * HC_FETCH_CTAS_PER_SM));
    k_fetch<OutT, D, W, kHalfSplit, kScaleF16, 0><<<grid, kFetchWarps * 32, 0, s>>>(p);
    return cudaGetLastError();
  }
}

template <int W, bool kScaleF16>
cudaError_t dispatch(int out_dtype, int d, bool half_split, const FetchParams& p, cudaStream_t s) {
#define HC_FETCH_CASE(T)                                                                  \
  if (d == 64)                                                                            \
    return half_split ? launch_t<T, 64, W, true, kScaleF16>(p, s)                         \
                      : launch_t<T, 64, W, false, kScaleF16>(p, s);                       \
  return half_split ? launch_t<T, 128, W, true, kScaleF16>(p, s)                          \
                    : launch_t<T, 128, W, false, kScaleF16>(p, s);
  switch (out_dtype) {
    case HC_F32: { HC_FETCH_CASE(float) }
    case HC_F16: { HC_FETCH_CASE(__half) }
    case HC_BF16: { HC_FETCH_CASE(__nv_bfloat16) }
  }
#undef HC_FETCH_CASE
  return cudaErrorInvalidValue;
}

}  // namespace fetch_detail
}  // namespace hc
