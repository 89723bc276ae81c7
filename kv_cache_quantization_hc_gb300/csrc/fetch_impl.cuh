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
// lanes cover a row, 512/d rows per pass.  The warp loads its table entries
// once, issues every pass's code loads before any arithmetic, then converts
// and stores.  Each store instruction writes 8 output elements per lane;
// neighbouring lanes write neighbouring 16-byte pieces of one token row, and
// the 8 warps of a CTA write neighbouring heads.
#pragma once

#include "hc_internal.cuh"

namespace hc {
namespace fetch_detail {

enum WireKind { kFp8 = 0, kInt4 = 1, kRaw = 2 };

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
};
template <typename OutT>
struct Codes<kRaw, OutT> {
  Raw8<OutT> lo, hi;
};

__device__ __forceinline__ void fp8x8_to_float(uint2 c, float s, float (&x)[8]) {
  const uint32_t w[2] = {c.x, c.y};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __nv_fp8x2_storage_t pr = static_cast<__nv_fp8x2_storage_t>(w[i >> 1] >> (16 * (i & 1)));
    const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pr, __NV_E4M3);
    __half2 h;
    memcpy(&h, &hr, 4);
    const float2 f = __half22float2(h);  // exact: E4M3 values are fp16 values
    x[2 * i] = f.x * s;                  // one fp32 rounding of the exact product
    x[2 * i + 1] = f.y * s;
  }
}

__device__ __forceinline__ void int4x8_to_float(uint32_t c, float s, float (&x)[8]) {
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int v = static_cast<int32_t>(c << (28 - 4 * e)) >> 28;  // sign-extend nibble e
    x[e] = static_cast<float>(v) * s;  // exact: |v| <= 7 times a scale of <= 24 bits
  }
}

template <typename OutT, int D, int W, bool kHalfSplit, bool kScaleF16>
__global__ void __launch_bounds__(kThreads) k_fetch(FetchParams p) {
  using G = FetchGeom<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (gw >= sub_slab_count(p.n_layers, p.n_blocks, p.H, p.B)) return;
  const SlabCoord c = slab_coord(gw, p.H, p.n_blocks, p.B / kRowsPerWarp);

  const int32_t slot = __ldg(p.dst_slots + c.j);
  const int32_t nv = p.n_valid ? __ldg(p.n_valid + c.j) : p.B;
  const int32_t di = __ldg(p.delta_idx + c.j);
  {
    int bad = 0;
    if (slot < 0 || slot >= p.num_slots) bad |= HC_DEVERR_SLOT;
    if (nv < 1 || nv > p.B) bad |= HC_DEVERR_NVALID;
    if (di < 0 || di >= p.n_distinct) bad |= HC_DEVERR_DELTA;
    if (bad) {
      if (lane == 0) flag_error(p.err, bad);
      return;
    }
  }
  const int row0 = c.sub * kRowsPerWarp;
  if (row0 >= nv) return;  // the whole sub-slab is padding

  const int q = lane % G::kLanesPerRow;
  const int r = lane / G::kLanesPerRow;
  const int c_lo = 8 * q;
  const int c_hi = D / 2 + 8 * q;

  // ---- rotation table entries (K only; warp-uniform branch)
  float cs[8], sn[8];
  const bool is_k = c.kv == 0;
  if (is_k) {
    const float4* tab = reinterpret_cast<const float4*>(p.table + static_cast<int64_t>(di) * D);
    // float4 k of a row holds pairs 2k and 2k+1 as (c, s, c, s)
    float4 t4[4];
    if (kHalfSplit) {
#pragma unroll
      for (int i = 0; i < 4; ++i) t4[i] = __ldg(tab + 4 * q + i);        // pairs 8q .. 8q+7
    } else {
      t4[0] = __ldg(tab + 2 * q);                                          // pairs 4q .. 4q+3
      t4[1] = __ldg(tab + 2 * q + 1);
      t4[2] = __ldg(tab + D / 8 + 2 * q);                                  // pairs d/4+4q ..
      t4[3] = __ldg(tab + D / 8 + 2 * q + 1);
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      cs[2 * i] = t4[i].x;
      sn[2 * i] = t4[i].y;
      cs[2 * i + 1] = t4[i].z;
      sn[2 * i + 1] = t4[i].w;
    }
  }

  // ---- load every pass's codes (and scales) first
  Codes<W, OutT> cd[G::kPasses];
  float sc_lo[G::kPasses], sc_hi[G::kPasses];
  float s_slab = 1.f;
  const int64_t slab_rows = c.slab * static_cast<int64_t>(p.B);
  if (W == kFp8) s_slab = __ldg(static_cast<const float*>(p.scales) + c.slab);
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = row0 + r + i * G::kRowsPerPass;
    const bool valid = t < nv;
    const int64_t row = slab_rows + t;
    if constexpr (W == kFp8) {
      const uint8_t* b = static_cast<const uint8_t*>(p.codes) + row * D;
      cd[i].lo = valid ? __ldcs(reinterpret_cast<const uint2*>(b + c_lo)) : make_uint2(0, 0);
      cd[i].hi = valid ? __ldcs(reinterpret_cast<const uint2*>(b + c_hi)) : make_uint2(0, 0);
    } else if constexpr (W == kInt4) {
      const uint8_t* b = static_cast<const uint8_t*>(p.codes) + row * (D / 2);
      cd[i].lo = valid ? __ldcs(reinterpret_cast<const unsigned int*>(b + c_lo / 2)) : 0u;
      cd[i].hi = valid ? __ldcs(reinterpret_cast<const unsigned int*>(b + c_hi / 2)) : 0u;
      const int gpr = D / p.group;
      const int64_t sb = row * gpr;
      if (kScaleF16) {
        const __half* S = static_cast<const __half*>(p.scales);
        sc_lo[i] = valid ? __half2float(__ldg(S + sb + c_lo / p.group)) : 0.f;
        sc_hi[i] = valid ? __half2float(__ldg(S + sb + c_hi / p.group)) : 0.f;
      } else {
        const float* S = static_cast<const float*>(p.scales);
        sc_lo[i] = valid ? __ldg(S + sb + c_lo / p.group) : 0.f;
        sc_hi[i] = valid ? __ldg(S + sb + c_hi / p.group) : 0.f;
      }
    } else {
      const OutT* b = static_cast<const OutT*>(p.codes) + row * D;
      cd[i].lo = valid ? load8_stream(b + c_lo) : raw8_zero<OutT>();
      cd[i].hi = valid ? load8_stream(b + c_hi) : raw8_zero<OutT>();
    }
  }

  OutT* dst = static_cast<OutT*>(is_k ? p.k : p.v) + c.l * p.layer_stride +
              static_cast<int64_t>(slot) * p.slot_stride + c.h * D;
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = row0 + r + i * G::kRowsPerPass;
    if (t >= nv) continue;
    float lo[8], hi[8];
    if constexpr (W == kFp8) {
      fp8x8_to_float(cd[i].lo, s_slab, lo);
      fp8x8_to_float(cd[i].hi, s_slab, hi);
    } else if constexpr (W == kInt4) {
      int4x8_to_float(cd[i].lo, sc_lo[i], lo);
      int4x8_to_float(cd[i].hi, sc_hi[i], hi);
    } else {
      raw8_to_float(cd[i].lo, lo);
      raw8_to_float(cd[i].hi, hi);
    }
    if (is_k) {
      if (kHalfSplit) {
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float x1 = lo[e], x2 = hi[e];
          lo[e] = x1 * cs[e] - x2 * sn[e];
          hi[e] = x1 * sn[e] + x2 * cs[e];
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float x1 = lo[2 * e], x2 = lo[2 * e + 1];
          lo[2 * e] = x1 * cs[e] - x2 * sn[e];
          lo[2 * e + 1] = x1 * sn[e] + x2 * cs[e];
          x1 = hi[2 * e];
          x2 = hi[2 * e + 1];
          hi[2 * e] = x1 * cs[4 + e] - x2 * sn[4 + e];
          hi[2 * e + 1] = x1 * sn[4 + e] + x2 * cs[4 + e];
        }
      }
    }
    OutT* o = dst + static_cast<int64_t>(t) * p.H * D;
    store8(o + c_lo, lo);
    store8(o + c_hi, hi);
  }
}

template <typename OutT, int D, int W, bool kHalfSplit, bool kScaleF16>
cudaError_t launch_t(const FetchParams& p, cudaStream_t s) {
  const int64_t warps = sub_slab_count(p.n_layers, p.n_blocks, p.H, p.B);
  const int64_t grid = (warps + kWarps - 1) / kWarps;
  k_fetch<OutT, D, W, kHalfSplit, kScaleF16><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(p);
  return cudaGetLastError();
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
