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
// passes.  CTAs are persistent (two per SM) and step through "units" of 8
// consecutive sub-slabs.  The pipeline per warp is three deep: the block
// table entry for unit i+2 is requested, the rows of unit i+1 are loaded
// (16-bit sources: into a second register buffer), and unit i is quantized
// and stored - so neither the table lookup nor the row loads sit on the
// critical path.  The FP8 slab amax needs all B/16 sub-slabs of a block;
// those warps are in the same CTA and combine through shared memory.  INT4
// groups lie inside a token row, so INT4 needs no cross-warp step.
//
// Quotients without a division per element.  The codes are defined through
// the IEEE quotient q* = fp32(x / s).  With r = fp32(1/s) and the bracketing
// multipliers r_lo = fp32(r (1 - 2^-20)), r_hi = fp32(r (1 + 2^-20)), the
// products q_lo = fp32(x r_lo) and q_hi = fp32(x r_hi) satisfy
// |q_lo| < |q*| < |q_hi| (three roundings of at most 2^-24 each cannot undo a
// 2^-20 relative offset; when x/s is so small that fp32 underflows, all three
// are far below the smallest code step and encode alike).  The quantizer is
// monotone in |q| for a fixed sign, so when q_lo and q_hi give the same code,
// that is the code of q*.  Only when they differ (q* within about 2^-20 of a
// rounding boundary, roughly one element in 10^5) is the IEEE division
// evaluated, out of line, for those 8 elements.  A scale below the smallest
// normal fp32 (fp16 for INT4 fp16 scales, where clamping can then matter)
// takes the division path.  Products are formed two at a time (FMUL2).
//
// Reads use the streaming cache hint (each element is read once); codes are
// written with streaming stores.
#include <algorithm>

#include "hc_internal.cuh"

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

__device__ __forceinline__ uint32_t fp8x2(float2 v) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

__device__ __noinline__ uint2 fp8x8_exact(float2 a, float2 b, float2 c, float2 d, float s) {
  auto q = [s](float2 v) { return fp8x2(make_float2(__fdiv_rn(v.x, s), __fdiv_rn(v.y, s))); };
  return make_uint2(q(a) | (q(b) << 16), q(c) | (q(d) << 16));
}

// 8 E4M3 codes of x[0..7] / s (see the file comment).
__device__ __forceinline__ uint2 fp8x8(const float2 (&x)[4], float s, const Brackets& br) {
  uint32_t lo[4], hi[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    lo[e] = fp8x2(__fmul2_rn(x[e], br.lo));
    hi[e] = fp8x2(__fmul2_rn(x[e], br.hi));
  }
  const uint2 wl = make_uint2(lo[0] | (lo[1] << 16), lo[2] | (lo[3] << 16));
  const uint2 wh = make_uint2(hi[0] | (hi[1] << 16), hi[2] | (hi[3] << 16));
  if (((wl.x ^ wh.x) | (wl.y ^ wh.y)) != 0u || !br.ok) return fp8x8_exact(x[0], x[1], x[2], x[3], s);
  return wl;
}

// Nibble of round_half_even(q) for |q| < 2^22: adding 1.5 * 2^23 leaves the
// nearest-even integer in the low mantissa bits (one IEEE rounding); its low
// four bits are the 4-bit two's complement.
constexpr float kRintMagic = 12582912.0f;

__device__ __forceinline__ uint32_t pack_nibbles(const uint32_t (&b)[8]) {
  uint32_t out = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) out |= (b[e] & 0xfu) << (4 * e);
  return out;
}

__device__ __noinline__ uint32_t int4x8_exact(float2 a, float2 b, float2 c, float2 d, float s) {
  const float x[8] = {a.x, a.y, b.x, b.y, c.x, c.y, d.x, d.y};
  uint32_t out = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    const int q = min(7, max(-7, __float2int_rn(__fdiv_rn(x[e], s))));
    out |= (static_cast<uint32_t>(q) & 0xfu) << (4 * e);
  }
  return out;
}

// 8 INT4 nibbles of clamp(rint(x[0..7] / s)) (see the file comment).
__device__ __forceinline__ uint32_t int4x8(const float2 (&x)[4], float s, const Brackets& br) {
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
  uint32_t diff = 0;
#pragma unroll
  for (int e = 0; e < 8; ++e) diff |= bl[e] ^ bh[e];
  if (diff != 0u || !br.ok) return int4x8_exact(x[0], x[1], x[2], x[3], s);
  return pack_nibbles(bl);
}

// Block-table entries a warp needs for one unit.
struct SlotInfo {
  int32_t slot, nv;
};

__device__ __forceinline__ SlotInfo fetch_slot(const EncodeParams& p, const Where& w) {
  SlotInfo s{0, 0};
  if (w.active) {
    s.slot = __ldg(p.src_slots + w.j);
    s.nv = p.n_valid ? __ldg(p.n_valid + w.j) : p.B;
  }
  return s;
}

__device__ __forceinline__ int slot_errors(const EncodeParams& p, const SlotInfo& s) {
  int bad = 0;
  if (s.slot < 0 || s.slot >= p.num_slots) bad |= HC_DEVERR_SLOT;
  if (s.nv < 1 || s.nv > p.B) bad |= HC_DEVERR_NVALID;
  return bad;
}

template <typename SrcT, int D>
__device__ __forceinline__ void load_rows(const EncodeParams& p, const Where& w, const SlotInfo& si,
                                          int chunk, int rr, Raw8<SrcT> (&raw)[EncodeGeom<D>::kPasses]) {
  using G = EncodeGeom<D>;
  const bool ok = w.active && slot_errors(p, si) == 0;
  const SrcT* base = static_cast<const SrcT*>(w.kv ? p.v : p.k) +
                     static_cast<int64_t>(w.l) * p.layer_stride +
                     static_cast<int64_t>(ok ? si.slot : 0) * p.slot_stride + w.h * D + chunk * 8;
  const int row0 = static_cast<int>(w.sub) * kRowsPerWarp + rr;
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = row0 + i * G::kRowsPerPass;
    raw[i] = (ok && t < si.nv) ? load8_stream(base + static_cast<int64_t>(t) * p.H * D)
                               : raw8_zero<SrcT>();
  }
}

template <typename SrcT, int D>
__device__ __forceinline__ void quantize_fp8(const EncodeParams& p, const Where& w,
                                             const SlotInfo& si, int chunk, int rr, int warp,
                                             int lane, float* s_amax,
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
  if (!ok) return;

  const float s = __fdiv_rn(amax, 448.0f);
  const Brackets br = brackets(s, 0x1p-126f);
  uint8_t* out = p.codes + w.slab * static_cast<int64_t>(p.B) * D + chunk * 8;
  const int row0 = static_cast<int>(w.sub) * kRowsPerWarp + rr;
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = row0 + i * G::kRowsPerPass;
    uint2 c = make_uint2(0u, 0u);
    if (t < si.nv && s != 0.f) {
      float2 x[4];
      raw8_to_float2(raw[i], x);
      c = fp8x8(x, s, br);
    }
    __stcs(reinterpret_cast<uint2*>(out + static_cast<int64_t>(t) * D), c);
  }
  if (w.sub == 0 && lane == 0) static_cast<float*>(p.scales)[w.slab] = s;
}

template <typename SrcT, int D, bool kScaleF16>
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
  const int lanes_per_group = p.group / 8;  // 4, 8 or 16; groups never straddle rows
  const int groups_per_row = D / p.group;
  uint8_t* out = p.codes + w.slab * static_cast<int64_t>(p.B) * (D / 2) + chunk * 4;
  const int64_t scale_row0 = w.slab * static_cast<int64_t>(p.B) * groups_per_row;
  const int g = (chunk * 8) / p.group;
  const bool scale_writer = (chunk % lanes_per_group) == 0;
  const int row0 = static_cast<int>(w.sub) * kRowsPerWarp + rr;
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = row0 + i * G::kRowsPerPass;
    AbsMax<SrcT> am;
    am.add(raw[i]);
    float amax = am.value();
    for (int o = 1; o < lanes_per_group; o <<= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const bool valid = t < si.nv;
    float s = __fdiv_rn(amax, 7.0f);
    __half s16 = __float2half_rn(s);
    if (kScaleF16) s = __half2float(s16);
    if (!valid) {
      s = 0.f;
      s16 = __float2half_rn(0.f);
    }
    uint32_t packed = 0;
    if (s != 0.f) {
      float2 x[4];
      raw8_to_float2(raw[i], x);
      packed = int4x8(x, s, brackets(s, kScaleF16 ? 0x1p-14f : 0x1p-126f));
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
}

// kWire: 0 = FP8, 1 = INT4 fp16 scales, 2 = INT4 fp32 scales.
template <typename SrcT, int D, int kWire>
__global__ void __launch_bounds__(kThreads, 2) k_encode(EncodeParams p) {
  using G = EncodeGeom<D>;
  constexpr bool kDoubleBuffer = sizeof(SrcT) == 2;
  __shared__ float s_amax[2][kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = lane % G::kChunksPerRow, rr = lane / G::kChunksPerRow;
  const uint32_t stride = gridDim.x;
  uint32_t c = blockIdx.x;
  if (c >= p.grid.units) return;  // uniform over the CTA

  auto process = [&](const Where& w, const SlotInfo& si, const Raw8<SrcT>(&raw)[G::kPasses],
                     int parity) {
    if constexpr (kWire == 0)
      quantize_fp8<SrcT, D>(p, w, si, chunk, rr, warp, lane, s_amax[parity], raw);
    else
      quantize_int4<SrcT, D, kWire == 1>(p, w, si, chunk, rr, lane, raw);
  };

  Where w0 = locate(p.grid, c * kWarps + warp);
  SlotInfo s0 = fetch_slot(p, w0);
  if constexpr (kDoubleBuffer) {
    Where w1 = locate(p.grid, (c + stride) * kWarps + warp);
    SlotInfo s1 = fetch_slot(p, w1);
    Raw8<SrcT> cur[G::kPasses];
    load_rows<SrcT, D>(p, w0, s0, chunk, rr, cur);
    int parity = 0;
    for (; c < p.grid.units; c += stride) {
      const Where w2 = locate(p.grid, (c + 2 * stride) * kWarps + warp);
      const SlotInfo s2 = fetch_slot(p, w2);
      Raw8<SrcT> nxt[G::kPasses];
      load_rows<SrcT, D>(p, w1, s1, chunk, rr, nxt);
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
    for (; c < p.grid.units; c += stride) {
      const Where w1 = locate(p.grid, (c + stride) * kWarps + warp);
      const SlotInfo s1 = fetch_slot(p, w1);
      Raw8<SrcT> cur[G::kPasses];
      load_rows<SrcT, D>(p, w0, s0, chunk, rr, cur);
      process(w0, s0, cur, parity);
      parity ^= 1;
      w0 = w1;
      s0 = s1;
    }
  }
}

template <typename SrcT, int D, int kWire>
cudaError_t encode_t(const EncodeParams& p, cudaStream_t s) {
  const uint32_t grid = static_cast<uint32_t>(
      std::min<int64_t>(p.grid.units, static_cast<int64_t>(device_sm_count()) * 2));
  k_encode<SrcT, D, kWire><<<grid, kThreads, 0, s>>>(p);
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

cudaError_t launch_encode_int4(int dtype, int d, bool scale_f16, const EncodeParams& p,
                               cudaStream_t s) {
  return scale_f16 ? encode_dispatch<1>(dtype, d, p, s) : encode_dispatch<2>(dtype, d, p, s);
}

}  // namespace hc
