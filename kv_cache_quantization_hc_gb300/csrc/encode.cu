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
// Work decomposition: one warp per 16-token sub-slab.  Each lane owns one
// 8-element chunk of a token row (16 bytes for fp16/bf16, 32 for fp32) per
// pass; 256/d rows per pass, d/16 passes per sub-slab.  All of a sub-slab's
// loads are issued before any arithmetic, so a warp keeps d*16*elem bytes in
// flight.  The FP8 slab amax needs every sub-slab of the block: the B/16
// warps of a slab (always in the same CTA) combine their partial amax through
// shared memory.  INT4 groups lie inside one token row, so INT4 needs no
// cross-warp step.
//
// Reads use the streaming cache hint (each element is read once); codes are
// written with streaming stores.
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
// evaluated.  A scale below the smallest normal fp32 takes the division path
// for the whole slab, since 1/s may not be representable.
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
  float lo, hi;
  bool ok;  // s is a normal fp32, so 1/s and the brackets are accurate
};

__device__ __forceinline__ Brackets brackets(float s) {
  Brackets b;
  const float r = __frcp_rn(s);
  b.lo = r * (1.0f - 0x1p-20f);
  b.hi = r * (1.0f + 0x1p-20f);
  b.ok = s >= 0x1p-126f;
  return b;
}

// clamp(round_half_even(q), -7, 7) for |q| < 2^22: adding 1.5 * 2^23 leaves
// the nearest-even integer in the low mantissa bits (one IEEE rounding).
__device__ __forceinline__ int int4_round(float q) {
  const int n = __float_as_int(q + 12582912.0f) - 0x4B400000;
  return min(7, max(-7, n));
}

__device__ __forceinline__ uint32_t fp8x2(float lo, float hi) {
  return static_cast<uint32_t>(
      __nv_cvt_float2_to_fp8x2(make_float2(lo, hi), __NV_SATFINITE, __NV_E4M3));
}

// Common front half: locate the sub-slab, validate its block, load its rows.
template <typename SrcT, int D>
struct SubSlab {
  using G = EncodeGeom<D>;
  SlabCoord c;
  int32_t nv;
  bool ok;
  int chunk, row0;
  Raw8<SrcT> raw[G::kPasses];

  __device__ __forceinline__ void load(const EncodeParams& p, int64_t gw, int lane, bool active) {
    const int wps = p.B / kRowsPerWarp;
    c = slab_coord(active ? gw : 0, p.H, p.n_blocks, wps);
    int32_t slot = 0;
    nv = 0;
    ok = false;
    if (active) {
      slot = __ldg(p.src_slots + c.j);
      nv = p.n_valid ? __ldg(p.n_valid + c.j) : p.B;
      int bad = 0;
      if (slot < 0 || slot >= p.num_slots) bad |= HC_DEVERR_SLOT;
      if (nv < 1 || nv > p.B) bad |= HC_DEVERR_NVALID;
      ok = bad == 0;
      if (bad && lane == 0) flag_error(p.err, bad);
    }
    chunk = lane % G::kChunksPerRow;
    row0 = c.sub * kRowsPerWarp + lane / G::kChunksPerRow;
    const SrcT* base = static_cast<const SrcT*>(c.kv ? p.v : p.k) + c.l * p.layer_stride +
                       static_cast<int64_t>(slot) * p.slot_stride + c.h * D + chunk * 8;
#pragma unroll
    for (int i = 0; i < G::kPasses; ++i) {
      const int t = row0 + i * G::kRowsPerPass;
      raw[i] = (ok && t < nv) ? load8_stream(base + static_cast<int64_t>(t) * p.H * D)
                              : raw8_zero<SrcT>();
    }
  }
};

template <typename SrcT, int D>
__global__ void __launch_bounds__(kThreads) k_encode_fp8(EncodeParams p) {
  using G = EncodeGeom<D>;
  __shared__ float s_amax[kWarps];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const bool active = gw < sub_slab_count(p.n_layers, p.n_blocks, p.H, p.B);

  SubSlab<SrcT, D> ss;
  ss.load(p, gw, lane, active);

  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) amax = fmaxf(amax, raw8_absmax(ss.raw[i]));
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
  const int wps = p.B / kRowsPerWarp;
  if (wps > 1) {  // uniform over the CTA
    if (lane == 0) s_amax[warp] = amax;
    __syncthreads();
    const int first = warp - ss.c.sub;
    amax = 0.f;
    for (int w = 0; w < wps; ++w) amax = fmaxf(amax, s_amax[first + w]);
  }
  if (!ss.ok) return;

  const float s = __fdiv_rn(amax, 448.0f);
  const Brackets br = brackets(s);
  uint8_t* out = p.codes + ss.c.slab * static_cast<int64_t>(p.B) * D + ss.chunk * 8;
#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = ss.row0 + i * G::kRowsPerPass;
    float x[8];
    raw8_to_float(ss.raw[i], x);
    uint32_t w[2] = {0u, 0u};
    if (t < ss.nv && s != 0.f) {
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float x0 = x[2 * e], x1 = x[2 * e + 1];
        uint32_t pr = fp8x2(x0 * br.lo, x1 * br.lo);
        if (pr != fp8x2(x0 * br.hi, x1 * br.hi) || !br.ok)
          pr = fp8x2(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
        w[e >> 1] |= pr << (16 * (e & 1));
      }
    }
    __stcs(reinterpret_cast<uint2*>(out + static_cast<int64_t>(t) * D), make_uint2(w[0], w[1]));
  }
  if (ss.c.sub == 0 && lane == 0) static_cast<float*>(p.scales)[ss.c.slab] = s;
}

template <typename SrcT, int D, bool kScaleF16>
__global__ void __launch_bounds__(kThreads) k_encode_int4(EncodeParams p) {
  using G = EncodeGeom<D>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gw = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  const bool active = gw < sub_slab_count(p.n_layers, p.n_blocks, p.H, p.B);
  if (!active) return;

  SubSlab<SrcT, D> ss;
  ss.load(p, gw, lane, true);
  if (!ss.ok) return;

  const int lanes_per_group = p.group / 8;        // 4, 8 or 16; groups never straddle rows
  const int groups_per_row = D / p.group;
  uint8_t* out = p.codes + ss.c.slab * static_cast<int64_t>(p.B) * (D / 2) + ss.chunk * 4;
  const int64_t scale_row0 = ss.c.slab * static_cast<int64_t>(p.B) * groups_per_row;
  const int g = (ss.chunk * 8) / p.group;
  const bool scale_writer = (ss.chunk % lanes_per_group) == 0;

#pragma unroll
  for (int i = 0; i < G::kPasses; ++i) {
    const int t = ss.row0 + i * G::kRowsPerPass;
    float amax = raw8_absmax(ss.raw[i]);
    for (int o = 1; o < lanes_per_group; o <<= 1)
      amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const bool valid = t < ss.nv;
    float s = __fdiv_rn(amax, 7.0f);
    __half s16 = __float2half_rn(s);
    if (kScaleF16) s = __half2float(s16);
    if (!valid) {
      s = 0.f;
      s16 = __float2half_rn(0.f);
    }
    float x[8];
    raw8_to_float(ss.raw[i], x);
    uint32_t packed = 0;
    if (s != 0.f) {
      const Brackets br = brackets(s);
#pragma unroll
      for (int e = 0; e < 8; ++e) {
        int q = int4_round(x[e] * br.lo);
        if (q != int4_round(x[e] * br.hi) || !br.ok) q = int4_round(__fdiv_rn(x[e], s));
        packed |= (static_cast<uint32_t>(q) & 0xfu) << (4 * e);
      }
    }
    __stcs(reinterpret_cast<uint32_t*>(out + static_cast<int64_t>(t) * (D / 2)), packed);
    if (scale_writer) {
      const int64_t si = scale_row0 + static_cast<int64_t>(t) * groups_per_row + g;
      if (kScaleF16)
        static_cast<__half*>(p.scales)[si] = s16;
      else
        static_cast<float*>(p.scales)[si] = s;
    }
  }
}

template <typename SrcT, int D>
cudaError_t encode_fp8_t(const EncodeParams& p, cudaStream_t s) {
  const int64_t warps = sub_slab_count(p.n_layers, p.n_blocks, p.H, p.B);
  const int64_t grid = (warps + kWarps - 1) / kWarps;
  k_encode_fp8<SrcT, D><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <typename SrcT, int D>
cudaError_t encode_int4_t(bool f16, const EncodeParams& p, cudaStream_t s) {
  const int64_t warps = sub_slab_count(p.n_layers, p.n_blocks, p.H, p.B);
  const int64_t grid = (warps + kWarps - 1) / kWarps;
  if (f16)
    k_encode_int4<SrcT, D, true><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(p);
  else
    k_encode_int4<SrcT, D, false><<<static_cast<unsigned>(grid), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

template <int D>
cudaError_t encode_fp8_d(int dtype, const EncodeParams& p, cudaStream_t s) {
  switch (dtype) {
    case HC_F32: return encode_fp8_t<float, D>(p, s);
    case HC_F16: return encode_fp8_t<__half, D>(p, s);
    case HC_BF16: return encode_fp8_t<__nv_bfloat16, D>(p, s);
  }
  return cudaErrorInvalidValue;
}

template <int D>
cudaError_t encode_int4_d(int dtype, bool f16, const EncodeParams& p, cudaStream_t s) {
  switch (dtype) {
    case HC_F32: return encode_int4_t<float, D>(f16, p, s);
    case HC_F16: return encode_int4_t<__half, D>(f16, p, s);
    case HC_BF16: return encode_int4_t<__nv_bfloat16, D>(f16, p, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace

cudaError_t launch_encode_fp8(int dtype, int d, const EncodeParams& p, cudaStream_t s) {
  return d == 64 ? encode_fp8_d<64>(dtype, p, s) : encode_fp8_d<128>(dtype, p, s);
}

cudaError_t launch_encode_int4(int dtype, int d, bool scale_f16, const EncodeParams& p,
                               cudaStream_t s) {
  return d == 64 ? encode_int4_d<64>(dtype, scale_f16, p, s)
                 : encode_int4_d<128>(dtype, scale_f16, p, s);
}

}  // namespace hc
