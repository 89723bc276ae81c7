// Pieces shared by the encode kernels (encode.cu, encode_rows.cu): E4M3
// conversion, the corrected-quotient FP8 codes for 16-bit sources, the
// division-free amax / 7, and the source block-table lookups.
#pragma once

#include "hc_internal.cuh"

namespace hc {
namespace {

__device__ __forceinline__ uint32_t fp8x2(float2 v) {
  return static_cast<uint32_t>(__nv_cvt_float2_to_fp8x2(v, __NV_SATFINITE, __NV_E4M3));
}

// 8 E4M3 codes for 16-bit sources: the quotient corrected by its exact
// residual, q1 = fp32(x r), e = fma(-q1, s, x), q = fma(e, r, q1), with
// r = fp32(1/s) correctly rounded (Markstein, IBM J. Res. Dev. 34(1), 1990),
// then one RNE-satfinite conversion.  q equals fp32(x / s) for every pair of
// fp16 values and every pair of bf16 values (x, amax) with |x| <= amax and
// s = fp32(amax / 448) >= 2^-90, or s that value rounded to fp16 (the
// row-scaled wire): the library's encoders are checked on all 16-bit pairs
// against IEEE arithmetic (tests/test_gpu_exhaustive16.py).
// Exact E4M3 ties (x = 3/4 amax gives q = 336) therefore need no special
// step.  The corrected quotient of -0 is +0, so the sign bits of the inputs
// are OR-ed into the codes (for any other input the sign is already there).
template <typename SrcT>
__device__ __forceinline__ uint2 fp8x8_corrected(const Raw8<SrcT>& raw, float s, float r) {
  static_assert(sizeof(SrcT) == 2, "16-bit sources only");
  float2 x[4];
  raw8_to_float2(raw, x);
  const float2 ns2 = make_float2(-s, -s), r2 = make_float2(r, r);
  uint32_t c[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 q1 = __fmul2_rn(x[e], r2);
    const float2 res = __ffma2_rn(q1, ns2, x[e]);
    c[e] = fp8x2(__ffma2_rn(res, r2, q1));
  }
  const uint4 v = raw.w[0];  // sign of element k at bit 16k + 15 of the 8 packed inputs
  return make_uint2((c[0] | (c[1] << 16)) | (__byte_perm(v.x, v.y, 0x7531) & 0x80808080u),
                    (c[2] | (c[3] << 16)) | (__byte_perm(v.z, v.w, 0x7531) & 0x80808080u));
}

// 8 E4M3 codes by IEEE division (s = 0 gives codes 0).
template <typename SrcT>
__device__ __noinline__ uint2 fp8x8_divide(Raw8<SrcT> raw, float s) {
  if (s == 0.f) return make_uint2(0u, 0u);
  float2 x[4];
  raw8_to_float2(raw, x);
  uint32_t c[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) c[e] = fp8x2(make_float2(__fdiv_rn(x[e].x, s), __fdiv_rn(x[e].y, s)));
  return make_uint2(c[0] | (c[1] << 16), c[2] | (c[3] << 16));
}

// fp32(a / 7) for every non-negative finite fp32 a, without a division: the
// product with fp32(1/7) is corrected by its exact residual (Markstein's
// correction, as in int4x8_corrected).  Checked against the IEEE division on
// the GPU for all 2^31 non-negative finite fp32 values: no mismatch.
__device__ __forceinline__ float div7(float a) {
  const float r7 = 0.142857149f;  // fp32(1/7)
  const float q1 = a * r7;
  return fmaf(fmaf(-q1, 7.0f, a), r7, q1);
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

}  // namespace
}  // namespace hc
