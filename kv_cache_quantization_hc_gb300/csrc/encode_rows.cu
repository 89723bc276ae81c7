// Row-scaled FP8 encode: gather paged K/V blocks through the source block
// table and quantize every (layer, block, kv, head, token) row of d channels
// to E4M3 with its own scale:
//   s32 = fp32(amax / 448),  s = fp16_rne(s32) (fp16 scales) or s32,
//   code = E4M3_rn_satfinite(fp32(x / s)) with the stored s.
// This is the granularity whose sizes match the FP8 frame the page prints
// (131,072 fp16 values -> 133,120 payload bytes, 1.97x).
// ["HyperCache - Distributed KV-cache quantization and relative RoPE reuse",
//  "Example output" part B, "FP8 (E4M3) Wire Quantization" and the live TCP
//  fetch frame.]
//
// One warp per 16-token sub-slab of one (layer, block, kv, head), one unit of
// 8 sub-slabs per CTA.  A lane loads 32 contiguous source bytes of a row per
// pass (16 channels of a 16-bit source, 8 of fp32); the lanes of a row combine
// their maxima with shuffles.  Rows past n_valid are loaded (they lie inside
// the slot) and given scale 0 and codes 0.
//
// Quotients: 16-bit sources use the residual-corrected product with the
// correctly rounded reciprocal of the stored scale (fp8x8_corrected), checked
// on every 16-bit (x, amax) pair for both scale types; fp32 sources, and
// scales outside that domain (0, +inf after an fp16 overflow), divide.
#include <cfloat>

#include "encode_common.cuh"

namespace hc {
namespace {

// fp32(a / 448) for non-negative finite a: div7's exact a / 7 scaled by 2^-6,
// which is exact while the result is a normal fp32 number (a >= 2^-116);
// smaller values divide.
__device__ __forceinline__ float div448(float a) {
  return a >= 0x1p-116f ? div7(a) * 0x1p-6f : __fdiv_rn(a, 448.0f);
}

// Warps are independent (one sub-slab each, a scale per row): CTAs of
// kRowsWarps warps, 4 (8 per SM for 16-bit sources), which measured 0.75%
// faster than 8-warp CTAs on the Qwen3-8B step.
#ifndef HC_ROWS_ENCODE_WARPS
#define HC_ROWS_ENCODE_WARPS 4
#endif
constexpr int kRowsWarps = HC_ROWS_ENCODE_WARPS;

template <typename SrcT, int D, bool kScaleF16>
__global__ void __launch_bounds__(kRowsWarps * 32, (sizeof(SrcT) == 2 ? 4 : 2) * 8 / kRowsWarps)
    k_encode_fp8_rows(EncodeParams p) {
  constexpr int kRaws = sizeof(SrcT) == 2 ? 2 : 1;  // Raw8 pieces (8 elements) per lane and row
  constexpr int kElems = 8 * kRaws;
  constexpr int kLanesPerRow = D / kElems;
  constexpr int kRowsPerPass = 32 / kLanesPerRow;
  constexpr int kPasses = kRowsPerWarp / kRowsPerPass;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int chunk = lane % kLanesPerRow, rr = lane / kLanesPerRow;
  const Where w = locate(p.grid, blockIdx.x * kRowsWarps + warp);
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
                    static_cast<int64_t>(si.slot) * p.slot_stride + w.h * D + chunk * kElems +
                    row0 * row_stride;
  Raw8<SrcT> raw[kPasses][kRaws];
#pragma unroll
  for (int i = 0; i < kPasses; ++i)
#pragma unroll
    for (int k = 0; k < kRaws; ++k) raw[i][k] = load8_stream(src + i * kRowsPerPass * row_stride + 8 * k);

  const int64_t row_index = w.slab * static_cast<int64_t>(p.B) + row0;  // wire row of pass 0
  uint8_t* out = p.codes + row_index * D + chunk * kElems;
#pragma unroll
  for (int i = 0; i < kPasses; ++i) {
    AbsMax<SrcT> am;
#pragma unroll
    for (int k = 0; k < kRaws; ++k) am.add(raw[i][k]);
    float amax = am.value();
#pragma unroll
    for (int o = 1; o < kLanesPerRow; o <<= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const bool valid = row0 + i * kRowsPerPass < si.nv;
    const float s32 = valid ? div448(amax) : 0.f;
    const __half s16 = __float2half_rn(s32);
    const float s = kScaleF16 ? __half2float(s16) : s32;
    uint8_t* o = out + i * kRowsPerPass * D;
    if constexpr (sizeof(SrcT) == 2) {
      uint2 c0, c1;
      if (s >= 0x1p-90f && s <= FLT_MAX) {
        const float r = __frcp_rn(s);
        c0 = fp8x8_corrected(raw[i][0], s, r);
        c1 = fp8x8_corrected(raw[i][1], s, r);
      } else {  // 0 (codes 0), or +inf (codes of +-0)
        c0 = fp8x8_divide(raw[i][0], s);
        c1 = fp8x8_divide(raw[i][1], s);
      }
      __stcs(reinterpret_cast<uint4*>(o), make_uint4(c0.x, c0.y, c1.x, c1.y));
    } else {
      __stcs(reinterpret_cast<uint2*>(o), fp8x8_divide(raw[i][0], s));
    }
    if (chunk == 0) {
      const int64_t si_ = row_index + i * kRowsPerPass;
      if (kScaleF16)
        static_cast<__half*>(p.scales)[si_] = s16;
      else
        static_cast<float*>(p.scales)[si_] = s;
    }
  }
}

template <typename SrcT, int D>
cudaError_t rows_t(bool scale_f16, const EncodeParams& p, cudaStream_t s) {
  const uint32_t ctas = (p.grid.total + kRowsWarps - 1) / kRowsWarps;
  if (scale_f16)
    k_encode_fp8_rows<SrcT, D, true><<<ctas, kRowsWarps * 32, 0, s>>>(p);
  else
    k_encode_fp8_rows<SrcT, D, false><<<ctas, kRowsWarps * 32, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_encode_fp8_rows(int dtype, int d, bool scale_f16, const EncodeParams& p,
                                   cudaStream_t s) {
#define HC_ROWS_CASE(T) \
  return d == 64 ? rows_t<T, 64>(scale_f16, p, s) : rows_t<T, 128>(scale_f16, p, s);
  switch (dtype) {
    case HC_F32: HC_ROWS_CASE(float)
    case HC_F16: HC_ROWS_CASE(__half)
    case HC_BF16: HC_ROWS_CASE(__nv_bfloat16)
  }
#undef HC_ROWS_CASE
  return cudaErrorInvalidValue;
}

}  // namespace hc
