// Drift-ranked token selection: which tokens to recompute after cached chunks
// are reordered.  Layer-0 K/V depends only on the embeddings, so the rotated
// layer-0 KV is exact; the tokens whose layer-0 hidden state drifted most are
// recomputed through the deeper layers.
// ["HyperCache - Distributed KV-cache quantization and relative RoPE reuse",
//  "Core Design", selective recomputation: about 15% of the tokens, those
//  whose layer-0 hidden state moved furthest, are recomputed, as in
//  CacheBlend.]
//
//   drift[s][t]  = fp32 sqrt( sum_c (fresh - cached)^2 ), summed in fp32;
//   selected[s]  = the k tokens of sequence s with the largest drift (ties to
//                  the lower index), ascending.
//
// k_drift: one warp per token row, 16-byte loads of both rows, an fma per
// element, a fixed shuffle tree.  k_select: one CTA per sequence.  The drift
// values are non-negative, so their fp32 bit patterns order like the values:
// a radix select over the four key bytes (shared-memory histograms, the bin
// found by one warp's scan) finds the k-th largest key tau and how many keys
// equal to tau belong to the top k;
// two block-wide scans then write, in index order, every token above tau and
// the first such number of tokens equal to it.
#include "hc_internal.cuh"

namespace hc {
namespace {

template <typename T>
__global__ void __launch_bounds__(kThreads) k_drift(SelectParams p) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int64_t gt = static_cast<int64_t>(blockIdx.x) * kWarps + warp;
  if (gt >= static_cast<int64_t>(p.n_seq) * p.n_tokens) return;
  const int64_t s = gt / p.n_tokens, t = gt - s * p.n_tokens;
  const int64_t off = s * p.seq_stride + t * p.token_stride;
  const T* a = static_cast<const T*>(p.cached) + off;
  const T* b = static_cast<const T*>(p.fresh) + off;
  float acc = 0.f;
#pragma unroll 4
  for (int c = lane * 8; c < p.hidden; c += 256) {
    float xa[8], xb[8];
    raw8_to_float(load8_stream(a + c), xa);
    raw8_to_float(load8_stream(b + c), xb);
#pragma unroll
    for (int e = 0; e < 8; ++e) {
      const float d = xb[e] - xa[e];
      acc = fmaf(d, d, acc);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
  if (lane == 0) p.drift[gt] = __fsqrt_rn(acc);
}

constexpr int kSelectThreads = 1024;

// Exclusive prefix count of `flag` over the CTA (in thread order) and the
// total; `warp_sums` holds 33 words of shared memory (32 warp counts, then
// the CTA's total).
__device__ __forceinline__ int block_scan(bool flag, uint32_t* warp_sums, int& total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint32_t ballot = __ballot_sync(0xffffffffu, flag);
  const int in_warp = __popc(ballot & ((1u << lane) - 1u));
  if (lane == 0) warp_sums[warp] = __popc(ballot);
  __syncthreads();
  if (warp == 0) {
    const uint32_t v = warp_sums[lane];
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += n;
    }
    warp_sums[lane] = incl - v;                    // exclusive
    if (lane == 31) warp_sums[32] = incl;          // total
  }
  __syncthreads();
  const int before = static_cast<int>(warp_sums[warp]) + in_warp;
  total = static_cast<int>(warp_sums[32]);
  __syncthreads();                                 // warp_sums is reused by the next scan
  return before;
}

__global__ void __launch_bounds__(kSelectThreads) k_select(SelectParams p) {
  __shared__ uint32_t hist[256];
  __shared__ uint32_t scan[33];
  __shared__ uint32_t s_prefix, s_left;
  const int s = blockIdx.x;
  const int n = p.n_tokens;
  const uint32_t* key = reinterpret_cast<const uint32_t*>(p.drift + static_cast<int64_t>(s) * n);
  uint32_t prefix = 0, mask = 0;
  uint32_t left = static_cast<uint32_t>(p.k);      // rank wanted among keys matching the prefix
  for (int shift = 24; shift >= 0; shift -= 8) {
    for (int i = threadIdx.x; i < 256; i += kSelectThreads) hist[i] = 0;
    __syncthreads();
    for (int t = threadIdx.x; t < n; t += kSelectThreads) {
      const uint32_t v = key[t];
      if ((v & mask) == prefix) atomicAdd(&hist[(v >> shift) & 0xffu], 1u);
    }
    __syncthreads();
    if (threadIdx.x < 32) {
      // warp 0: lane l holds bins 255 - 8l down to 248 - 8l; a scan over
      // the lanes' totals (highest bins first) finds the lane, then the bin
      const int lane = threadIdx.x;
      uint32_t c[8], tot = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        c[i] = hist[255 - 8 * lane - i];
        tot += c[i];
      }
      uint32_t incl = tot;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t nb = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += nb;
      }
      const uint32_t above_lane = incl - tot;  // keys in higher bins than this lane's
      const uint32_t hit = __ballot_sync(0xffffffffu, above_lane < left && incl >= left);
      if (lane == __ffs(hit) - 1) {
        uint32_t above = above_lane;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (above + c[i] >= left) {
            s_prefix = prefix | (static_cast<uint32_t>(255 - 8 * lane - i) << shift);
            s_left = left - above;
            break;
          }
          above += c[i];
        }
      }
    }
    __syncthreads();
    prefix = s_prefix;
    left = s_left;
    mask |= 0xffu << shift;
  }
  // prefix is the k-th largest key; `left` keys equal to it complete the top k.
  int32_t* out = p.selected + static_cast<int64_t>(s) * p.k;
  int eq_before = 0, written = 0;
  for (int base = 0; base < n; base += kSelectThreads) {
    const int t = base + threadIdx.x;
    const uint32_t v = t < n ? key[t] : 0u;
    const bool eq = t < n && v == prefix;
    int eq_total;
    const int eq_rank = eq_before + block_scan(eq, scan, eq_total);
    const bool take = t < n && (v > prefix || (eq && eq_rank < static_cast<int>(left)));
    int take_total;
    const int pos = written + block_scan(take, scan, take_total);
    if (take) out[pos] = t;
    eq_before += eq_total;
    written += take_total;
  }
}

template <typename T>
cudaError_t drift_t(const SelectParams& p, cudaStream_t s) {
  const int64_t rows = static_cast<int64_t>(p.n_seq) * p.n_tokens;
  k_drift<T><<<static_cast<uint32_t>((rows + kWarps - 1) / kWarps), kThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_drift_select(int dtype, const SelectParams& p, cudaStream_t s) {
  cudaError_t e = cudaErrorInvalidValue;
  switch (dtype) {
    case HC_F32: e = drift_t<float>(p, s); break;
    case HC_F16: e = drift_t<__half>(p, s); break;
    case HC_BF16: e = drift_t<__nv_bfloat16>(p, s); break;
  }
  if (e != cudaSuccess) return e;
  k_select<<<p.n_seq, kSelectThreads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hc
