// Rotation table of the fetch: for each distinct delta-m and pair i,
// (cos, sin)(delta_m * theta_i) with theta, the angle and cos/sin in fp64,
// each rounded once to fp32.
// ["HyperCache - Distributed KV-cache quantization and relative RoPE reuse",
//  "Core Design" relative RoPE paragraph; theta_i = base^(-2i/d) as in the
//  "Module 13: KV handoff" code listing, rope_cache.]
// The table is tiny (n_distinct x d/2 entries) next to the KV traffic; one
// thread per entry.
#include "hc_internal.cuh"

namespace hc {
namespace {

__global__ void k_delta_table(TableParams p) {
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(p.n_distinct) * p.half) return;
  const int i = static_cast<int>(idx % p.half);
  const int64_t n = idx / p.half;
  const double theta = p.inv_freq ? p.inv_freq[i] : p.theta[i];
  const double ang = static_cast<double>(p.delta_m[n]) * theta;
  double sv, cv;
  sincos(ang, &sv, &cv);
  reinterpret_cast<float2*>(p.table)[idx] = make_float2(__double2float_rn(cv), __double2float_rn(sv));
}

}  // namespace

cudaError_t launch_delta_table(const TableParams& p, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(p.n_distinct) * p.half;
  const int threads = 128;
  const int64_t grid = (n + threads - 1) / threads;
  k_delta_table<<<static_cast<unsigned>(grid), threads, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace hc
