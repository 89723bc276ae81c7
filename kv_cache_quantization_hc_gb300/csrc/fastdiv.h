// Division of 32-bit unsigned numerators below 2^31 by a run-time invariant
// divisor, as one high multiply, one add and one shift (Granlund and
// Montgomery, "Division by invariant integers using multiplication", 1994:
// m = floor(2^32 (2^s - d) / d) + 1 with s = ceil(log2 d), and
// n / d = (mulhi(n, m) + n) >> s).  The host builds the constants once per
// call; kernels use them to split flat work indices.
#pragma once

#include <stdint.h>

#if defined(__CUDACC__)
#define HC_HD __host__ __device__ __forceinline__
#else
#define HC_HD inline
#endif

namespace hc {

struct FastDivmod {
  uint32_t d = 1, m = 1, s = 0;

  FastDivmod() = default;
  explicit FastDivmod(uint32_t divisor) : d(divisor) {
    s = 0;
    while ((uint64_t{1} << s) < divisor) ++s;
    m = static_cast<uint32_t>(((uint64_t{1} << 32) * ((uint64_t{1} << s) - divisor)) / divisor + 1);
  }

  HC_HD uint32_t div(uint32_t n) const {  // requires n < 2^31
#if defined(__CUDA_ARCH__)
    const uint32_t hi = __umulhi(n, m);
#else
    const uint32_t hi = static_cast<uint32_t>((static_cast<uint64_t>(n) * m) >> 32);
#endif
    return (hi + n) >> s;
  }

  HC_HD void divmod(uint32_t n, uint32_t& q, uint32_t& r) const {
    q = div(n);
    r = n - q * d;
  }
};

}  // namespace hc
