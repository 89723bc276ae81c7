// Fetch instantiations for the FP8 E4M3 wire (one fp32 scale per slab).
#include "fetch_impl.cuh"

namespace hc {
cudaError_t launch_fetch_fp8(int out_dtype, int d, bool half_split, const FetchParams& p,
                             cudaStream_t s) {
  return fetch_detail::dispatch<fetch_detail::kFp8, false>(out_dtype, d, half_split, p, s);
}
}  // namespace hc
