// Fetch instantiations for the grouped INT4 wire (fp16 or fp32 scales).
#include "fetch_impl.cuh"

namespace hc {
cudaError_t launch_fetch_int4(int out_dtype, int d, bool half_split, bool scale_f16,
                              const FetchParams& p, cudaStream_t s) {
  return scale_f16
             ? fetch_detail::dispatch<fetch_detail::kInt4, true>(out_dtype, d, half_split, p, s)
             : fetch_detail::dispatch<fetch_detail::kInt4, false>(out_dtype, d, half_split, p, s);
}
}  // namespace hc
