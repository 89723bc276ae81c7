// Fetch instantiations for the row-scaled FP8 E4M3 wire (one fp16 or fp32
// scale per token row).
#include "fetch_impl.cuh"

namespace hc {
cudaError_t launch_fetch_fp8_rows(int out_dtype, int d, bool half_split, bool scale_f16,
                                  const FetchParams& p, cudaStream_t s) {
  return scale_f16
             ? fetch_detail::dispatch<fetch_detail::kFp8Rows, true>(out_dtype, d, half_split, p, s)
             : fetch_detail::dispatch<fetch_detail::kFp8Rows, false>(out_dtype, d, half_split, p, s);
}
}  // namespace hc
