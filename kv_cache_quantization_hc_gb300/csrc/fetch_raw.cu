// Fetch instantiations for the unquantized wire (values already in the paged
// dtype): the pure rotate + scatter path.
#include "fetch_impl.cuh"

namespace hc {
cudaError_t launch_fetch_raw(int out_dtype, int d, bool half_split, const FetchParams& p,
                             cudaStream_t s) {
  return fetch_detail::dispatch<fetch_detail::kRaw, false>(out_dtype, d, half_split, p, s);
}
}  // namespace hc
