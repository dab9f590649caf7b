// mxnorm_warp_fp8.cu -- warp-row kernels for the MXNorm pass for FP8 E4M3
// codes (no rotation).  One format per translation unit, so the formats
// compile in parallel.
#include "mx_warp.cuh"

namespace mxnorm {

cudaError_t launch_warp_row_e4m3(const WarpRowArgs& a, cudaStream_t s) {
  return warp_row::launch_fmt<kFmtE4M3, true>(a, s);
}

}  // namespace mxnorm
