// mxnorm_warp_fp8_cast.cu -- warp-row kernels for the cast-only FP8 E4M3
// form (kernel 2 of the two-pass RMSNorm baseline).  One format per
// translation unit, so the formats compile in parallel.
#include "mx_warp.cuh"

namespace mxnorm {

cudaError_t launch_warp_row_e4m3_cast(const WarpRowArgs& a, cudaStream_t s) {
  return warp_row::launch_fmt<kFmtE4M3, false>(a, s);
}

}  // namespace mxnorm
